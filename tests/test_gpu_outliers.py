"""Static outlier retention on the GPU against the oracle, bit for bit
("Resumo Técnico: TetraJet-v2", §2C, OutControl): calibration channel amax,
top-k channel selection, and the split FP4 / FP8 quantization."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import FMT_O, as_oracle_input, assert_eq, bits, check_q, npy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _act(shape, seed, dtype=torch.bfloat16, channel_seed=77):
    """A batch of the outlier-channel activation recipe (shared channels)."""
    return W.channel_act(shape, seed=seed, channel_seed=channel_seed,
                         n_outlier_cols=shape[1] // 16).to(dtype)


def _calib_batches(shape, n, seed, dtype):
    """n calibration batches of the activation recipe (same outlier channels)."""
    return [_act(shape, seed + t, dtype) for t in range(n)]


def _select_parity(amax_gpu, k):
    sel = fq.fq_select_channels(amax_gpu, k)
    torch.cuda.synchronize()
    ref = oracle.select_channels(npy(amax_gpu), k)
    assert_eq("idx", npy(sel.idx), ref["idx"])
    assert_eq("bitmap", npy(sel.bitmap).view(np.uint32), ref["bitmap"])
    assert_eq("fp8_scale", npy(sel.fp8_scale).view(np.uint32), ref["fp8_scale"].view(np.uint32))
    return sel, ref


def _outlier_parity(x, sel, fmt, rnd=fq.RNE, seed=0, offset=0, xhat_dtype=None):
    rows, cols = x.shape
    cfg = fq.Config(fmt, rnd, seed, offset)
    out, fp8, xhat, mask = fq.fq_quantize_outliers(x, cfg, sel, xhat_dtype=xhat_dtype)
    torch.cuda.synchronize()
    ref = oracle.quantize_outliers(as_oracle_input(x), npy(sel.idx), npy(sel.fp8_scale),
                                   FMT_O[fmt], rnd, seed, offset)
    check_q("fp4", out, ref, fmt)
    assert_eq("fp8", npy(fp8), ref["fp8"])
    if xhat.dtype == torch.bfloat16:
        assert_eq("xhat(bf16)", bits(xhat), oracle.f32_to_bf16_bits(ref["xhat"]))
    else:
        assert_eq("xhat(f32)", bits(xhat), ref["xhat"].view(np.uint32))
    nbytes = (rows * cols + 7) // 8
    assert_eq("mask", npy(mask)[:nbytes], ref["mask"].view(np.uint8)[:nbytes])
    return ref, (out, fp8, xhat, mask)


# ------------------------------------------------------------------ calibration
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_channel_amax_running_window(dtype):
    shape = (300, 1040)                  # rows ragged against the row stripes; cols % 32 != 0
    amax = torch.zeros(shape[1], dtype=torch.float32, device=DEV)
    want = None
    for xb in _calib_batches(shape, 3, seed=41, dtype=dtype):
        fq.fq_channel_amax(xb.to(DEV), amax)
        want = oracle.channel_amax(as_oracle_input(xb), want)
    torch.cuda.synchronize()
    assert_eq("channel_amax", npy(amax).view(np.uint32), want.view(np.uint32))


def test_channel_amax_tall_and_single_row():
    for shape in ((1, 64), (70001, 16)):
        x = W.normal(shape, 3.0, seed=5)
        a = fq.fq_channel_amax(x.to(DEV))
        torch.cuda.synchronize()
        assert_eq("channel_amax", npy(a).view(np.uint32),
                  oracle.channel_amax(as_oracle_input(x)).view(np.uint32))


# ------------------------------------------------------------------ selection
@pytest.mark.parametrize("cols,k", [(1040, 0), (1040, 1), (1040, 104), (1040, 1040),
                                    (16, 3), (16384, 1638)])
def test_select_channels(cols, k):
    g = torch.Generator().manual_seed(cols + k)
    a = torch.rand(cols, generator=g) * 4.0
    a[torch.randperm(cols, generator=g)[: cols // 8]] = 2.0   # ties across the k-th place
    a[: cols // 16] = 0.0                                      # zero channels
    a[cols // 3] = 1e30
    _select_parity(a.to(DEV), k)


def test_select_channels_all_equal_and_max_channels():
    _select_parity(torch.full((1000,), 0.5, device=DEV), 37)   # ties only: lowest indices
    cols, k = fq.MAX_CHANNELS, fq.MAX_CHANNELS // 10
    a = torch.rand(cols, generator=torch.Generator().manual_seed(9)).to(DEV)
    sel = fq.fq_select_channels(a, k)
    torch.cuda.synchronize()
    # at this size, compare with a stable descending sort (ties: lower index)
    av = npy(a)
    order = np.lexsort((np.arange(cols), -av.astype(np.float64)))
    want = np.sort(order[:k]).astype(np.int32)
    assert_eq("idx", npy(sel.idx), want)
    assert int(np.unpackbits(npy(sel.bitmap).view(np.uint8)).sum()) == k


# ------------------------------------------------------------------ split quantization
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_quantize_outliers_small(dtype, fmt, rnd):
    rows, cols = 200, 384                          # ragged against the 256-block CTA sweep
    calib = _calib_batches((rows, cols), 2, seed=7, dtype=dtype)
    amax = torch.zeros(cols, dtype=torch.float32, device=DEV)
    for xb in calib:
        fq.fq_channel_amax(xb.to(DEV), amax)
    sel, _ = _select_parity(amax, cols // 10)
    # the quantized batch is not a calibration batch: some kept values exceed
    # 448 s_c (saturate, clipped in the mask)
    x = _act((rows, cols), 8, dtype)
    x[5] = x[5] * 3.0
    x[9, :] = 0.0
    x[11, 3] = -0.0
    _outlier_parity(x.to(DEV), sel, fmt, rnd, seed=0xF00D, offset=11)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_quantize_outliers_whole_warp_spans(dtype, fmt, rnd):
    """Rows of a whole number of 32-block spans (1024 columns: 64 blocks of 16
    or 32 of 32): the retained elements come from the shared sorted column
    list rather than a per-warp search."""
    rows, cols = 96, 1024
    calib = _calib_batches((rows, cols), 2, seed=17, dtype=dtype)
    amax = torch.zeros(cols, dtype=torch.float32, device=DEV)
    for xb in calib:
        fq.fq_channel_amax(xb.to(DEV), amax)
    sel, _ = _select_parity(amax, cols // 10)
    x = _act((rows, cols), 18, dtype)
    x[3] = x[3] * 3.0
    x[7, :] = 0.0
    x[10, 5] = -0.0
    _outlier_parity(x.to(DEV), sel, fmt, rnd, seed=0xBEEF, offset=3)


def test_quantize_outliers_whole_spans_every_channel_kept():
    rows, cols = 8, 512
    x = W.nvfp4_act(shape=(rows, cols), seed=19, n_outlier_cols=4).to(DEV)
    sel, _ = _select_parity(fq.fq_channel_amax(x), cols)
    for fmt in (fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL):
        _outlier_parity(x, sel, fmt)


@pytest.mark.parametrize("k", [8192, 8200])
def test_quantize_outliers_long_channel_lists(k):
    """8192 retained channels (the longest list kept in shared memory) and
    8200 (the per-warp search instead), on 16384 columns."""
    rows, cols = 4, 16384
    x = W.channel_act((rows, cols), seed=20, channel_seed=21, n_outlier_cols=64).to(DEV)
    sel, _ = _select_parity(fq.fq_channel_amax(x), k)
    _outlier_parity(x, sel, fq.NVFP4)


@pytest.mark.parametrize("cols,k", [(16384, 1638), (16896, 1689), (16384, 1100)])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.NVFP4_2LEVEL])
def test_quantize_outliers_both_sides_of_the_keep_mask_image(cols, k, fmt):
    """BF16 rows of up to 16384 columns zero their retained elements with a
    keep-mask image of the row held in shared memory; longer rows test the
    bitmap bit by bit.  One row length on each side with 10% of channels
    kept, and 1100 kept channels on 16384 columns, whose list and image just
    fit in 48 KB of dynamic shared memory beside the kernel's static part."""
    rows = 8
    x = W.channel_act((rows, cols), seed=22, channel_seed=23,
                      n_outlier_cols=64).to(torch.bfloat16).to(DEV)
    sel, _ = _select_parity(fq.fq_channel_amax(x), k)
    _outlier_parity(x, sel, fmt)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_quantize_outliers_k_zero_matches_plain_fakequant(fmt):
    rows, cols = 64, 256
    x = W.nvfp4_act(shape=(rows, cols), seed=12, n_outlier_cols=4).to(DEV)
    sel = fq.fq_select_channels(torch.rand(cols, device=DEV), 0)
    out, fp8, xhat, mask = fq.fq_quantize_outliers(x, fq.Config(fmt), sel)
    xh2, mask2, rq, _ = fq.fq_fakequant_ste(x, fq.Config(fmt), want_row_q=True)
    torch.cuda.synchronize()
    assert_eq("xhat", bits(xhat), bits(xh2))
    assert_eq("mask", npy(mask), npy(mask2))
    assert_eq("codes", npy(out.codes), npy(rq.codes))
    assert_eq("scales", npy(out.scales), npy(rq.scales))


def test_quantize_outliers_every_channel_kept():
    rows, cols = 32, 128
    x = W.nvfp4_act(shape=(rows, cols), seed=13, n_outlier_cols=4).to(DEV)
    a = fq.fq_channel_amax(x)
    sel, _ = _select_parity(a, cols)
    for fmt in (fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL):
        _outlier_parity(x, sel, fmt)


def test_quantize_outliers_zero_scale_channel():
    """A kept channel whose calibration amax is 0 has scale 0: its values
    quantize to (signed) zero and fall outside the mask unless zero."""
    rows, cols = 16, 64
    x = W.normal((rows, cols), 1.0, seed=14).to(DEV)
    a = fq.fq_channel_amax(x)
    a[8] = 0.0
    a[9] = 0.0
    sel = fq.fq_select_channels(a, cols - 1)   # ties: keeps channel 8 (scale 0), drops 9
    assert 8 in npy(sel.idx) and 9 not in npy(sel.idx)
    _outlier_parity(x, sel, fq.NVFP4)


def test_outlier_retention_lowers_block_error():
    """The point of retention: the ordinary elements of rows that share blocks
    with outlier channels are reconstructed better than by plain NVFP4."""
    rows, cols = 512, 1024
    x = W.channel_act((rows, cols), seed=15, n_outlier_cols=16).to(DEV)
    sel = fq.fq_select_channels(fq.fq_channel_amax(x), 16)
    _, _, xh_keep, _ = fq.fq_quantize_outliers(x, fq.Config(fq.NVFP4), sel,
                                               xhat_dtype=torch.float32)
    xh_plain, _, _, _ = fq.fq_fakequant_ste(x, fq.Config(fq.NVFP4), xhat_dtype=torch.float32)
    keep = torch.zeros(cols, dtype=torch.bool, device=DEV)
    keep[sel.idx.long()] = True
    xf = x.float()
    e_keep = (xh_keep - xf)[:, ~keep].pow(2).mean().item()
    e_plain = (xh_plain - xf)[:, ~keep].pow(2).mean().item()
    assert e_keep < 0.5 * e_plain


# ------------------------------------------------------------------ full size
@pytest.mark.slow
def test_full_activation_outliers_nvfp4():
    """8192 x 8192 BF16 activation, 10% of the channels kept (calibration on
    two other batches with the same outlier channels), NVFP4 nearest-even."""
    cfg = W.WORKLOADS["channel_act"]
    shape = cfg["shape"]
    amax = torch.zeros(shape[1], dtype=torch.float32, device=DEV)
    for t in (1, 2):
        fq.fq_channel_amax(W.channel_act(shape, seed=cfg["seed"] + t).to(DEV), amax)
    sel, _ = _select_parity(amax, shape[1] // 10)
    x = W.channel_act(shape).to(DEV)
    _outlier_parity(x, sel, fq.NVFP4, xhat_dtype=torch.bfloat16)


def test_column_half_composes_from_quantize_col():
    """The backward (column-wise, X^T) half of retention: X^T's 16x1 blocks
    lie inside single channels, so for every channel that is not kept they
    are fq_quantize(COL) of x under the masked tensor amax -- the amax that
    fq_quantize_outliers leaves in its workspace."""
    rows, cols = 256, 512
    x = _act((rows, cols), 21).to(DEV)
    sel = fq.fq_select_channels(fq.fq_channel_amax(x), cols // 10)
    cfg = fq.Config(fq.NVFP4)
    ws = fq.workspace(cfg, rows, cols, DEV)
    fq.fq_quantize_outliers(x, cfg, sel, ws=ws)
    amax_masked = ws[:4].view(torch.float32)
    _, cq = fq.fq_quantize(x, cfg, orient=fq.COL, amax_in=amax_masked)
    torch.cuda.synchronize()
    xz = as_oracle_input(x).copy()
    kept = npy(sel.idx)
    xz[:, kept] = 0.0
    ref = oracle.quantize(xz, oracle.NVFP4, orient=oracle.ROWCOL)["col"]
    other = np.setdiff1d(np.arange(cols), kept)
    assert_eq("col.codes", npy(cq.codes)[other], ref["codes"][other])
    assert_eq("col.scales", npy(cq.scales)[other], ref["scales"][other])
    assert_eq("col.tscale", npy(cq.tscale)[:1].view(np.uint32),
              ref["tscale"].reshape(-1)[:1].view(np.uint32))
