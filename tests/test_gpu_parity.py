"""GPU vs oracle, bit for bit, through the C ABI (needs a GB300).

Small cases span several tiles with ragged tails; the large cases are the
five workloads at their full sizes, in the same launch configuration the
benchmark times."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import (FMT_O, as_oracle_input, assert_eq, bits, check_q, fakequant_parity,
                        npy)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _dev(t):
    return t.to(DEV)


# ------------------------------------------------------------------ small, ragged
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_row_small(dtype, fmt, rnd):
    rows, cols = 37, 384                        # ragged row count, several CTAs' worth
    x = W.normal((rows, cols), 1.0, seed=10 + fmt).to(dtype)
    x[3, 5] = 80.0
    x[7, :16] = 0.0
    fakequant_parity(_dev(x), fmt, rnd, seed=0xABCDEF1234, offset=7)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_rowcol_small_ragged_tiles(dtype, fmt, rnd):
    rows = 384 if fmt == fq.NVFP4_2LEVEL else 224   # not a multiple of the 64-row tile
    cols = 384 if fmt == fq.NVFP4_2LEVEL else 160   # not a multiple of the 64-col tile
    x = W.nvfp4_act(shape=(rows, cols), seed=20 + fmt, n_outlier_cols=3).to(dtype)
    fakequant_parity(_dev(x), fmt, rnd, seed=99, offset=3, orient=fq.ROWCOL)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_col_only_and_quantize_entry(fmt):
    rows, cols = 256, 256
    x = _dev(W.nvfp4_act(shape=(rows, cols), seed=5, n_outlier_cols=2))
    cfg = fq.Config(fmt, fq.RNE)
    _, cq = fq.fq_quantize(x, cfg, orient=fq.COL)
    rq, _ = fq.fq_quantize(x, cfg, orient=fq.ROW)
    torch.cuda.synchronize()
    ref = oracle.quantize(as_oracle_input(x), FMT_O[fmt], orient=oracle.ROWCOL)
    check_q("col", cq, ref["col"], fmt)
    check_q("row", rq, ref["row"], fmt)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_dequantize_matches_oracle_and_fakequant(fmt, ydt):
    rows, cols = 64, 512
    x = _dev(W.grad_2level(shape=(rows, cols), seed=8))
    cfg = fq.Config(fmt, fq.RNE)
    rq, _ = fq.fq_quantize(x, cfg)
    y = fq.fq_dequantize(rq, rows, cols, cfg, y_dtype=ydt)
    xhat, _, _, _ = fq.fq_fakequant_ste(x, cfg, xhat_dtype=ydt, want_mask=False)
    torch.cuda.synchronize()
    assert_eq("dequant==fakequant", bits(y), bits(xhat))
    q = {"codes": npy(rq.codes), "scales": npy(rq.scales)}
    if rq.tscale is not None:
        q["tscale"] = npy(rq.tscale)
    ref = oracle.dequantize(q, rows, cols, FMT_O[fmt])
    want = oracle.f32_to_bf16_bits(ref) if ydt == torch.bfloat16 else ref.view(np.uint32)
    assert_eq("dequant", bits(y), want)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ste_backward(dtype):
    rows, cols = 48, 256
    x = _dev(W.nvfp4_act(shape=(rows, cols), seed=3, n_outlier_cols=4).to(dtype))
    dy = _dev(W.normal((rows, cols), 1.0, seed=4).to(dtype))
    _, mask, _, _ = fq.fq_fakequant_ste(x, fq.Config(fq.NVFP4))
    dx = fq.fq_ste_backward(dy, mask)
    torch.cuda.synchronize()
    m = npy(mask)[: (rows * cols + 7) // 8]
    words = np.zeros(((rows * cols + 31) // 32) * 4, np.uint8)
    words[: m.size] = m
    want = oracle.ste_backward(bits(dy), words.view(np.uint32))
    assert_eq("dx", bits(dx), want)


def test_amax_and_amax_in():
    x = _dev(W.nvfp4_act(shape=(512, 1024), seed=6))
    a = fq.fq_amax(x)
    torch.cuda.synchronize()
    assert float(npy(a)[0]) == oracle.amax(as_oracle_input(x))
    # a caller-supplied amax (e.g. delayed scaling) is used as given
    given = torch.tensor([123.5], dtype=torch.float32, device=DEV)
    cfg = fq.Config(fq.NVFP4)
    rq, _ = fq.fq_quantize(x, cfg, amax_in=given)
    torch.cuda.synchronize()
    ref = oracle.quantize(as_oracle_input(x), oracle.NVFP4, amax_in=123.5)
    check_q("row", rq, ref["row"], fq.NVFP4)


# ------------------------------------------------------------------ edge cases
def test_zero_tensor_and_negative_zero():
    for fmt in (fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL):
        x = torch.zeros((128, 256), dtype=torch.bfloat16)   # double block: rows % 128
        x[1] = -0.0
        fakequant_parity(_dev(x), fmt, orient=fq.ROWCOL)


def test_single_row_single_block():
    x = torch.tensor([[0.25, -0.75, 1.25, 5.0, 6.0, -3.5, 0.0, -0.1, 2.5, 1.75, 0.3, -6.0, 3.0,
                       4.4, 0.74, 1.1]], dtype=torch.float32)
    fakequant_parity(_dev(x), fq.NVFP4)
    fakequant_parity(_dev(torch.cat([x, x * 1e-3], 1)), fq.MXFP4)


def test_e4m3_scale_ties_and_saturation():
    """Blocks whose amax is 6 x (an E4M3 midpoint) hit exact scale ties under
    s_g = 1 (a 2688 anchor); others saturate or underflow the scale."""
    vals = [float(oracle.e4m3_value(c)) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    amaxes = [6.0 * m for m in mids] + [6.0 * v for v in vals] + [2688.0, 1e-7, 6 * 2.0 ** -11]
    nb = len(amaxes)
    x = torch.zeros((1, 16 * (nb + 1)), dtype=torch.float32)
    for i, a in enumerate(amaxes):
        x[0, 16 * i] = a
        x[0, 16 * i + 1] = -a * 0.37
        x[0, 16 * i + 2] = a * 0.9
    x[0, 16 * nb] = 2688.0
    fakequant_parity(_dev(x), fq.NVFP4)


def test_saturation_near_six_and_subnormals():
    g = torch.Generator().manual_seed(1)
    x = torch.randn((64, 256), generator=g) * 1e-39          # FP32 subnormals
    x[0] = torch.linspace(-8, 8, 256)
    x[1, ::16] = 6.0
    x[2] = 5.9999995
    fakequant_parity(_dev(x.contiguous()), fq.MXFP4, orient=fq.ROWCOL)
    y = x.clone()
    y[3:] = y[3:] * 1e30                                      # keep NVFP4 amax in range
    fakequant_parity(_dev(y), fq.NVFP4, orient=fq.ROWCOL)
    fakequant_parity(_dev(y), fq.NVFP4, rnd=fq.SR, seed=1, orient=fq.ROWCOL)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("orient", [fq.ROW, fq.ROWCOL])
def test_bf16_subnormal_blocks(fmt, orient):
    """BF16 blocks whose values, and so whose amax, are BF16 subnormals, with
    mixed signs and signed zeros: the BF16 kernels reduce the block amax on
    packed pairs.  One normal value in every row's and every column's
    128-element run keeps the tensor and outer scales normal (MXFP4 scales
    such blocks by 2^127)."""
    g = torch.Generator().manual_seed(7)
    rows, cols = 128, 512
    x = torch.randn((rows, cols), generator=g) * 1e-39
    x[:, 3::16] = -0.0
    x[5, :] = 0.0
    x[1, 0:32] = -2.0 ** -133                    # the smallest BF16 subnormal
    c = torch.arange(cols)
    x[c % rows, c] = torch.where(c % 3 == 0, -1.0, 1.0)
    xb = x.to(torch.bfloat16)
    assert ((xb.float().abs() < 2.0 ** -126) & (xb != 0)).sum() > 10000
    fakequant_parity(_dev(xb), fmt, orient=orient)
    fakequant_parity(_dev(xb), fmt, rnd=fq.SR, seed=3, orient=orient)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("orient", [fq.ROW, fq.ROWCOL])
def test_tiny_tensor_and_outer_scales(dtype, fmt, orient):
    """Tensors (NVFP4) and 1x128 / 128x1 runs (double block) whose amax is
    about 1e-37: the tensor or outer scale amax / 2688 is an FP32 subnormal,
    where the scale codes need the two divisions themselves.  Magnitudes stay
    within a factor 2 of the amax, so every block's s_eff keeps a finite
    reciprocal."""
    g = torch.Generator().manual_seed(11)
    rows, cols = 256, 384
    mag = 0.5 + 0.5 * torch.rand((rows, cols), generator=g)
    sign = torch.where(torch.rand((rows, cols), generator=g) < 0.5, -1.0, 1.0)
    scale = torch.tensor([1e-37, 5e-37, 2.5e-36, 7e-37])[torch.arange(rows) % 4]
    x = (sign * mag * scale[:, None]).to(dtype)
    assert (x != 0).all()
    fakequant_parity(_dev(x), fmt, orient=orient)
    fakequant_parity(_dev(x), fmt, rnd=fq.SR, seed=5, offset=2, orient=orient)


# ------------------------------------------------------------------ Hadamard transform
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt,rnd", [(fq.NVFP4_2LEVEL, fq.SR), (fq.NVFP4_2LEVEL, fq.RNE),
                                     (fq.MXFP4, fq.SR), (fq.MXFP4, fq.RNE)])
def test_rht_row_and_column(dtype, fmt, rnd):
    rows, cols = 256, 384
    x = W.grad_2level(shape=(rows, cols), seed=31).to(dtype)
    x[:, 5] *= 200.0                      # an outlier channel for the transform to spread
    fakequant_parity(_dev(x), fmt, rnd, seed=17, offset=4, orient=fq.ROWCOL, rht_seed=0xC0FFEE)
    fakequant_parity(_dev(x), fmt, rnd, seed=17, offset=4, orient=fq.ROW, rht_seed=99)


def test_rht_rejected_for_per_tensor_nvfp4():
    x = _dev(W.grad_2level(shape=(64, 128), seed=1))
    with pytest.raises(fq.FqError) as e:
        fq.fq_quantize(x, fq.Config(fq.NVFP4, fq.SR, 1, 0, rht_seed=5))
    assert e.value.status == 5


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.slow
def test_full_nvfp4_small_fp32():
    x = W.nvfp4_small()
    fakequant_parity(_dev(x), fq.NVFP4, xhat_dtype=torch.float32)


@pytest.mark.slow
def test_full_mxfp4_weight():
    x = W.mxfp4_weight()
    fakequant_parity(_dev(x), fq.MXFP4, xhat_dtype=torch.bfloat16)


@pytest.mark.slow
def test_full_nvfp4_activation_rowcol():
    x = W.nvfp4_act()
    ref, (xhat, mask, rq, cq) = fakequant_parity(_dev(x), fq.NVFP4, orient=fq.ROWCOL,
                                                 xhat_dtype=torch.bfloat16)
    # the outlier channels' transposed 16x1 blocks carry the largest scales
    cs = npy(cq.scales)
    col_max = cs.max(axis=1)
    assert (np.sort(col_max)[-8:] > np.median(col_max)).all()


@pytest.mark.slow
def test_full_grad_2level_sr_bias():
    x = W.grad_2level()
    ref, (xhat, _, rq, _) = fakequant_parity(_dev(x), fq.NVFP4_2LEVEL, rnd=fq.SR, seed=0x5EED,
                                             xhat_dtype=torch.float32)
    xd = as_oracle_input(x).astype(np.float64)
    bias = abs((npy(xhat).astype(np.float64) - xd).mean()) / np.abs(xd).mean()
    assert bias < 1e-3


@pytest.mark.slow
def test_full_grad_rht_rowcol():
    """The benchmarked backward-operand call at full size: a BF16 [16384, 4096]
    Laplace gradient, 16-point random Hadamard transform, double-block NVFP4
    with stochastic rounding, row and column orientations in one call
    ("Resumo Técnico: TetraJet-v2", §2C and §2A)."""
    x = _dev(W.grad_2level(seed=6))
    cfg = fq.Config(fq.NVFP4_2LEVEL, fq.SR, 0x5EED, 3, rht_seed=0xB00F)
    rq, cq = fq.fq_quantize(x, cfg, orient=fq.ROWCOL)
    torch.cuda.synchronize()
    ref = oracle.quantize(as_oracle_input(x), oracle.NVFP4_2LEVEL, oracle.SR, 0x5EED, 3,
                          orient=oracle.ROWCOL, rht_seed=0xB00F)
    check_q("row", rq, ref["row"], fq.NVFP4_2LEVEL)
    check_q("col", cq, ref["col"], fq.NVFP4_2LEVEL)


@pytest.mark.parametrize("rows", [1, 16, 256, 257])
def test_nvfp4_row_sizes_around_the_small_workload(rows):
    """NVFP4 row-wise fake quantization of 1 to 257 rows of 1024 (the small
    workload is 256 x 1024), FP32 nearest-even and BF16 stochastic."""
    x = W.nvfp4_small(shape=(rows, 1024), seed=40 + rows)
    x[0, 3] = 37.0
    fakequant_parity(_dev(x), fq.NVFP4, xhat_dtype=torch.float32)
    fakequant_parity(_dev(x.to(torch.bfloat16)), fq.NVFP4, rnd=fq.SR, seed=5, offset=2)
