"""Block-scaled FP4 GEMM on the tensor cores against the oracle (the float64
product of the dequantized operands; "Aprimorando gpt-oss para Precisão e
Desempenho com Treinamento Consciente à Quantização", "O que há de novo";
"Resumo Técnico: TetraJet-v2", §2A).

The products of FP4 values and E4M3 scales are exact in FP32; the tensor
cores accumulate them in FP32, and the tensor scales multiply the result
once.  So |C - C_ref| <= 2^-16 sum_k |deq(a)_mk deq(b)_nk| (about 2^-24 per
accumulation step, with room for the 256-element K-tiles), plus half a BF16
ulp (2^-8 |C_ref|, with margin) when C is stored in BF16."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import npy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _qdict(q):
    return {"codes": npy(q.codes), "scales": npy(q.scales), "tscale": npy(q.tscale)[:1]}


def _check(m, n, k, seed, c_dtype=torch.float32, a_scale=1.0):
    a = (W.normal((m, k), a_scale, seed=seed) ).to(DEV)
    b = W.normal((n, k), 0.02, seed=seed + 1).to(DEV)
    cfg = fq.Config(fq.NVFP4)
    qa, _ = fq.fq_quantize(a, cfg)
    qb, _ = fq.fq_quantize(b, cfg)
    c, err = fq.fq_gemm(qa, qb, m, n, k, c_dtype=c_dtype)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    da = oracle.dequantize(_qdict(qa), m, k).astype(np.float64)
    db = oracle.dequantize(_qdict(qb), n, k).astype(np.float64)
    ref = oracle.gemm(_qdict(qa), _qdict(qb), m, n, k)
    bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T)
    if c_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(ref)
    got = npy(c.float()).astype(np.float64)
    bad = ~(np.abs(got - ref) <= bound)  # NaN fails too
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4], got[bad][:4], ref[bad][:4])
    return got, ref


def test_gemm_uniform_block_scales():
    """Every 1x16 block of both operands has the same amax (hence the same
    E4M3 scale code): the result does not depend on where the scales sit, so
    this isolates the code operands from the scale layout."""
    m, n, k = 128, 128, 256
    g = torch.Generator().manual_seed(11)
    a = torch.randn((m, k), generator=g).clamp(-2.5, 2.5)
    b = torch.randn((n, k), generator=g).clamp(-2.5, 2.5)
    a[:, ::16] = 3.0
    b[:, ::16] = -3.0
    cfg = fq.Config(fq.NVFP4)
    qa, _ = fq.fq_quantize(a.to(DEV), cfg)
    qb, _ = fq.fq_quantize(b.to(DEV), cfg)
    assert len(np.unique(npy(qa.scales))) == 1 and len(np.unique(npy(qb.scales))) == 1
    c, err = fq.fq_gemm(qa, qb, m, n, k)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.gemm(_qdict(qa), _qdict(qb), m, n, k)
    da = oracle.dequantize(_qdict(qa), m, k).astype(np.float64)
    db = oracle.dequantize(_qdict(qb), n, k).astype(np.float64)
    bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T)
    got = npy(c).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound), (got[:2, :4], ref[:2, :4])


def test_gemm_one_tile():
    _check(128, 128, 256, seed=1)


def test_gemm_several_tiles_and_k_tiles():
    _check(256, 384, 1024, seed=2)


def test_gemm_bf16_output_and_scale():
    _check(384, 256, 2048, seed=3, c_dtype=torch.bfloat16, a_scale=30.0)


def test_gemm_long_k():
    _check(128, 256, 8192, seed=4)


def test_gemm_many_tiles():
    """Several times more tiles than CTAs fit on the GPU at once: the tiles
    run in waves, and each new CTA allocates and frees its tensor memory."""
    _check(2560, 4096, 512, seed=5)


@pytest.mark.slow
def test_full_gemm_8192_sampled_rows():
    """The benchmarked 8192^3 product: 48 rows of C spread over all row
    blocks against the oracle (all columns)."""
    m = n = k = 8192
    a = W.normal((m, k), 1.0, seed=20, dtype=torch.bfloat16, device=DEV)
    b = W.normal((n, k), 0.02, seed=21, dtype=torch.bfloat16, device=DEV)
    cfg = fq.Config(fq.NVFP4)
    qa, _ = fq.fq_quantize(a, cfg)
    qb, _ = fq.fq_quantize(b, cfg)
    c, err = fq.fq_gemm(qa, qb, m, n, k, c_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = np.linspace(0, m - 1, 48).astype(np.int64)
    rt = torch.as_tensor(rows, device=DEV)
    qsub = {"codes": npy(qa.codes[rt]), "scales": npy(qa.scales[rt]), "tscale": npy(qa.tscale)[:1]}
    ref = oracle.gemm(qsub, _qdict(qb), len(rows), n, k)
    da = oracle.dequantize(qsub, len(rows), k).astype(np.float64)
    db = oracle.dequantize(_qdict(qb), n, k).astype(np.float64)
    bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T) + 2.0 ** -8 * np.abs(ref)
    got = npy(c[rt].float()).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)


def test_qat_linear_layer_three_gemms():
    """The three GEMMs of a QAT linear layer Y = X W^T from the quantizers'
    own outputs: forward Y = deq(X) deq(W)^T from the row-wise codes; the input
    gradient dX = deq(dY) deq(W^T)^T with W^T from the column-wise pass of W;
    the weight gradient dW = deq(dY^T) deq(X^T)^T from the column-wise passes
    of dY and X ("Resumo Técnico: TetraJet-v2", §2A: 1x16 groups and the
    transposed operands of the backward pass)."""
    m, n, k = 256, 512, 768           # tokens, output features, input features
    cfg = fq.Config(fq.NVFP4)
    x = W.nvfp4_act(shape=(m, k), seed=30, n_outlier_cols=2).to(DEV)
    w = W.normal((n, k), 0.02, seed=31, dtype=torch.bfloat16, device=DEV)
    dy = W.grad_2level(shape=(m, n), seed=32).to(DEV)
    xr, xc = fq.fq_quantize(x, cfg, orient=fq.ROWCOL)      # X [m,k] and X^T [k,m]
    wr, wc = fq.fq_quantize(w, cfg, orient=fq.ROWCOL)      # W [n,k] and W^T [k,n]
    dr, dc = fq.fq_quantize(dy, cfg, orient=fq.ROWCOL)     # dY [m,n] and dY^T [n,m]
    cases = [("Y", xr, wr, m, n, k), ("dX", dr, wc, m, k, n), ("dW", dc, xc, n, k, m)]
    for name, qa, qb, mm, nn, kk in cases:
        c, err = fq.fq_gemm(qa, qb, mm, nn, kk)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, name
        ref = oracle.gemm(_qdict(qa), _qdict(qb), mm, nn, kk)
        da = oracle.dequantize(_qdict(qa), mm, kk).astype(np.float64)
        db = oracle.dequantize(_qdict(qb), nn, kk).astype(np.float64)
        bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T)
        got = npy(c).astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound), name


@pytest.mark.parametrize("m,n,k", [(200, 160, 2880), (1, 32, 32), (130, 96, 544),
                                   (256, 5760, 2880)])
def test_gemm_shapes_off_the_tile_grid(m, n, k):
    """m free, n and k multiples of 32: the parts of the 128 x 128 x 256 tiles
    past the operands are zero-filled (gpt-oss's 2880 and 5760 included)."""
    _check(m, n, k, seed=m + n + k)
