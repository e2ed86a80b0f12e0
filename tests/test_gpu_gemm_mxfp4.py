"""MXFP4 block-scaled GEMM on the tensor cores (E8M0 scales per 1x32 block,
scale_vec::2X) against the oracle (the float64 product of the dequantized
operands; "Aprimorando gpt-oss para Precisão e Desempenho com Treinamento
Consciente à Quantização", "O que há de novo": MXFP4).  Bound as for NVFP4:
|C - C_ref| <= 2^-16 sum_k |deq(a)_mk deq(b)_nk| (+ 2^-8 |C_ref| for BF16 C);
the power-of-two scales make the products exact."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import npy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _qd(q):
    return {"codes": npy(q.codes), "scales": npy(q.scales)}


def _run(a, b, c_dtype=torch.float32):
    m, k = a.shape
    n = b.shape[0]
    cfg = fq.Config(fq.MXFP4)
    qa, _ = fq.fq_quantize(a.to(DEV), cfg)
    qb, _ = fq.fq_quantize(b.to(DEV), cfg)
    c, err = fq.fq_gemm(qa, qb, m, n, k, cfg, c_dtype=c_dtype)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.gemm(_qd(qa), _qd(qb), m, n, k, oracle.MXFP4)
    da = oracle.dequantize(_qd(qa), m, k, oracle.MXFP4).astype(np.float64)
    db = oracle.dequantize(_qd(qb), n, k, oracle.MXFP4).astype(np.float64)
    bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T)
    if c_dtype == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(ref)
    got = npy(c.float()).astype(np.float64)
    bad = ~(np.abs(got - ref) <= bound)  # NaN fails too
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:4], got[bad][:4], ref[bad][:4])
    return qa, qb


def test_mxfp4_gemm_uniform_block_scales():
    """Every 1x32 block has the same amax, so every E8M0 code is equal: the
    result does not depend on where the scales sit."""
    g = torch.Generator().manual_seed(21)
    a = torch.randn((128, 256), generator=g).clamp(-2.5, 2.5)
    b = torch.randn((128, 256), generator=g).clamp(-2.5, 2.5)
    a[:, ::32] = 3.0
    b[:, ::32] = -3.0
    qa, qb = _run(a, b)
    assert len(np.unique(npy(qa.scales))) == 1 and len(np.unique(npy(qb.scales))) == 1


def test_mxfp4_gemm_varied_scales():
    """Block amaxes spread over many binades (rows and 1x32 blocks scaled by
    powers of two), so each scale must reach its own block."""
    m, n, k = 256, 384, 1024
    a = W.normal((m, k), 1.0, seed=22)
    b = W.mxfp4_weight(shape=(n, k), seed=23).float()
    ga = torch.Generator().manual_seed(24)
    a = a * torch.pow(2.0, torch.randint(-6, 7, (m, k // 32), generator=ga).float()
                      ).repeat_interleave(32, dim=1)
    _run(a, b)


def test_mxfp4_gemm_bf16_output_long_k():
    _run(W.normal((128, 4096), 0.5, seed=25), W.normal((256, 4096), 0.02, seed=26),
         c_dtype=torch.bfloat16)


@pytest.mark.parametrize("m,n,k", [(200, 160, 2880), (3, 64, 96)])
def test_mxfp4_gemm_shapes_off_the_tile_grid(m, n, k):
    _run(W.normal((m, k), 1.0, seed=m), W.normal((n, k), 0.02, seed=n))
