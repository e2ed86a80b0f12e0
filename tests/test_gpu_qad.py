"""The QAD distillation loss on the GPU against the float64 oracle
("Quantization-Aware Distillation for NVFP4 Inference Accuracy Recovery", §2
Metodologia: KL(teacher || student) at softmax temperature T, and its
student-logit gradient).

The kernel computes in FP32, so results are compared within bounds derived
from its rounding:
  loss_rows  |KL - KL_ref| <= 2e-5 + 1e-4 KL_ref.  The row's log-sum-exp
             difference enters KL one for one; its error is a few units of
             2^-24 times the number of terms each thread sums (about 50) plus
             the exponent arguments' rounding (|lse2| ~ 20): below 1e-5.
  dz         |dz - dz_ref| <= |g| / T ((p + q) 2^-15 + 2^-126), plus 2^-8 |dz_ref| when
             the gradient is stored in BF16: p and q carry a relative error of
             at most about 2^-17 (exponent arguments, exp2f's 2 ulp, the sums),
             and rounding to BF16 moves a value by at most 2^-9 relative.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import as_oracle_input, npy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _softmax64(z, T):
    a = z.astype(np.float64) / T
    a -= a.max(axis=1, keepdims=True)
    e = np.exp(a)
    return e / e.sum(axis=1, keepdims=True)


def _check(zt, zs, T=1.0, g=None, dz_dtype=None, rows_sel=None, out=None):
    """Run the kernel on device logits zt, zs and compare the selected rows
    (all by default) with the oracle."""
    rows, vocab = zt.shape
    if out is None:
        out = fq.fq_qad_kl(zt, zs, temperature=T, grad_scale=g, dz_dtype=dz_dtype)
    loss, mean, dz, err = out
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    sel = np.arange(rows) if rows_sel is None else np.asarray(rows_sel)
    st = torch.as_tensor(sel, device=zt.device)
    xt = as_oracle_input(zt[st].contiguous())
    xs = as_oracle_input(zs[st].contiguous())
    gg = (1.0 / rows) if g is None else g
    ref = oracle.qad_kl(xt, xs, temperature=T, grad_scale=gg)
    got = npy(loss)[sel].astype(np.float64)
    want = ref["loss_rows"]
    bad = ~(np.abs(got - want) <= 2e-5 + 1e-4 * np.abs(want))  # NaN fails too
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], want[bad][:5])
    if rows_sel is None:
        m = float(npy(mean)[0])
        assert abs(m - ref["loss_mean"]) <= 2e-5 + 1e-4 * abs(ref["loss_mean"])
    if dz is not None:
        gd = npy(dz[st].float()).astype(np.float64)
        p, q = _softmax64(xt, T), _softmax64(xs, T)
        # (values below FP32's normal range may come out flushed: 2^-126 floor)
        tol = abs(gg) / T * ((p + q) * 2.0 ** -15 + 2.0 ** -126)
        if dz.dtype == torch.bfloat16:
            tol = tol + 2.0 ** -8 * np.abs(ref["dz"])
        bad = ~(np.abs(gd - ref["dz"]) <= tol)
        assert not bad.any(), (np.argwhere(bad)[:5], gd[bad][:5], ref["dz"][bad][:5])
    return out, ref


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,vocab", [(3, 8), (5, 1000), (7, 32000), (4, 40000), (3, 201088)])
def test_qad_kl_shapes(dtype, rows, vocab):
    """Cluster sizes 1, 2, 4 and 8 (the chunk of a row per CTA shrinks with
    the vocabulary), chunks whose length is not a multiple of the sweep."""
    zt, zs = W.qad_logits((rows, vocab), seed=rows + vocab, dtype=dtype)
    _check(zt.to(DEV), zs.to(DEV))


@pytest.mark.parametrize("dz_dtype", [torch.float32, torch.bfloat16])
def test_qad_kl_temperature_scale_and_gradient_dtype(dz_dtype):
    zt, zs = W.qad_logits((9, 4096), seed=3, dtype=torch.bfloat16)
    _check(zt.to(DEV), zs.to(DEV), T=2.0, g=0.5, dz_dtype=dz_dtype)
    _check(zt.to(DEV), zs.to(DEV), T=0.7, g=-3.0, dz_dtype=dz_dtype)


def test_qad_kl_many_rows_per_cluster():
    """More rows than clusters on the GPU: the persistent loop and the
    next-row prefetch run many times per cluster."""
    zt, zs = W.qad_logits((1500, 1024), seed=4, dtype=torch.bfloat16)
    _check(zt.to(DEV), zs.to(DEV))


def test_qad_kl_identical_and_peaked():
    zt, _ = W.qad_logits((6, 2048), seed=5, dtype=torch.float32)
    zt[0, 17] = 80.0                    # nearly one-hot teacher row
    zt[1] = 0.0                         # uniform row
    out, ref = _check(zt.to(DEV), zt.clone().to(DEV))
    assert np.all(np.abs(npy(out[0])) <= 2e-5)
    zs = zt.clone()
    zs[0, 17] = 70.0
    zs[2] += 1000.0                     # large logits (the oracle sees the same rounded values)
    _check(zt.to(DEV), zs.to(DEV))


def test_qad_kl_forward_only_and_empty():
    zt, zs = W.qad_logits((4, 512), seed=6, dtype=torch.bfloat16)
    _check(zt.to(DEV), zs.to(DEV), out=fq.fq_qad_kl(zt.to(DEV), zs.to(DEV), want_grad=False))
    e = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    loss, mean, dz, err = fq.fq_qad_kl(e, e)
    torch.cuda.synchronize()
    assert loss.numel() == 0 and float(mean.item()) == 0.0 and int(err.item()) == 0


@pytest.mark.slow
def test_full_qad_logits_sampled_rows():
    """4096 x 201088 BF16 logits (the benchmarked call): 32 rows spread over
    the tensor against the oracle, and on every row KL >= 0 and the gradient
    summing to about zero."""
    c = W.WORKLOADS["qad_logits"]
    zt, zs = W.qad_logits(c["shape"], seed=c["seed"], device=DEV)
    rows = c["shape"][0]
    sel = np.linspace(0, rows - 1, 32).astype(np.int64)
    out, _ = _check(zt, zs, rows_sel=sel)
    loss, mean, dz, _ = out
    assert bool((loss >= -2e-5).all())
    # sum_v (q - p) = 0; BF16 rounding moves each term by at most 2^-9 of
    # |dz| <= (p + q) / rows, so a row sums to at most 2^-8 / rows
    rowsum = dz.float().sum(dim=1).abs()
    assert float(rowsum.max()) <= 2.0 ** -8 / rows
