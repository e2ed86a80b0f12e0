"""Pins of the oracle's block-scaled FP4 GEMM (C = deq(A) deq(B)^T, the
forward GEMM of a QAT linear layer on NVFP4 / MXFP4 operands: "Aprimorando
gpt-oss para Precisão e Desempenho com Treinamento Consciente à
Quantização", "O que há de novo"; "Resumo Técnico: TetraJet-v2", §2A)
against brute force, exactly representable operands, and exact scalings."""
import numpy as np
import pytest

import oracle


def _q(x, fmt):
    r = oracle.quantize(np.ascontiguousarray(x, np.float32), fmt)["row"]
    return {k: r[k] for k in ("codes", "scales", "tscale") if k in r}


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_brute_force_small(fmt):
    g = np.random.default_rng(1)
    m, n, k = 3, 5, 64
    a = g.standard_normal((m, k)).astype(np.float32)
    b = g.standard_normal((n, k)).astype(np.float32)
    qa, qb = _q(a, fmt), _q(b, fmt)
    c = oracle.gemm(qa, qb, m, n, k, fmt)
    da = oracle.dequantize(qa, m, k, fmt)
    db = oracle.dequantize(qb, n, k, fmt)
    for i in range(m):
        for j in range(n):
            want = 0.0
            for t in range(k):
                want += float(da[i, t]) * float(db[j, t])
            assert c[i, j] == pytest.approx(want, rel=1e-12, abs=1e-12)


def test_exact_grid_operands_mxfp4():
    """Values on the E2M1 grid with a +-6 in every 1x32 block quantize
    exactly under MXFP4 (scale 2^0), so the GEMM is the exact product of the
    inputs."""
    g = np.random.default_rng(2)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    m, n, k = 8, 6, 128

    def draw(r):
        x = grid[g.integers(0, 8, (r, k))] * np.where(g.random((r, k)) < 0.5, -1, 1)
        x[:, ::32] = 6.0
        return x.astype(np.float32)
    a, b = draw(m), draw(n)
    c = oracle.gemm(_q(a, oracle.MXFP4), _q(b, oracle.MXFP4), m, n, k, oracle.MXFP4)
    assert np.array_equal(c, a.astype(np.float64) @ b.astype(np.float64).T)


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4])
def test_power_of_two_scaling(fmt):
    """Scaling an operand by 2^e moves only its scales, so C scales by 2^e."""
    g = np.random.default_rng(3)
    m, n, k = 16, 8, 256
    a = g.standard_normal((m, k)).astype(np.float32)
    b = (g.standard_normal((n, k)) * 0.01).astype(np.float32)
    c = oracle.gemm(_q(a, fmt), _q(b, fmt), m, n, k, fmt)
    c8 = oracle.gemm(_q(a * np.float32(8.0), fmt), _q(b, fmt), m, n, k, fmt)
    assert np.array_equal(c8, c * 8.0)


def test_transposed_roles():
    """C(B, A) is C(A, B) transposed."""
    g = np.random.default_rng(4)
    a = g.standard_normal((4, 64)).astype(np.float32)
    b = g.standard_normal((7, 64)).astype(np.float32)
    qa, qb = _q(a, oracle.NVFP4), _q(b, oracle.NVFP4)
    assert np.allclose(oracle.gemm(qa, qb, 4, 7, 64), oracle.gemm(qb, qa, 7, 4, 64).T,
                       rtol=1e-14, atol=0)
