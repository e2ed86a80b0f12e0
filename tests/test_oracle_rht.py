"""Pins for the oracle's 16-point randomized Hadamard transform (CPU only):
scipy's Sylvester Hadamard matrix in binary64, exactness on dyadic inputs,
involution, norm preservation and the GEMM invariance that motivates it
("Resumo Técnico: TetraJet-v2", §2C)."""
import numpy as np
import pytest
from scipy.linalg import hadamard

import oracle

RNG = np.random.default_rng(99)
H16 = hadamard(16).astype(np.float64)


def _d(signs):
    return np.array([-1.0 if (signs >> i) & 1 else 1.0 for i in range(16)])


@pytest.mark.parametrize("signs", [0, 0xFFFF, 0xA5C3, oracle.rht_signs(7, 0)])
def test_rht16_is_scaled_hadamard_of_signed_input(signs):
    # dyadic inputs: every FP32 step is exact, so the result equals binary64
    x = RNG.integers(-64, 65, size=16).astype(np.float32) / 8
    got = oracle.rht16(x, signs).astype(np.float64)
    want = 0.25 * (H16 @ (_d(signs) * x.astype(np.float64)))
    assert np.array_equal(got, want)
    # general inputs: within the rounding of four FP32 additions
    y = RNG.standard_normal(16).astype(np.float32)
    got = oracle.rht16(y, signs).astype(np.float64)
    want = 0.25 * (H16 @ (_d(signs) * y.astype(np.float64)))
    assert np.max(np.abs(got - want)) <= 4 * 2.0 ** -23 * np.abs(y).sum()


def test_rht16_inverse_and_norm():
    signs = oracle.rht_signs(1234, 5)
    x = RNG.integers(-100, 101, size=16).astype(np.float32) / 16
    z = oracle.rht16(x, signs)
    back = oracle.rht16(z, 0) * _d(signs).astype(np.float32)   # (1/4 H) is its own inverse
    assert np.array_equal(back, x)
    y = RNG.standard_normal(16).astype(np.float32)
    zy = oracle.rht16(y, signs).astype(np.float64)
    assert abs(np.linalg.norm(zy) - np.linalg.norm(y.astype(np.float64))) < 1e-5


def test_rht_signs_come_from_philox():
    for seed, off in [(1, 0), (7, 3), (0xFFFFFFFF, 12345)]:
        out = oracle.philox4x32_10([0, 0, 2, off], [seed, 0])
        assert oracle.rht_signs(seed, off) == out[0] & 0xFFFF


def test_rht_keeps_gemm_products():
    """Transforming both operands along the reduction dimension with the same
    signs leaves A @ B^T unchanged (the transform is orthogonal)."""
    a = RNG.standard_normal((8, 64)).astype(np.float32)
    b = RNG.standard_normal((5, 64)).astype(np.float32)
    ta = oracle.rht_rows(a, 42, 1).astype(np.float64)
    tb = oracle.rht_rows(b, 42, 1).astype(np.float64)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    assert np.allclose(ta @ tb.T, ref, atol=1e-4)
    # different signs do not
    tc = oracle.rht_rows(b, 43, 1).astype(np.float64)
    assert not np.allclose(ta @ tc.T, ref, atol=1e-2)


def test_rht_spreads_an_outlier():
    x = np.zeros((1, 16), np.float32)
    x[0, 3] = 64.0
    z = oracle.rht_rows(x, 9, 0)
    assert np.allclose(np.abs(z), 16.0)        # one spike becomes 16 equal magnitudes


def test_rht_quantize_column_is_row_of_transpose():
    x = RNG.standard_normal((128, 256)).astype(np.float32)
    r = oracle.quantize(x, oracle.NVFP4_2LEVEL, oracle.SR, seed=3, orient=oracle.ROWCOL,
                        rht_seed=11)
    t = oracle.quantize(np.ascontiguousarray(x.T), oracle.NVFP4_2LEVEL, oracle.SR, seed=3,
                        orient=oracle.ROW, rht_seed=11)["row"]
    # the column pass uses stream 1 for SR, so compare with RNE for equality of the transform
    r2 = oracle.quantize(x, oracle.NVFP4_2LEVEL, oracle.RNE, orient=oracle.COL, rht_seed=11)
    t2 = oracle.quantize(np.ascontiguousarray(x.T), oracle.NVFP4_2LEVEL, oracle.RNE,
                         rht_seed=11)["row"]
    assert np.array_equal(r2["col"]["codes"], t2["codes"])
    assert np.array_equal(r2["col"]["scales"], t2["scales"])
    assert r["col"]["codes"].shape == t["codes"].shape
