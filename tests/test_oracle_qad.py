"""Pins of the oracle's distillation loss ("Quantization-Aware Distillation
for NVFP4 Inference Accuracy Recovery", §2 Metodologia: KL divergence from
the teacher's to the student's output distribution at softmax temperature 1)
against results fixed outside the oracle: the closed form of two-outcome
distributions, scipy's relative entropy, central finite differences of the
loss, and invariants of softmax and KL."""
import math

import numpy as np
import pytest

import oracle

scipy_special = pytest.importorskip("scipy.special")


def _logits(rows, vocab, seed, scale=3.0, noise=0.3):
    g = np.random.default_rng(seed)
    zt = (g.standard_normal((rows, vocab)) * scale).astype(np.float32)
    zs = (zt + g.standard_normal((rows, vocab)) * noise).astype(np.float32)
    return zt, zs


def test_two_outcome_closed_form():
    """V = 2 with logits (a, 0) and (b, 0): p = sigmoid(a), q = sigmoid(b) and
    KL is the Bernoulli relative entropy; dz = (q - p, p - q) / rows."""
    cases = [(1.0, 0.0), (0.0, 1.0), (-2.5, 3.0), (4.0, 4.0), (7.0, -1.0)]
    zt = np.array([[a, 0.0] for a, _ in cases], np.float32)
    zs = np.array([[b, 0.0] for _, b in cases], np.float32)
    r = oracle.qad_kl(zt, zs)
    n = len(cases)
    for i, (a, b) in enumerate(cases):
        p = 1.0 / (1.0 + math.exp(-a))
        q = 1.0 / (1.0 + math.exp(-b))
        kl = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert r["loss_rows"][i] == pytest.approx(kl, rel=1e-12, abs=1e-15)
        assert r["dz"][i, 0] == pytest.approx((q - p) / n, rel=1e-12, abs=1e-16)
        assert r["dz"][i, 1] == pytest.approx((p - q) / n, rel=1e-12, abs=1e-16)
    assert r["loss_mean"] == pytest.approx(float(np.mean(r["loss_rows"])), rel=1e-15)


def test_asymmetric_direction():
    """KL(p || q) with p the teacher: swapping the operands changes the value."""
    zt = np.array([[3.0, 0.0, -1.0]], np.float32)
    zs = np.array([[0.0, 0.5, 0.0]], np.float32)
    fwd = oracle.qad_kl(zt, zs)["loss_rows"][0]
    rev = oracle.qad_kl(zs, zt)["loss_rows"][0]
    p = scipy_special.softmax(zt[0].astype(np.float64))
    q = scipy_special.softmax(zs[0].astype(np.float64))
    assert fwd == pytest.approx(float(np.sum(p * np.log(p / q))), rel=1e-12)
    assert abs(fwd - rev) > 0.1


@pytest.mark.parametrize("vocab", [5, 1000, 32000])
def test_matches_scipy_relative_entropy(vocab):
    zt, zs = _logits(4, vocab, seed=vocab)
    r = oracle.qad_kl(zt, zs)
    for i in range(4):
        p = scipy_special.softmax(zt[i].astype(np.float64))
        q = scipy_special.softmax(zs[i].astype(np.float64))
        want = float(np.sum(scipy_special.rel_entr(p, q)))
        assert r["loss_rows"][i] == pytest.approx(want, rel=1e-10, abs=1e-15)
        np.testing.assert_allclose(r["dz"][i], (q - p) / 4, rtol=1e-10, atol=1e-18)


def test_gradient_by_finite_differences():
    """dz is the derivative of g * KL_r with respect to the student logits."""
    zt, zs = _logits(3, 7, seed=3, scale=1.5, noise=0.8)
    g = 0.37
    r = oracle.qad_kl(zt, zs, temperature=1.3, grad_scale=g)
    h = 1e-3
    # central differences of the oracle's float64 loss along each coordinate; the
    # logits are FP32 inputs, so step by an exactly representable h
    for i in range(3):
        for v in range(7):
            up, dn = zs.copy(), zs.copy()
            up[i, v] += np.float32(h)
            dn[i, v] -= np.float32(h)
            hh = (float(up[i, v]) - float(dn[i, v])) / 2
            fu = oracle.qad_kl(zt, up, temperature=1.3)["loss_rows"][i]
            fd = oracle.qad_kl(zt, dn, temperature=1.3)["loss_rows"][i]
            num = g * (fu - fd) / (2 * hh)
            assert r["dz"][i, v] == pytest.approx(num, rel=1e-5, abs=1e-9)


def test_identical_distributions():
    zt, _ = _logits(3, 257, seed=4)
    r = oracle.qad_kl(zt, zt.copy())
    assert np.all(r["loss_rows"] == 0.0)
    assert np.all(r["dz"] == 0.0)


def test_shift_invariance_and_nonnegativity():
    zt, zs = _logits(5, 300, seed=5)
    # logits on a 2^-10 grid below 2^10 in magnitude, so that the shifts are exact
    zt, zs = (np.round(z * 1024) / 1024 for z in (zt, zs))
    base = oracle.qad_kl(zt, zs)
    shifted = oracle.qad_kl(zt + np.float32(8.0), zs - np.float32(16.0))
    np.testing.assert_allclose(shifted["loss_rows"], base["loss_rows"], rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(shifted["dz"], base["dz"], rtol=1e-9, atol=1e-18)
    assert np.all(base["loss_rows"] > 0.0)
    np.testing.assert_allclose(base["dz"].sum(axis=1), 0.0, atol=1e-15)
    # logits near 1000 overflow exp() in float64 unless the maximum is taken out
    big = oracle.qad_kl(zt + np.float32(1000.0), zs + np.float32(992.0))
    np.testing.assert_allclose(big["loss_rows"], base["loss_rows"], rtol=1e-9, atol=1e-15)


def test_temperature_scales_the_logits():
    """T divides the logits, and the gradient carries a further 1 / T."""
    zt = np.array([[2.0, -4.0, 6.0, 0.5]], np.float32)
    zs = np.array([[1.0, -2.0, 8.0, 0.0]], np.float32)
    t2 = oracle.qad_kl(zt, zs, temperature=2.0)
    t1 = oracle.qad_kl(zt / 2, zs / 2, temperature=1.0)   # halving is exact
    assert t2["loss_rows"][0] == pytest.approx(t1["loss_rows"][0], rel=1e-14)
    np.testing.assert_allclose(t2["dz"], t1["dz"] / 2, rtol=1e-13)


def test_one_hot_teacher_is_cross_entropy():
    """A teacher whose distribution is (numerically) one-hot reduces KL to the
    student's cross entropy on that class, the task loss that QAT uses."""
    zs = np.array([[0.3, -1.2, 2.0, 0.0]], np.float32)
    zt = np.array([[-200.0, -200.0, 200.0, -200.0]], np.float32)
    r = oracle.qad_kl(zt, zs)
    ce = -float(scipy_special.log_softmax(zs[0].astype(np.float64))[2])
    assert r["loss_rows"][0] == pytest.approx(ce, rel=1e-12)
