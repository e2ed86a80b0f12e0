"""Tensor-level pins for the oracle (CPU only).

1. An independent vectorised restatement built on library primitives (torch's
   float8_e4m3fn cast for the E4M3 scale, numpy.frexp for the E8M0 exponent, a
   threshold ladder for E2M1 instead of the oracle's brute-force search) must
   agree bit-for-bit with the oracle on random tensors.
2. Invariants of the method: grid round trip, range and error bounds, the
   double-block / per-tensor equivalence, stochastic-rounding unbiasedness.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import workloads

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)


def _e4m3_from_torch(s):
    t = torch.from_numpy(np.ascontiguousarray(s, dtype=np.float32))
    c = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.uint8)
    c = np.where(s >= 448.0, np.uint8(0x7E), c)
    v = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    return c, v


def _ladder(a):
    return ((a > 0.25).astype(np.int32) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
            + (a > 2.5) + (a >= 3.5) + (a > 5.0))


def vectorised(x, fmt):
    rows, cols = x.shape
    B = 32 if fmt == oracle.MXFP4 else 16
    xb = x.reshape(rows, cols // B, B)
    amax_b = np.abs(xb).max(-1).astype(np.float32)
    out = {}
    with np.errstate(divide="ignore", invalid="ignore"):
        if fmt == oracle.MXFP4:
            _, e = np.frexp(amax_b)
            k = np.where(amax_b == 0, -127, np.clip(e - 1 - 2, -127, 127))
            sc = (k + 127).astype(np.uint8)
            s_eff = np.ldexp(np.float32(1), k).astype(np.float32)
            r = np.ldexp(np.float32(1), -k).astype(np.float32)
        else:
            if fmt == oracle.NVFP4:
                s_outer = np.full(amax_b.shape, np.float32(np.abs(x).max()) / np.float32(2688),
                                  dtype=np.float32)
                out["tscale"] = s_outer.reshape(-1)[:1]
            else:
                a128 = np.abs(x.reshape(rows, cols // 128, 128)).max(-1).astype(np.float32)
                s_o = (a128 / np.float32(2688)).astype(np.float32)
                out["tscale"] = s_o
                s_outer = np.repeat(s_o, 8, axis=1)
            s_b = np.where(s_outer == 0, np.float32(0), (amax_b / np.float32(6)) / s_outer)
            s_b = s_b.astype(np.float32)
            sc, sv = _e4m3_from_torch(s_b)
            s_eff = (sv * s_outer).astype(np.float32)
            r = np.where(s_eff == 0, np.float32(0), np.float32(1) / s_eff).astype(np.float32)
    y = (xb * r[..., None]).astype(np.float32)
    mag = _ladder(np.abs(y))
    code = (mag + 8 * np.signbit(y)).astype(np.uint8)
    xhat = (np.where(np.signbit(y), -GRID[mag], GRID[mag]) * s_eff[..., None]).astype(np.float32)
    mask_bits = (np.abs(xb) <= (np.float32(6) * s_eff)[..., None]).reshape(-1)
    flat = code.reshape(-1)
    out["codes"] = (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8).reshape(rows, cols // 2)
    out["scales"] = sc.reshape(rows, cols // B)
    out["xhat"] = xhat.reshape(rows, cols)
    pad = (-mask_bits.size) % 32
    mb = np.concatenate([mask_bits, np.zeros(pad, bool)]).reshape(-1, 32).astype(np.uint64)
    out["mask"] = (mb << np.arange(32, dtype=np.uint64)).sum(-1).astype(np.uint32)
    return out


def _test_tensor(rows=48, cols=512, seed=0):
    g = np.random.default_rng(seed)
    x = g.standard_normal((rows, cols)).astype(np.float32)
    x[3, :] *= 300.0                               # a loud row
    x[:, 7] *= 50.0                                # an outlier channel
    x[5, 16:32] = 0.0                              # an all-zero 16-block
    x[6, 0:128] = -0.0                             # an all-negative-zero 128-block
    x[7, 40] = 1e-39                               # a subnormal input
    x[9, :] *= 1e-6
    return x


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL])
def test_oracle_matches_vectorised_restatement(fmt):
    x = _test_tensor()
    got = oracle.quantize(x, fmt, want_xhat=True, want_mask=True)["row"]
    ref = vectorised(x, fmt)
    for k in ("codes", "scales", "mask"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["xhat"].view(np.uint32), ref["xhat"].view(np.uint32))
    if fmt != oracle.MXFP4:
        assert np.array_equal(got["tscale"].reshape(-1).view(np.uint32),
                              ref["tscale"].reshape(-1).view(np.uint32))


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.NVFP4_2LEVEL])
def test_oracle_matches_vectorised_restatement_tiny_scales(fmt):
    """Tensor and outer amax near 1e-37: the tensor / outer scale amax / 2688
    is an FP32 subnormal, where the scale code rests on IEEE division with
    gradual underflow.  Magnitudes within a factor 2 of each row's scale keep
    every block's s_eff reciprocal finite."""
    g = np.random.default_rng(11)
    rows, cols = 64, 256
    mag = 0.5 + 0.5 * g.random((rows, cols))
    sign = np.where(g.random((rows, cols)) < 0.5, -1.0, 1.0)
    scale = np.array([1e-37, 5e-37, 2.5e-36, 7e-37])[np.arange(rows) % 4]
    x = (sign * mag * scale[:, None]).astype(np.float32)
    got = oracle.quantize(x, fmt, want_xhat=True, want_mask=True)["row"]
    assert np.min(got["tscale"]) < np.finfo(np.float32).tiny        # subnormal scales
    ref = vectorised(x, fmt)
    for k in ("codes", "scales", "mask"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["xhat"].view(np.uint32), ref["xhat"].view(np.uint32))
    assert np.array_equal(got["tscale"].reshape(-1).view(np.uint32),
                          ref["tscale"].reshape(-1).view(np.uint32))


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL])
def test_oracle_matches_vectorised_restatement_subnormal_blocks(fmt):
    """Blocks of FP32 subnormals with signed zeros, under normal tensor and
    outer scales (one value of 1 in every row's 128-run): MXFP4 scales them by
    2^127, the E4M3 formats give them a zero scale."""
    g = np.random.default_rng(7)
    rows, cols = 32, 256
    x = (g.standard_normal((rows, cols)) * 1e-39).astype(np.float32)
    x[:, 3::16] = -0.0
    x[2, 0:32] = -np.float32(2.0 ** -149)
    c = np.arange(cols)
    x[c % rows, c] = 1.0
    assert ((np.abs(x) < np.finfo(np.float32).tiny) & (x != 0)).sum() > 5000
    got = oracle.quantize(x, fmt, want_xhat=True, want_mask=True)["row"]
    ref = vectorised(x, fmt)
    for k in ("codes", "scales", "mask"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["xhat"].view(np.uint32), ref["xhat"].view(np.uint32))


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL])
def test_dequantize_reproduces_quantizer_xhat(fmt):
    x = _test_tensor(seed=3)
    q = oracle.quantize(x, fmt, want_xhat=True)["row"]
    xh = oracle.dequantize(q, *x.shape, fmt=fmt)
    assert np.array_equal(xh.view(np.uint32), q["xhat"].view(np.uint32))


def test_grid_roundtrip_mxfp4_and_unit_scale_nvfp4():
    """I1: a block made of grid values times a representable scale quantizes
    back to the same codes and scale."""
    g = np.random.default_rng(7)
    codes = g.integers(0, 16, size=(32, 256))
    codes[:, ::16] = 7                       # every 16-block holds +6 (defines the scale)
    vals = np.array([oracle.e2m1_value(int(c)) for c in range(16)], dtype=np.float32)
    k = g.integers(-20, 20, size=(32, 8))
    x = (vals[codes] * np.ldexp(np.float32(1), np.repeat(k, 32, axis=1))).astype(np.float32)
    q = oracle.quantize(x, oracle.MXFP4, want_xhat=True)["row"]
    assert np.array_equal(q["xhat"], x)
    assert np.array_equal(q["scales"], (k + 127).astype(np.uint8))
    # NVFP4 with s_g = 1 (tensor amax 2688) and power-of-two E4M3 block scales
    kk = g.integers(-6, 6, size=(32, 16))
    kk[0, 0] = 8                             # 6 * 2^8 = 1536 < 2688: keep one 2688 below
    y = (vals[codes] * np.ldexp(np.float32(1), np.repeat(kk, 16, axis=1))).astype(np.float32)
    y[0, 16:32] = 0.0
    y[0, 16] = 2688.0
    q = oracle.quantize(y, oracle.NVFP4, want_xhat=True)["row"]
    assert float(q["tscale"][0]) == 1.0
    keep = np.ones_like(y, bool)
    keep[0, 16:32] = False
    assert np.array_equal(q["xhat"][keep], y[keep])


@pytest.mark.parametrize("fmt", [oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL])
def test_range_and_error_bounds(fmt):
    """I2 |xhat| <= 6 s_eff; I3 unclipped elements are within half a grid gap
    (times s_eff, plus the reciprocal's rounding) of x."""
    x = _test_tensor(seed=11)
    q = oracle.quantize(x, fmt, want_xhat=True, want_mask=True)["row"]
    xh = q["xhat"].astype(np.float64)
    B = 32 if fmt == oracle.MXFP4 else 16
    rows, cols = x.shape
    xb = np.abs(x.astype(np.float64)).reshape(rows, cols // B, B)
    xhb = np.abs(xh).reshape(rows, cols // B, B)
    # block effective scale: decoding code 2 (value 1.0) under each scale gives s_eff exactly
    ones = {"codes": np.full((rows, cols // 2), 0x22, np.uint8), "scales": q["scales"]}
    if "tscale" in q:
        ones["tscale"] = q["tscale"]
    s_eff = oracle.dequantize(ones, rows, cols, fmt=fmt).reshape(rows, cols // B, B)[..., 0]
    s_eff = s_eff.astype(np.float64)
    assert (xhb <= 6.0 * s_eff[..., None] * (1 + 2.0 ** -23)).all()   # fp32 product rounding
    bits = np.unpackbits(q["mask"].view(np.uint8), bitorder="little")[: rows * cols]
    unclipped = bits.reshape(rows, cols // B, B).astype(bool)
    a = xb / np.where(s_eff == 0, 1.0, s_eff)[..., None]
    gap = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    err = np.abs(xb - xhb)
    bound = gap / 2 * s_eff[..., None] * (1 + 1e-6) + 1e-45
    assert (err[unclipped] <= bound[unclipped]).all()


def test_double_block_equals_per_tensor_when_outer_amax_is_uniform():
    """I4: if every 1x128 block has the same amax A, double-block quantization
    equals NVFP4 whose tensor amax is A."""
    g = np.random.default_rng(5)
    x = g.uniform(-1, 1, size=(16, 512)).astype(np.float32)
    A = np.float32(3.75)
    blocks = x.reshape(16, 4, 128)
    pos = g.integers(0, 128, size=(16, 4))
    for i in range(16):
        for j in range(4):
            blocks[i, j, pos[i, j]] = A if (i + j) % 2 else -A
    x = blocks.reshape(16, 512)
    a = oracle.quantize(x, oracle.NVFP4_2LEVEL, want_xhat=True)["row"]
    b = oracle.quantize(x, oracle.NVFP4, want_xhat=True)["row"]
    assert np.array_equal(a["codes"], b["codes"])
    assert np.array_equal(a["scales"], b["scales"])
    assert np.array_equal(a["xhat"], b["xhat"])
    assert (a["tscale"] == b["tscale"][0]).all()


def test_zero_tensor():
    x = np.zeros((4, 128), np.float32)
    x[1] = -0.0
    for fmt in (oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL):
        q = oracle.quantize(x, fmt, want_xhat=True, want_mask=True)["row"]
        assert (q["scales"] == 0).all()
        assert (q["codes"][0] == 0).all() and (q["codes"][1] == 0x88).all()
        assert not q["xhat"].any() and np.signbit(q["xhat"][1]).all()
        assert (q["mask"] == 0xFFFFFFFF).all()
        if fmt != oracle.MXFP4:
            assert not q["tscale"].any()


def test_column_wise_is_row_wise_of_transpose():
    x = _test_tensor(rows=64, cols=128, seed=2)
    r = oracle.quantize(x, oracle.NVFP4, orient=oracle.ROWCOL)
    t = oracle.quantize(np.ascontiguousarray(x.T), oracle.NVFP4, orient=oracle.ROW)["row"]
    assert np.array_equal(r["col"]["codes"], t["codes"])
    assert np.array_equal(r["col"]["scales"], t["scales"])
    # the transposed blocks of an outlier column carry the large scales
    assert r["col"]["scales"][7].min() > np.median(r["col"]["scales"])


@pytest.mark.slow
def test_stochastic_rounding_is_unbiased_on_laplace_gradients():
    """E[SR(x)] = x ("Resumo Técnico: TetraJet-v2", §2A): the mean error of
    double-block SR on Laplace(0, 1e-3) gradients is below 1e-3 of mean |x|,
    while nearest-even rounding of the same tensor is deterministic."""
    x = workloads.grad_2level(shape=(512, 4096), seed=3).float().numpy()
    q = oracle.quantize(x, oracle.NVFP4_2LEVEL, rounding=oracle.SR, seed=0x5EED,
                        want_xhat=True)["row"]
    xh = q["xhat"].astype(np.float64)
    xd = x.astype(np.float64)
    bias = abs((xh - xd).mean()) / np.abs(xd).mean()
    assert bias < 1e-3
    q2 = oracle.quantize(x, oracle.NVFP4_2LEVEL, rounding=oracle.SR, seed=0x5EED + 1,
                         want_xhat=True)["row"]
    assert not np.array_equal(q2["codes"], q["codes"])       # the seed matters
    q3 = oracle.quantize(x, oracle.NVFP4_2LEVEL, rounding=oracle.SR, seed=0x5EED,
                         want_xhat=True)["row"]
    assert np.array_equal(q3["codes"], q["codes"])           # and fully decides the bits
