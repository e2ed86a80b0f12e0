"""Pins for the oracle's scalar format primitives (CPU only).

Each check compares the oracle with something that does not share its
arithmetic: exact-rational tables derived from the bit-field definitions,
torch's float8 / bfloat16 casts, and cuRAND's host Philox4x32-10 generator.
"""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from exact_formats import (e2m1_exact, e2m1_rne_exact, e4m3_encode_exact, e4m3_exact,
                           e8m0_exact, floor_log2_exact, sr_up_count_exact)

RNG = np.random.default_rng(12345)


def _f32(v):
    return float(np.float32(v))


# ---------------------------------------------------------------- E2M1
def test_e2m1_decode_matches_bitfields():
    for c in range(16):
        got = oracle.e2m1_value(c)
        assert got == float(e2m1_exact(c)), c
        assert math.copysign(1.0, got) == (-1.0 if c & 8 else 1.0), c


def _e2m1_probe_values():
    grid = [float(e2m1_exact(c)) for c in range(8)]
    pts = set()
    for g in grid:
        pts.add(g)
    for a, b in zip(grid[:-1], grid[1:]):
        m = np.float32((a + b) / 2)
        pts.update([float(m), float(np.nextafter(m, np.float32(0))),
                    float(np.nextafter(m, np.float32(10)))])
    for v in (6.0, 5.0):
        f = np.float32(v)
        pts.update([float(np.nextafter(f, np.float32(0))), float(np.nextafter(f, np.float32(99)))])
    pts.update([1e-30, 1e-45, 7.0, 100.0, 3.4e38, 0.0])
    pts.update(float(v) for v in RNG.uniform(0, 8, 2000).astype(np.float32))
    pts.update(float(v) for v in RNG.uniform(0, 0.3, 200).astype(np.float32))
    vals = sorted(pts)
    return vals + [-v for v in vals]


def test_e2m1_nearest_even_against_exact():
    for y in _e2m1_probe_values():
        assert oracle.e2m1_round_nearest(y) == e2m1_rne_exact(y), y


def test_e2m1_tie_table():
    # ties go to the even code: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    table = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 6.0: 7, 7.0: 7}
    for y, code in table.items():
        assert oracle.e2m1_round_nearest(y) == code
        assert oracle.e2m1_round_nearest(-y) == code | 8
    assert oracle.e2m1_round_nearest(-0.1) == 8
    assert oracle.e2m1_round_nearest(-0.0) == 8
    assert oracle.e2m1_round_nearest(0.0) == 0


def test_e2m1_grid_roundtrip():
    for c in range(16):
        assert oracle.e2m1_round_nearest(oracle.e2m1_value(c)) == c


# ---------------------------------------------------------------- E4M3
def test_e4m3_decode_all_codes_vs_exact_and_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    tv = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    for c in range(256):
        got = oracle.e4m3_value(c)
        ex = e4m3_exact(c)
        if ex is None:
            assert math.isnan(got) and math.isnan(tv[c]), c
        else:
            assert got == float(ex) == tv[c], c
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def _e4m3_probe_values():
    vals = sorted(float(e4m3_exact(c)) for c in range(0x7F))
    pts = set(vals)
    for a, b in zip(vals[:-1], vals[1:]):
        m = np.float32((a + b) / 2)
        pts.update([float(m), float(np.nextafter(m, np.float32(0))),
                    float(np.nextafter(m, np.float32(1e9)))])
    pts.update(float(v) for v in np.exp(RNG.uniform(np.log(1e-5), np.log(447.9), 3000)).astype(np.float32))
    pts.update([0.0, 1e-30, 2.0 ** -10, float(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))])
    return sorted(pts)


def test_e4m3_encode_vs_exact_and_torch():
    vals = _e4m3_probe_values()
    t = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    for s, tc in zip(vals, t):
        got = oracle.e4m3_encode(s)
        assert got == e4m3_encode_exact(s), s
        if s <= 448.0:
            assert got == tc, s


def test_e4m3_encode_saturates():
    for s in (448.0, 448.5, 463.9, 464.0, 480.0, 1e6, 3.4e38):
        assert oracle.e4m3_encode(s) == 0x7E


# ---------------------------------------------------------------- E8M0
def test_e8m0_decode_vs_exact_and_torch():
    for c in range(256):
        got = oracle.e8m0_value(c)
        ex = e8m0_exact(c)
        if ex is None:
            assert math.isnan(got)
        else:
            assert got == float(ex), c
    if hasattr(torch, "float8_e8m0fnu"):
        codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
        tv = codes.view(torch.float8_e8m0fnu).to(torch.float32).tolist()
        for c in range(255):
            assert oracle.e8m0_value(c) == tv[c], c


def test_e8m0_shared_exponent_vs_exact():
    probes = [0.0, 1e-45, 1e-40, 2.0 ** -126, 2.0 ** -125, 2.0 ** -124, 0.05, 1.0, 4.0, 6.0,
              7.99, 8.0, 3.4e38]
    for k in range(-130, 128):
        if -149 <= k <= 127:
            p = np.float32(2.0 ** k)
            probes += [float(p), float(np.nextafter(p, np.float32(0)))]
    probes += [float(v) for v in np.exp(RNG.uniform(-100, 88, 2000)).astype(np.float32)]
    for a in probes:
        got = oracle.e8m0_for_amax(a)
        if a == 0.0:
            assert got == 0
            continue
        k = min(max(floor_log2_exact(a) - 2, -127), 127)
        assert got == k + 127, a
        # the block maximum lands in [4, 8) after scaling unless clamped
        if -127 < k < 127:
            assert 4 <= Fraction(a) / Fraction(2) ** k < 8


# ---------------------------------------------------------------- bfloat16
def test_bf16_nearest_even_vs_torch():
    bits = RNG.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    ties = (RNG.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    bits = np.concatenate([bits, ties])
    x = bits.view(np.float32)
    keep = np.isfinite(x)
    x = x[keep]
    got = oracle.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- Philox
def _curand():
    cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcurand.so"),
             "libcurand.so", "libcurand.so.10"]
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not available")


def test_philox_against_curand_host_generator():
    """cuRAND's host Philox4x32-10 generator lays its output out as 65536
    subsequences: output block b is Philox(counter = (b // 65536 as a 64-bit
    value in words 0-1, b % 65536 in word 2, 0), key = seed)."""
    lib = _curand()
    gen = ctypes.c_void_p()
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        cases = [(0, 0), (0x1234567887654321, 0), (5, 4 * 7), (0xDEADBEEF, 4 * 65536 * 3 + 4 * 11),
                 (77, 4 * 65536 * (1 << 32) + 4 * 5), (2 ** 64 - 1, 4 * 65536 * 0x0001_0002_0003)]
        for seed, off in cases:
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(off)) == 0
            buf = (ctypes.c_uint * 16)()
            assert lib.curandGenerate(gen, buf, 16) == 0
            for j in range(4):
                b = off // 4 + j
                c, t = b // 65536, b % 65536
                want = oracle.philox4x32_10([c & 0xFFFFFFFF, c >> 32, t, 0],
                                            [seed & 0xFFFFFFFF, seed >> 32])
                assert list(buf)[4 * j:4 * j + 4] == want, (seed, off, j)
    finally:
        lib.curandDestroyGenerator(gen)


def test_sr_draw_layout():
    """Element idx takes half (idx % 2) of word (idx % 8) // 2 of the Philox
    block with counter (idx // 8, stream, offset)."""
    seed = 0x0123456789ABCDEF
    for idx in [0, 1, 7, 8, 12345, 2 ** 33 + 5]:
        for stream, offset in [(0, 0), (1, 0), (0, 99)]:
            g = idx // 8
            out = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, stream, offset],
                                       [seed & 0xFFFFFFFF, seed >> 32])
            j = idx % 8
            assert oracle.sr_draw(seed, idx, stream, offset) == (out[j // 2] >> (16 * (j % 2))) & 0xFFFF


# ---------------------------------------------------------------- stochastic rounding
def test_sr_exact_up_counts():
    """Over all 65536 values of u, the number that round up is ceil(frac * 65536)."""
    ys = [0.0, 0.5, 3.0, 0.1, 0.25, 0.75, 1.3, 2.2, 2.999, 4.5, 5.0, 5.9999995, 1e-20,
          float(np.float32(1.0 / 3.0))]
    ys += [float(v) for v in RNG.uniform(0, 6, 6).astype(np.float32)]
    us = range(65536)
    for y in ys:
        grid = [float(e2m1_exact(c)) for c in range(8)]
        lo = max(i for i in range(8) if grid[i] <= y)
        ups = 0
        for u in us:
            c = oracle.e2m1_round_stochastic(y, u)
            assert c in (lo, lo + 1), (y, u, c)
            ups += c == lo + 1
        assert ups == sr_up_count_exact(y), y
    # negative values mirror, saturation is deterministic
    assert oracle.e2m1_round_stochastic(-0.75, 0) == 8 | 2
    assert oracle.e2m1_round_stochastic(-0.75, 65535) == 8 | 1
    for u in (0, 1234, 65535):
        assert oracle.e2m1_round_stochastic(6.0, u) == 7
        assert oracle.e2m1_round_stochastic(-9.0, u) == 15
