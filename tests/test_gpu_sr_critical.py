"""Stochastic rounding at its critical points, GPU against the oracle, bit for
bit (needs a GB300).

The reading of stochastic rounding ("Resumo Técnico: TetraJet-v2", §2A: an
unbiased rounding of the backward operands): with lo the grid value at or
below |y|, g the gap above it and F = 65536 (|y| - lo) / g, the magnitude
rounds up iff the element's 16-bit uniform u < F.  The kernels decide this with floating-point steps (a
rounded-toward-zero multiply-add of the gap against an operand built from u),
which are exact only by an argument about the bits of F; the places where a
slip would show are the values of y whose F is an integer k or lies one ulp
either side of it, where u = k - 1 and u = k must go opposite ways.

Each MXFP4 block holds the anchor 4.0 (so the block scale is exactly 2^0 and
y = x) and 31 values from a list of such critical points in every gap of the
E2M1 grid, both signs, plus saturating and tiny values.  Over 2^22 blocks
every value meets about 217 thousand Philox draws, so about 96% of the 65536
u values occur for each, and both of the critical u = k - 1 and u = k for
about nine in ten of the integer-F values.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from gpu_common import assert_eq, npy

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BLOCKS = 1 << 22


def critical_values() -> np.ndarray:
    gaps = [(0.0, 0.5), (0.5, 0.5), (1.0, 0.5), (1.5, 0.5), (2.0, 1.0), (3.0, 1.0), (4.0, 2.0)]
    ks = [0, 1, 2, 63, 64, 65, 4095, 4096, 32767, 32768, 32769, 65472, 65534, 65535]
    vals = []
    for lo, g in gaps:
        for k in ks:
            y = np.float32(lo + g * k / 65536.0)          # exact: g k / 65536 has <= 17 bits
            assert float(y) == lo + g * k / 65536.0
            vals += [y, np.nextafter(y, np.float32(np.inf)), np.nextafter(y, np.float32(0))]
    vals += [np.float32(v) for v in (6.0, 6.25, 7.999, 5.9999995, 1e-30, 2.0 ** -20, 1e-40)]
    v = np.unique(np.array(vals, dtype=np.float32))
    v = v[v >= 0]
    return np.concatenate([v, -v])


def test_stochastic_rounding_critical_points():
    vals = critical_values()
    idx = np.arange(BLOCKS * 31, dtype=np.int64) % vals.size
    x = np.empty((BLOCKS, 32), dtype=np.float32)
    x[:, 0] = 4.0
    x[:, 1:] = vals[idx].reshape(BLOCKS, 31)
    seed, offset = 0x0DDC0FFEE, 9
    cfg = fq.Config(fq.MXFP4, fq.SR, seed, offset)
    q, _ = fq.fq_quantize(torch.from_numpy(x).cuda(), cfg)
    torch.cuda.synchronize()
    assert (npy(q.scales) == 127).all()                   # every block scale is 2^0
    ref = oracle.quantize(x, oracle.MXFP4, oracle.SR, seed, offset)["row"]
    assert_eq("codes", npy(q.codes), ref["codes"])
    # the round-up share of each value follows its F (a loose check of the draws)
    codes = npy(q.codes)
    lo_n, hi_n = codes & 0xF, codes >> 4
    c = np.empty((BLOCKS, 32), dtype=np.uint8)
    c[:, 0::2], c[:, 1::2] = lo_n, hi_n
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)[c[:, 1:] & 7].reshape(-1)
    y = np.abs(x[:, 1:].reshape(-1).astype(np.float64))
    for v in np.unique(np.abs(vals)):
        if v >= 6.0 or v == 0.0:
            continue
        sel = y == v
        lo = max(m for m in mags_grid() if m <= v)
        gap = next(m for m in mags_grid() if m > v) - lo
        f = (v - lo) / gap
        up = (mags[sel] > lo).mean()
        assert abs(up - f) < 0.01, (v, up, f)


def mags_grid():
    return (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
