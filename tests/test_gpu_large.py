"""Tensors of more than 2^31 elements (needs a GB300; about 15 GB of device
memory).  Every flat element, block, scale and mask index past 2^31 must be
formed in 64 bits: the checks read the outputs of the rows that lie entirely
beyond element 2^31, and of the transposed blocks at the end of the tensor,
and compare them with the oracle run on just those rows (row-wise blocks are
row-local; the NVFP4 tensor amax is fixed by construction).

x is BF16 [65664, 32768] = 2,151,677,952 elements, N(0, 1) from seed 17, with
one element of 1000 at the very end: it is the tensor amax (N(0, 1) draws of
this many elements stay far below it), so an amax pass that stops short of
the last element gives a different tensor scale.
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import as_oracle_input, assert_eq, bits, npy

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda"
ROWS, COLS = 65664, 32768
PEAK = 1000.0
# rows whose every element has a flat index >= 2^31 (2^31 / 32768 = 65536)
SAMPLE_ROWS = (65536, 65600, ROWS - 2, ROWS - 1)
SAMPLE_COLS = (0, 12345, COLS - 1)


@pytest.fixture(scope="module")
def x():
    assert ROWS * COLS > 2 ** 31
    t = W.normal((ROWS, COLS), 1.0, seed=17, dtype=torch.bfloat16, device=DEV)
    t[-1, -1] = PEAK
    torch.cuda.synchronize()
    yield t
    del t
    torch.cuda.empty_cache()


def _rows(x, r0, r1):
    return as_oracle_input(x[r0:r1])


def test_tensor_amax_reaches_the_last_element(x):
    am = fq.fq_amax(x)
    torch.cuda.synchronize()
    assert float(npy(am)[0]) == PEAK


def test_nvfp4_rowcol_past_2g(x):
    cfg = fq.Config(fq.NVFP4)
    rq, cq = fq.fq_quantize(x, cfg, orient=fq.ROWCOL)
    torch.cuda.synchronize()
    for r in SAMPLE_ROWS:
        ref = oracle.quantize(_rows(x, r, r + 1), oracle.NVFP4, amax_in=PEAK)["row"]
        assert_eq(f"row {r} codes", npy(rq.codes[r:r + 1]), ref["codes"])
        assert_eq(f"row {r} scales", npy(rq.scales[r:r + 1]), ref["scales"])
    assert_eq("tscale", npy(rq.tscale)[:1].view(np.uint32),
              np.array([np.float32(PEAK) / np.float32(2688.0)], np.float32).view(np.uint32))
    # transposed blocks of the last 256 rows in a few columns: row c of X^T
    tail = 256
    for c in SAMPLE_COLS:
        xt = np.ascontiguousarray(_rows(x, ROWS - tail, ROWS)[:, c][None, :])
        ref = oracle.quantize(xt, oracle.NVFP4, amax_in=PEAK)["row"]
        assert_eq(f"col {c} codes", npy(cq.codes[c, (ROWS - tail) // 2:])[None, :],
                  ref["codes"])
        assert_eq(f"col {c} scales", npy(cq.scales[c, (ROWS - tail) // 16:])[None, :],
                  ref["scales"])
    del rq, cq


def test_mxfp4_fakequant_and_ste_past_2g(x):
    cfg = fq.Config(fq.MXFP4)
    xhat, mask, rq, _ = fq.fq_fakequant_ste(x, cfg, want_mask=True, want_row_q=True)
    torch.cuda.synchronize()
    mb = COLS // 8          # mask bytes per row
    r0, r1 = SAMPLE_ROWS[0], SAMPLE_ROWS[0] + 8
    ref = oracle.quantize(_rows(x, r0, r1), oracle.MXFP4, want_xhat=True, want_mask=True)["row"]
    assert_eq("codes", npy(rq.codes[r0:r1]), ref["codes"])
    assert_eq("scales", npy(rq.scales[r0:r1]), ref["scales"])
    assert_eq("xhat", bits(xhat[r0:r1]), oracle.f32_to_bf16_bits(ref["xhat"]))
    assert_eq("mask", npy(mask[r0 * mb:r1 * mb]), ref["mask"].view(np.uint8)[:(r1 - r0) * mb])
    # the last row, whose final block holds the peak (MXFP4 scales each block
    # by its own amax)
    rl = ROWS - 1
    ref = oracle.quantize(_rows(x, rl, ROWS), oracle.MXFP4, want_xhat=True, want_mask=True)["row"]
    assert_eq("last row xhat", bits(xhat[rl:]), oracle.f32_to_bf16_bits(ref["xhat"]))
    assert_eq("last row mask", npy(mask[rl * mb:ROWS * mb]), ref["mask"].view(np.uint8)[:mb])
    del xhat, rq
    # the STE backward over the same 2^31+ elements, dy = x
    dx = fq.fq_ste_backward(x, mask)
    torch.cuda.synchronize()
    for r in (r0, rl):
        m = npy(mask[r * mb:(r + 1) * mb]).view(np.uint32)
        want = oracle.ste_backward(bits(x[r:r + 1]).reshape(-1), m)   # BF16 bits in and out
        assert_eq(f"dx row {r}", bits(dx[r:r + 1]).reshape(-1), want)
    del dx, mask
