"""Exhaustive check of the GPU E2M1 encoder: every FP32 bit pattern with
|y| < 8 (both signs, zeros and subnormals included), 2.18 G values, goes
through the MXFP4 quantizer in 32-element blocks whose first element is the
anchor 4.0, so that the shared scale is exactly 2^0 and the kernel encodes
the value itself.  Codes must equal the oracle's, computed on the host cores
by a spawned process pool (started before the first GPU call)."""
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LIMIT = 0x41000000                    # bit pattern of 8.0f: payloads are [0, 8)
PER_BLOCK = 31
BLOCKS = 1 << 20                      # blocks per chunk
PAYLOAD = PER_BLOCK * BLOCKS          # payload values per chunk
NCHUNK_POS = (LIMIT + PAYLOAD - 1) // PAYLOAD


def _chunk_input(k: int) -> np.ndarray:
    """Chunk k < NCHUNK_POS: positive patterns; k >= NCHUNK_POS: the same with
    the sign bit set.  Returns a [BLOCKS, 32] float32 array."""
    neg = k >= NCHUNK_POS
    base = (k % NCHUNK_POS) * PAYLOAD
    p = np.arange(base, base + PAYLOAD, dtype=np.int64)
    p = np.where(p < LIMIT, p, 0).astype(np.uint32)          # pad the tail with +0
    if neg:
        p |= np.uint32(0x80000000)
    x = np.empty((BLOCKS, 32), dtype=np.uint32)
    x[:, 0] = np.float32(4.0).view(np.uint32)
    x[:, 1:] = p.reshape(BLOCKS, PER_BLOCK)
    return x.view(np.float32)


def _oracle_codes(k: int) -> np.ndarray:
    import oracle
    x = _chunk_input(k)
    return oracle.quantize(x, oracle.MXFP4)["row"]["codes"]


def test_e2m1_encoder_exhaustive():
    import oracle
    oracle.build()
    nchunks = 2 * NCHUNK_POS
    workers = max(1, min(16, (os.cpu_count() or 2) - 1))
    ctx = mp.get_context("spawn")
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as pool:
        futs = {k: pool.submit(_oracle_codes, k) for k in range(nchunks)}
        from fp4_quantization_aware_fq_gb300 import fq
        cfg = fq.Config(fq.MXFP4)
        row = fq.alloc_qtensor(BLOCKS, 32, fq.MXFP4, "cuda")
        for k in range(nchunks):
            x = torch.from_numpy(_chunk_input(k)).cuda()
            fq.fq_quantize(x, cfg, row_out=row)
            got = row.codes.cpu().numpy()
            sc = row.scales.cpu().numpy()
            assert (sc == 127).all()
            want = futs[k].result()
            if not np.array_equal(got, want):
                bad = np.argwhere(got != want)[0]
                xin = _chunk_input(k)[bad[0], 2 * bad[1]:2 * bad[1] + 2]
                raise AssertionError(f"chunk {k}: first mismatch at {tuple(bad)}, inputs "
                                     f"{xin.view(np.uint32)} gpu={got[tuple(bad)]:#x} "
                                     f"oracle={want[tuple(bad)]:#x}")
