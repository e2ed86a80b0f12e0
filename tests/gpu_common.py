"""Helpers for GPU-vs-oracle parity tests: run the CUDA path through the
C ABI binding and the oracle on the same inputs, compare bit for bit."""
import numpy as np
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads

FMT_O = {fq.NVFP4: oracle.NVFP4, fq.MXFP4: oracle.MXFP4, fq.NVFP4_2LEVEL: oracle.NVFP4_2LEVEL}


def as_oracle_input(x: torch.Tensor) -> np.ndarray:
    """The exact FP32 values the kernel sees (BF16 widened bit-exactly); a
    row-pitched view is taken as its dense copy."""
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return oracle.bf16_bits_to_f32(workloads.bf16_bits(x)).reshape(x.shape)
    return x.detach().cpu().numpy().astype(np.float32)


def npy(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return workloads.bf16_bits(t)
    return npy(t).view(np.uint32)


def assert_eq(name, got: np.ndarray, want: np.ndarray):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        first = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {first}: "
                             f"gpu={got[first]!r} oracle={want[first]!r}")


def check_q(name, q: fq.QTensor, ref: dict, fmt: int):
    assert_eq(name + ".codes", npy(q.codes), ref["codes"])
    assert_eq(name + ".scales", npy(q.scales), ref["scales"])
    if fmt == fq.NVFP4:
        assert_eq(name + ".tscale", npy(q.tscale)[:1].view(np.uint32),
                  ref["tscale"].reshape(-1)[:1].view(np.uint32))
    elif fmt == fq.NVFP4_2LEVEL:
        assert_eq(name + ".tscale", npy(q.tscale).view(np.uint32),
                  ref["tscale"].view(np.uint32))


def fakequant_parity(x: torch.Tensor, fmt: int, rnd: int = fq.RNE, seed: int = 0,
                     offset: int = 0, orient: int = fq.ROW, xhat_dtype=None, check_col=True,
                     rht_seed: int = 0):
    """Run fq_fakequant_ste (with row codes, optional column codes) on the GPU
    and the oracle; assert everything matches bit for bit."""
    rows, cols = x.shape
    cfg = fq.Config(fmt, rnd, seed, offset, rht_seed)
    xhat_dtype = xhat_dtype or x.dtype
    xhat, mask, rq, cq = fq.fq_fakequant_ste(x, cfg, xhat_dtype=xhat_dtype, want_mask=True,
                                             want_row_q=True,
                                             want_col_q=bool(orient & fq.COL))
    torch.cuda.synchronize()
    xo = as_oracle_input(x)
    ref = oracle.quantize(xo, FMT_O[fmt], rnd, seed, offset,
                          orient=(oracle.ROWCOL if orient & fq.COL else oracle.ROW),
                          want_xhat=True, want_mask=True, rht_seed=rht_seed)
    r = ref["row"]
    check_q("row", rq, r, fmt)
    if xhat_dtype == torch.bfloat16:
        assert_eq("xhat(bf16)", bits(xhat), oracle.f32_to_bf16_bits(r["xhat"]))
    else:
        assert_eq("xhat(f32)", bits(xhat), r["xhat"].view(np.uint32))
    nbytes = (rows * cols + 7) // 8
    assert_eq("mask", npy(mask)[:nbytes], r["mask"].view(np.uint8)[:nbytes])
    if orient & fq.COL and check_col:
        check_q("col", cq, ref["col"], fmt)
    return ref, (xhat, mask, rq, cq)
