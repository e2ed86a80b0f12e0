"""Buffers on a 16-byte but not a 32-byte boundary (needs a GB300).

The kernels load row blocks and store fake-quantized values, dequantized
values and GEMM outputs 32 bytes at a time when the buffer and its row pitch
are 32-byte aligned, and fall back to 16-byte accesses otherwise (the C ABI
asks for 16-byte alignment only).  These cases run every fallback: x, xhat,
y and C placed 16 bytes past a 32-byte boundary.  The quantizers are compared
with the oracle bit for bit; dequantize, the split quantizer and the GEMM bit
for bit with the same call on 32-byte-aligned buffers (each is checked against
the oracle elsewhere).
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import FMT_O, as_oracle_input, assert_eq, bits, check_q, npy

pytestmark = pytest.mark.gpu

DEV = "cuda"


def off16(shape, dtype):
    """An empty device tensor whose data starts 16 bytes past a 32-byte
    boundary."""
    n = int(np.prod(shape))
    esz = torch.empty((), dtype=dtype).element_size()
    buf = torch.empty(n * esz + 64, dtype=torch.uint8, device=DEV)
    start = (-buf.data_ptr()) % 32 + 16
    t = buf[start:start + n * esz].view(dtype).view(shape)
    assert t.data_ptr() % 32 == 16
    return t


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("orient", [fq.ROW, fq.ROWCOL])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float32])
def test_fakequant_with_unaligned_x_and_xhat(fmt, orient, xdt):
    rows, cols = 256, 384
    src = W.nvfp4_act(shape=(rows, cols), seed=30 + fmt, n_outlier_cols=2).to(xdt)
    x = off16((rows, cols), xdt)
    x.copy_(src.to(DEV))
    for xhat_dt in (torch.bfloat16, torch.float32):
        xhat = off16((rows, cols), xhat_dt)
        cfg = fq.Config(fmt)
        _, mask, rq, cq = fq.fq_fakequant_ste(x, cfg, xhat=xhat, want_mask=True, want_row_q=True,
                                              want_col_q=bool(orient & fq.COL))
        torch.cuda.synchronize()
        ref = oracle.quantize(as_oracle_input(x), FMT_O[fmt],
                              orient=oracle.ROWCOL if orient & fq.COL else oracle.ROW,
                              want_xhat=True, want_mask=True)
        check_q("row", rq, ref["row"], fmt)
        if xhat_dt == torch.bfloat16:
            assert_eq("xhat", bits(xhat), oracle.f32_to_bf16_bits(ref["row"]["xhat"]))
        else:
            assert_eq("xhat", bits(xhat), ref["row"]["xhat"].view(np.uint32))
        nb = rows * cols // 8
        assert_eq("mask", npy(mask)[:nb], ref["row"]["mask"].view(np.uint8)[:nb])
        if orient & fq.COL:
            check_q("col", cq, ref["col"], fmt)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_dequantize_into_unaligned_y(fmt):
    rows, cols = 64, 256
    x = W.grad_2level(shape=(rows, cols), seed=31).to(DEV)
    cfg = fq.Config(fmt)
    rq, _ = fq.fq_quantize(x, cfg)
    dense = fq.fq_dequantize(rq, rows, cols, cfg, y_dtype=torch.float32)
    y = off16((rows, cols), torch.float32)
    fq.fq_dequantize(rq, rows, cols, cfg, y=y)
    torch.cuda.synchronize()
    assert_eq("y", bits(y.contiguous()), bits(dense))


def test_split_quantizer_with_unaligned_x_and_xhat():
    rows, cols, k = 64, 512, 51
    src = W.channel_act(shape=(rows, cols), n_outlier_cols=8)
    amax = torch.zeros(cols, dtype=torch.float32, device=DEV)
    fq.fq_channel_amax(src.to(DEV), amax)
    sel = fq.fq_select_channels(amax, k)
    x = off16((rows, cols), torch.float32)
    x.copy_(src.to(DEV))
    xhat = off16((rows, cols), torch.bfloat16)
    out, fp8, _, _ = fq.fq_quantize_outliers(x, fq.Config(fq.NVFP4), sel, xhat=xhat)
    aligned = torch.empty((rows, cols), dtype=torch.bfloat16, device=DEV)
    out2, fp82, _, _ = fq.fq_quantize_outliers(x.contiguous(), fq.Config(fq.NVFP4), sel,
                                               xhat=aligned)
    torch.cuda.synchronize()
    assert_eq("xhat", bits(xhat), bits(aligned))
    assert_eq("codes", npy(out.codes), npy(out2.codes))
    assert_eq("fp8", npy(fp8), npy(fp82))


def test_gemm_into_unaligned_c():
    m, n, k = 256, 256, 512
    a = W.normal((m, k), 1.0, seed=41).to(DEV)
    b = W.normal((n, k), 1.0, seed=42).to(DEV)
    cfg = fq.Config(fq.NVFP4)
    qa, _ = fq.fq_quantize(a, cfg)
    qb, _ = fq.fq_quantize(b, cfg)
    for dt in (torch.bfloat16, torch.float32):
        c_al, _ = fq.fq_gemm(qa, qb, m, n, k, cfg, c_dtype=dt)
        c = off16((m, n), dt)
        fq.fq_gemm(qa, qb, m, n, k, cfg, c=c)
        torch.cuda.synchronize()
        assert_eq(f"c {dt}", bits(c.contiguous()), bits(c_al))
