"""Row-pitched tensors through the C ABI (needs a GB300): x a column slice of
a wider tensor (ld > cols), y of fq_dequantize the same.  The kernels read
rows ld elements apart and must give, bit for bit, the oracle's result on the
dense copy.  The columns outside the slice hold values far larger than any
inside it, so a block, a tile or the tensor amax that reads one of them
changes the scales; fq_dequantize must leave them untouched."""
import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import FMT_O, as_oracle_input, assert_eq, bits, check_q, fakequant_parity, npy

pytestmark = pytest.mark.gpu

DEV = "cuda"
PAD = 3.0e4


def _slice(x: torch.Tensor, left: int, right: int) -> torch.Tensor:
    """x placed at column `left` of a wider device tensor whose other columns
    hold +-PAD; returns the [rows, cols] view (row pitch left + cols + right)."""
    rows, cols = x.shape
    wide = torch.empty((rows, left + cols + right), dtype=x.dtype)
    wide[:, :left] = PAD
    wide[:, left + cols:] = -PAD
    wide[:, left:left + cols] = x
    v = wide.to(DEV)[:, left:left + cols]
    assert v.stride(0) == left + cols + right and v.data_ptr() % 16 == 0
    return v


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_row_pitched_row_pass(dtype, fmt, rnd):
    rows, cols = 37, 384
    x = W.normal((rows, cols), 1.0, seed=40 + fmt).to(dtype)
    x[5, 7] = 90.0
    fakequant_parity(_slice(x, 16, 24), fmt, rnd, seed=0x1234567, offset=2)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
def test_row_pitched_rowcol_tiles(dtype, fmt, rnd):
    rows = 384 if fmt == fq.NVFP4_2LEVEL else 224
    cols = 384 if fmt == fq.NVFP4_2LEVEL else 160
    x = W.nvfp4_act(shape=(rows, cols), seed=50 + fmt, n_outlier_cols=2).to(dtype)
    fakequant_parity(_slice(x, 32, 8), fmt, rnd, seed=77, offset=5, orient=fq.ROWCOL)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_row_pitched_column_only(fmt):
    rows, cols = 256, 384
    x = _slice(W.nvfp4_act(shape=(rows, cols), seed=6, n_outlier_cols=2), 64, 64)
    cfg = fq.Config(fmt, fq.RNE)
    _, cq = fq.fq_quantize(x, cfg, orient=fq.COL)
    torch.cuda.synchronize()
    ref = oracle.quantize(as_oracle_input(x), FMT_O[fmt], orient=oracle.ROWCOL)
    check_q("col", cq, ref["col"], fmt)


def test_row_pitched_hadamard_rowcol():
    rows, cols = 256, 256
    x = _slice(W.grad_2level(shape=(rows, cols), seed=9), 8, 8)
    fakequant_parity(x, fq.NVFP4_2LEVEL, fq.SR, seed=5, offset=1, orient=fq.ROWCOL,
                     rht_seed=0xB00F)


def test_row_pitched_tensor_amax_ignores_the_other_columns():
    rows, cols = 64, 128
    x = W.normal((rows, cols), 1.0, seed=3)
    v = _slice(x, 16, 16)
    rq, _ = fq.fq_quantize(v, fq.Config(fq.NVFP4))
    torch.cuda.synchronize()
    want = np.float32(np.abs(x.numpy()).max()) / np.float32(2688.0)
    assert npy(rq.tscale)[0] == want


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_row_pitched_dequantize_output(fmt, ydt):
    rows, cols, left, right = 48, 256, 16, 48
    x = W.grad_2level(shape=(rows, cols), seed=12).to(DEV)
    cfg = fq.Config(fmt, fq.RNE)
    rq, _ = fq.fq_quantize(x, cfg)
    dense = fq.fq_dequantize(rq, rows, cols, cfg, y_dtype=ydt)
    wide = torch.full((rows, left + cols + right), 7.0, dtype=ydt, device=DEV)
    y = wide[:, left:left + cols]
    fq.fq_dequantize(rq, rows, cols, cfg, y=y)
    torch.cuda.synchronize()
    assert_eq("pitched == dense", bits(y.contiguous()), bits(dense))
    w = npy(wide.float())
    assert (w[:, :left] == 7.0).all() and (w[:, left + cols:] == 7.0).all()
