"""Python binding of the C ABI in include/fq.h (ctypes).

Argument marshalling only: every function passes device pointers of torch
tensors, sizes and the current CUDA stream to the library function of the
same name, and raises FqError on a non-zero status.  Output tensors that the
caller does not supply are allocated with torch (device memory is torch's
job here); no quantization arithmetic happens in Python.  The library must be
built (``build()``); loading fails loudly otherwise -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import build as _build

NVFP4, MXFP4, NVFP4_2LEVEL = 0, 1, 2
RNE, SR = 0, 1
ROW, COL, ROWCOL = 1, 2, 3
F32, BF16 = 0, 1
BLOCK = {NVFP4: 16, MXFP4: 32, NVFP4_2LEVEL: 16}

STATUS = {0: "FQ_OK", 1: "FQ_ERR_INVALID_ARG", 2: "FQ_ERR_SHAPE", 3: "FQ_ERR_ALIGN",
          4: "FQ_ERR_WORKSPACE", 5: "FQ_ERR_UNSUPPORTED", 6: "FQ_ERR_CUDA"}

HEADER = os.path.join(_build.INCLUDE, "fq.h")


class FqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("rounding", ctypes.c_int32),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint32),
                ("rht_seed", ctypes.c_uint32)]

    def __init__(self, format=NVFP4, rounding=RNE, seed=0, offset=0, rht_seed=0):
        super().__init__(format, rounding, seed, offset, rht_seed)


class _QT(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tscale", ctypes.c_void_p)]


@dataclass
class QTensor:
    """A quantized [rows, cols] tensor: packed codes, block scales and the
    tensor (NVFP4) or outer-block (double block) FP32 scales."""
    codes: torch.Tensor
    scales: torch.Tensor
    tscale: Optional[torch.Tensor]

    def _c(self) -> _QT:
        return _QT(self.codes.data_ptr(), self.scales.data_ptr(),
                   None if self.tscale is None else self.tscale.data_ptr())


def alloc_qtensor(rows: int, cols: int, fmt: int, device="cuda") -> QTensor:
    B = BLOCK[fmt]
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((rows, cols // B), dtype=torch.uint8, device=device)
    if fmt == NVFP4:
        tscale = torch.empty(4, dtype=torch.float32, device=device)
    elif fmt == NVFP4_2LEVEL:
        tscale = torch.empty((rows, max(cols // 128, 1)), dtype=torch.float32, device=device)
    else:
        tscale = None
    return QTensor(codes, scales, tscale)


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def declared_symbols() -> list:
    """Names of the entry points that include/fq.h declares."""
    with open(HEADER) as f:
        return re.findall(r"FQ_API\s+[^;(]*?\b(fq_\w+)\s*\(", f.read())


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built ({path} missing): run "
                               "fp4_quantization_aware_fq_gb300.build.build() first")
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        L.fq_workspace_size.argtypes = [P(Config), i64, i64]
        L.fq_workspace_size.restype = sz
        L.fq_osci_workspace_size.argtypes = [i32]
        L.fq_osci_workspace_size.restype = sz
        L.fq_amax.argtypes = [vp, i32, i64, vp, vp]
        L.fq_quantize.argtypes = [P(Config), vp, i32, i64, i64, i64, i32, P(_QT), P(_QT), vp, vp, sz,
                                  vp]
        L.fq_fakequant_ste.argtypes = [P(Config), vp, i32, i64, i64, i64, vp, i32, vp, P(_QT), P(_QT),
                                       vp, vp, sz, vp]
        L.fq_dequantize.argtypes = [P(Config), P(_QT), i64, i64, vp, i32, i64, vp]
        L.fq_ste_backward.argtypes = [vp, i32, vp, i64, vp, vp]
        L.fq_osci_update.argtypes = [P(Config), i32, P(i64), P(i64), P(vp), P(vp), P(vp), P(vp),
                                     P(_QT), P(_QT), P(vp), i32, P(vp), vp, sz, vp]
        L.fq_osci_reset.argtypes = [P(Config), i32, P(i64), P(i64), P(vp), P(vp), P(vp), P(_QT),
                                    ctypes.c_float, vp, vp]
        L.fq_osci_update_noalloc.argtypes = [P(Config), i32, P(i64), P(i64), P(vp), P(vp), P(vp),
                                             P(vp), P(_QT), P(_QT), P(vp), i32, P(vp), vp]
        L.fq_osci_update_reset.argtypes = [P(Config), i32, P(i64), P(i64), P(vp), P(vp), P(vp),
                                           P(vp), P(_QT), P(_QT), P(vp), i32, P(vp),
                                           ctypes.c_float, vp, vp, sz, vp]
        L.fq_channel_amax.argtypes = [vp, i32, i64, i64, vp, vp]
        L.fq_select_channels.argtypes = [vp, i64, i64, vp, vp, vp, vp]
        L.fq_quantize_outliers.argtypes = [P(Config), vp, i32, i64, i64, vp, i64, vp, P(_QT), vp,
                                           vp, i32, vp, vp, sz, vp]
        L.fq_qad_kl.argtypes = [vp, vp, i32, i64, i64, ctypes.c_float, ctypes.c_float, vp, vp,
                                vp, i32, vp, vp]
        L.fq_gemm.argtypes = [P(Config), P(_QT), P(_QT), i64, i64, i64, vp, i32, vp, sz, vp, vp]
        L.fq_gemm_workspace_size.argtypes = [i64, i64, i64]
        L.fq_gemm_workspace_size.restype = sz
        for name in ("fq_amax", "fq_quantize", "fq_fakequant_ste", "fq_dequantize",
                     "fq_ste_backward", "fq_osci_update", "fq_osci_reset",
                     "fq_osci_update_noalloc", "fq_osci_update_reset", "fq_channel_amax",
                     "fq_select_channels", "fq_quantize_outliers", "fq_qad_kl", "fq_gemm"):
            getattr(L, name).restype = ctypes.c_int
        L.fq_status_string.argtypes = [ctypes.c_int]
        L.fq_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def _check(st: int, what: str):
    if st != 0:
        raise FqError(st, what)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dims(x: torch.Tensor):
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("expected a contiguous 2-D tensor")
    return x.shape[0], x.shape[1]


def _dims_ld(x: torch.Tensor):
    """rows, cols and the row pitch of a 2-D tensor whose rows are dense
    (stride 1 along a row), such as a column slice of a wider tensor."""
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError("expected a 2-D tensor with unit stride along its rows")
    rows, cols = x.shape
    return rows, cols, (x.stride(0) if rows > 1 else cols)


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------
def fq_status_string(status: int) -> str:
    return lib().fq_status_string(status).decode()


def fq_workspace_size(cfg: Config, rows: int, cols: int) -> int:
    return lib().fq_workspace_size(ctypes.byref(cfg), rows, cols)


def fq_osci_workspace_size(ntensors: int) -> int:
    return lib().fq_osci_workspace_size(ntensors)


def workspace(cfg: Config, rows: int, cols: int, device="cuda") -> Optional[torch.Tensor]:
    n = fq_workspace_size(cfg, rows, cols)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None


def fq_amax(x: torch.Tensor, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().fq_amax(x.data_ptr(), _dtype_code(x), x.numel(), out.data_ptr(), _stream(stream)),
           "fq_amax")
    return out


def fq_quantize(x: torch.Tensor, cfg: Config, orient: int = ROW,
                row_out: Optional[QTensor] = None, col_out: Optional[QTensor] = None,
                amax_in: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                stream=None):
    rows, cols, ld = _dims_ld(x)
    if orient & ROW and row_out is None:
        row_out = alloc_qtensor(rows, cols, cfg.format, x.device)
    if orient & COL and col_out is None:
        col_out = alloc_qtensor(cols, rows, cfg.format, x.device)
    if ws is None:
        ws = workspace(cfg, rows, cols, x.device)
    rq = ctypes.byref(row_out._c()) if orient & ROW else None
    cq = ctypes.byref(col_out._c()) if orient & COL else None
    st = lib().fq_quantize(ctypes.byref(cfg), x.data_ptr(), _dtype_code(x), rows, cols, ld, orient,
                           rq, cq, _ptr(amax_in), _ptr(ws), 0 if ws is None else ws.numel(),
                           _stream(stream))
    _check(st, "fq_quantize")
    return (row_out if orient & ROW else None), (col_out if orient & COL else None)


def fq_fakequant_ste(x: torch.Tensor, cfg: Config, xhat: Optional[torch.Tensor] = None,
                     xhat_dtype=None, want_mask: bool = True,
                     mask: Optional[torch.Tensor] = None,
                     row_out: Optional[QTensor] = None, col_out: Optional[QTensor] = None,
                     want_row_q: bool = False, want_col_q: bool = False,
                     amax_in: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                     stream=None):
    rows, cols, ld = _dims_ld(x)
    if xhat is None:
        xhat = torch.empty((rows, cols), dtype=xhat_dtype or x.dtype, device=x.device)
    if mask is None and want_mask:
        mask = torch.empty(((rows * cols + 7) // 8 + 15) // 16 * 16, dtype=torch.uint8,
                           device=x.device)
    if row_out is None and want_row_q:
        row_out = alloc_qtensor(rows, cols, cfg.format, x.device)
    if col_out is None and want_col_q:
        col_out = alloc_qtensor(cols, rows, cfg.format, x.device)
    if ws is None:
        ws = workspace(cfg, rows, cols, x.device)
    rq = ctypes.byref(row_out._c()) if row_out is not None else None
    cq = ctypes.byref(col_out._c()) if col_out is not None else None
    st = lib().fq_fakequant_ste(ctypes.byref(cfg), x.data_ptr(), _dtype_code(x), rows, cols, ld,
                                xhat.data_ptr(), _dtype_code(xhat), _ptr(mask), rq, cq,
                                _ptr(amax_in), _ptr(ws), 0 if ws is None else ws.numel(),
                                _stream(stream))
    _check(st, "fq_fakequant_ste")
    return xhat, mask, row_out, col_out


def fq_dequantize(q: QTensor, rows: int, cols: int, cfg: Config,
                  y: Optional[torch.Tensor] = None, y_dtype=torch.float32, stream=None):
    if y is None:
        y = torch.empty((rows, cols), dtype=y_dtype, device=q.codes.device)
    if tuple(y.shape) != (rows, cols):
        raise ValueError("y must be [rows, cols]")
    _, _, ldy = _dims_ld(y)
    st = lib().fq_dequantize(ctypes.byref(cfg), ctypes.byref(q._c()), rows, cols, y.data_ptr(),
                             _dtype_code(y), ldy, _stream(stream))
    _check(st, "fq_dequantize")
    return y


def fq_ste_backward(dy: torch.Tensor, mask: torch.Tensor, dx: Optional[torch.Tensor] = None,
                    stream=None):
    if dx is None:
        dx = torch.empty_like(dy)
    st = lib().fq_ste_backward(dy.data_ptr(), _dtype_code(dy), mask.data_ptr(), dy.numel(),
                               dx.data_ptr(), _stream(stream))
    _check(st, "fq_ste_backward")
    return dx


def _arr(ctype, vals):
    return (ctype * max(len(vals), 1))(*vals)


def fq_osci_update(cfg: Config, master: Sequence[torch.Tensor], delta: Sequence[torch.Tensor],
                   dist_q: Sequence[torch.Tensor], dist_m: Sequence[torch.Tensor],
                   prev: Sequence[QTensor], nxt: Sequence[QTensor],
                   xhat: Optional[Sequence[torch.Tensor]] = None, xhat_dtype=torch.bfloat16,
                   mask: Optional[Sequence[torch.Tensor]] = None,
                   ws: Optional[torch.Tensor] = None, stream=None):
    n = len(master)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = _arr(i64, [m.shape[0] for m in master])
    cols = _arr(i64, [m.shape[1] for m in master])
    if ws is None:
        ws = torch.empty(max(fq_osci_workspace_size(n), 16), dtype=torch.uint8,
                         device=master[0].device)
    pq = (_QT * max(n, 1))(*[q._c() for q in prev])
    nq = (_QT * max(n, 1))(*[q._c() for q in nxt])
    st = lib().fq_osci_update(
        ctypes.byref(cfg), n, rows, cols, _arr(vp, [t.data_ptr() for t in master]),
        _arr(vp, [t.data_ptr() for t in delta]), _arr(vp, [t.data_ptr() for t in dist_q]),
        _arr(vp, [t.data_ptr() for t in dist_m]), pq, nq,
        None if xhat is None else _arr(vp, [t.data_ptr() for t in xhat]),
        BF16 if xhat_dtype == torch.bfloat16 else F32,
        None if mask is None else _arr(vp, [t.data_ptr() for t in mask]),
        ws.data_ptr(), ws.numel(), _stream(stream))
    _check(st, "fq_osci_update")


def fq_osci_update_reset(cfg: Config, master: Sequence[torch.Tensor],
                         delta: Sequence[torch.Tensor], dist_q: Sequence[torch.Tensor],
                         dist_m: Sequence[torch.Tensor], prev: Sequence[QTensor],
                         nxt: Sequence[QTensor], threshold: float = 4.0,
                         n_reset: Optional[torch.Tensor] = None,
                         xhat: Optional[Sequence[torch.Tensor]] = None, xhat_dtype=torch.bfloat16,
                         mask: Optional[Sequence[torch.Tensor]] = None,
                         ws: Optional[torch.Tensor] = None, stream=None):
    """The window's last update step with the OsciReset reset fused in."""
    n = len(master)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = _arr(i64, [m.shape[0] for m in master])
    cols = _arr(i64, [m.shape[1] for m in master])
    if ws is None:
        ws = torch.empty(max(fq_osci_workspace_size(n), 16), dtype=torch.uint8,
                         device=master[0].device)
    pq = (_QT * max(n, 1))(*[q._c() for q in prev])
    nq = (_QT * max(n, 1))(*[q._c() for q in nxt])
    st = lib().fq_osci_update_reset(
        ctypes.byref(cfg), n, rows, cols, _arr(vp, [t.data_ptr() for t in master]),
        _arr(vp, [t.data_ptr() for t in delta]), _arr(vp, [t.data_ptr() for t in dist_q]),
        _arr(vp, [t.data_ptr() for t in dist_m]), pq, nq,
        None if xhat is None else _arr(vp, [t.data_ptr() for t in xhat]),
        BF16 if xhat_dtype == torch.bfloat16 else F32,
        None if mask is None else _arr(vp, [t.data_ptr() for t in mask]), float(threshold),
        _ptr(n_reset), ws.data_ptr(), ws.numel(), _stream(stream))
    _check(st, "fq_osci_update_reset")
    return n_reset


def fq_osci_update_noalloc(cfg: Config, master: Sequence[torch.Tensor],
                           delta: Sequence[torch.Tensor], dist_q: Sequence[torch.Tensor],
                           dist_m: Sequence[torch.Tensor], prev: Sequence[QTensor],
                           nxt: Sequence[QTensor], xhat: Optional[Sequence[torch.Tensor]] = None,
                           xhat_dtype=torch.bfloat16,
                           mask: Optional[Sequence[torch.Tensor]] = None, stream=None):
    """fq_osci_update for callers that cannot allocate: no workspace argument;
    the library's own static device scratch holds the per-tensor amax (at most
    FQ_NOALLOC_MAX_TENSORS tensors per call; concurrent calls on the GPU race
    on that scratch).  This wrapper allocates nothing either."""
    n = len(master)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = _arr(i64, [m.shape[0] for m in master])
    cols = _arr(i64, [m.shape[1] for m in master])
    pq = (_QT * max(n, 1))(*[q._c() for q in prev])
    nq = (_QT * max(n, 1))(*[q._c() for q in nxt])
    st = lib().fq_osci_update_noalloc(
        ctypes.byref(cfg), n, rows, cols, _arr(vp, [t.data_ptr() for t in master]),
        _arr(vp, [t.data_ptr() for t in delta]), _arr(vp, [t.data_ptr() for t in dist_q]),
        _arr(vp, [t.data_ptr() for t in dist_m]), pq, nq,
        None if xhat is None else _arr(vp, [t.data_ptr() for t in xhat]),
        BF16 if xhat_dtype == torch.bfloat16 else F32,
        None if mask is None else _arr(vp, [t.data_ptr() for t in mask]), _stream(stream))
    _check(st, "fq_osci_update_noalloc")


def fq_osci_reset(cfg: Config, master: Sequence[torch.Tensor], dist_q: Sequence[torch.Tensor],
                  dist_m: Sequence[torch.Tensor], cur: Sequence[QTensor], threshold: float = 4.0,
                  n_reset: Optional[torch.Tensor] = None, stream=None):
    n = len(master)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = _arr(i64, [m.shape[0] for m in master])
    cols = _arr(i64, [m.shape[1] for m in master])
    cq = (_QT * max(n, 1))(*[q._c() for q in cur])
    st = lib().fq_osci_reset(
        ctypes.byref(cfg), n, rows, cols, _arr(vp, [t.data_ptr() for t in master]),
        _arr(vp, [t.data_ptr() for t in dist_q]), _arr(vp, [t.data_ptr() for t in dist_m]), cq,
        float(threshold), _ptr(n_reset), _stream(stream))
    _check(st, "fq_osci_reset")
    return n_reset


# --------------------------------------------------------------------------
# static outlier retention
# --------------------------------------------------------------------------
MAX_CHANNELS = 131072


def fq_channel_amax(x: torch.Tensor, amax: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """Running per-channel (column) max |x|; amax accumulates across calls."""
    rows, cols = _dims(x)
    if amax is None:
        amax = torch.zeros(cols, dtype=torch.float32, device=x.device)
    st = lib().fq_channel_amax(x.data_ptr(), _dtype_code(x), rows, cols, amax.data_ptr(),
                               _stream(stream))
    _check(st, "fq_channel_amax")
    return amax


@dataclass
class Outliers:
    """Kept channels: ascending indices, bitmap (int32 words), FP8 scales."""
    idx: torch.Tensor
    bitmap: torch.Tensor
    fp8_scale: torch.Tensor

    @property
    def k(self) -> int:
        return self.idx.numel()


def fq_select_channels(channel_amax: torch.Tensor, k: int, stream=None) -> Outliers:
    cols = channel_amax.numel()
    dev = channel_amax.device
    idx = torch.empty(max(k, 4), dtype=torch.int32, device=dev)
    bitmap = torch.empty(max((cols + 31) // 32, 4), dtype=torch.int32, device=dev)
    fp8_scale = torch.empty(max(k, 4), dtype=torch.float32, device=dev)
    st = lib().fq_select_channels(channel_amax.data_ptr(), cols, k, idx.data_ptr(),
                                  bitmap.data_ptr(), fp8_scale.data_ptr(), _stream(stream))
    _check(st, "fq_select_channels")
    return Outliers(idx[:k], bitmap[:(cols + 31) // 32], fp8_scale[:k])


def fq_quantize_outliers(x: torch.Tensor, cfg: Config, sel: Outliers,
                         out: Optional[QTensor] = None, fp8: Optional[torch.Tensor] = None,
                         xhat: Optional[torch.Tensor] = None, xhat_dtype=None,
                         want_q: bool = True, want_fp8: bool = True, want_xhat: bool = True,
                         want_mask: bool = True, mask: Optional[torch.Tensor] = None,
                         ws: Optional[torch.Tensor] = None, stream=None):
    """Split FP4 / FP8 quantization; returns (out, fp8, xhat, mask)."""
    rows, cols = _dims(x)
    k = sel.k
    dev = x.device
    if out is None and want_q:
        out = alloc_qtensor(rows, cols, cfg.format, dev)
    if fp8 is None and want_fp8:
        fp8 = torch.empty((rows, max(k, 1)), dtype=torch.uint8, device=dev)[:, :k]
    if xhat is None and want_xhat:
        xhat = torch.empty((rows, cols), dtype=xhat_dtype or x.dtype, device=dev)
    if mask is None and want_mask:
        mask = torch.empty(((rows * cols + 7) // 8 + 15) // 16 * 16, dtype=torch.uint8,
                           device=dev)
    if ws is None:
        ws = workspace(cfg, rows, cols, dev)
    oq = ctypes.byref(out._c()) if out is not None else None
    st = lib().fq_quantize_outliers(ctypes.byref(cfg), x.data_ptr(), _dtype_code(x), rows, cols,
                                    sel.bitmap.data_ptr(), k, sel.fp8_scale.data_ptr(), oq,
                                    _ptr(fp8), _ptr(xhat),
                                    _dtype_code(xhat) if xhat is not None else F32, _ptr(mask),
                                    _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check(st, "fq_quantize_outliers")
    return out, fp8, xhat, mask


# --------------------------------------------------------------------------
# QAD distillation loss
# --------------------------------------------------------------------------
def fq_qad_kl(teacher: torch.Tensor, student: torch.Tensor, temperature: float = 1.0,
              grad_scale: Optional[float] = None, want_grad: bool = True, dz_dtype=None,
              loss_rows: Optional[torch.Tensor] = None,
              loss_mean: Optional[torch.Tensor] = None, dz: Optional[torch.Tensor] = None,
              err: Optional[torch.Tensor] = None, stream=None):
    """Per-row KL(softmax(teacher / T) || softmax(student / T)), its mean, and
    the student-logit gradient grad_scale * (q - p) / T (grad_scale defaults
    to 1 / rows, the gradient of the mean).  Returns (loss_rows, loss_mean,
    dz, err); err is a device int32 that is non-zero if a shared-memory copy
    timed out (read it after synchronising)."""
    rows, vocab = _dims(teacher)
    if student.shape != teacher.shape or student.dtype != teacher.dtype:
        raise ValueError("teacher and student logits must share shape and dtype")
    dev = teacher.device
    if grad_scale is None:
        grad_scale = 1.0 / rows if rows else 0.0
    if loss_rows is None:
        loss_rows = torch.empty(max(rows, 4), dtype=torch.float32, device=dev)[:rows]
    if loss_mean is None:
        loss_mean = torch.empty(1, dtype=torch.float32, device=dev)
    if dz is None and want_grad:
        dz = torch.empty((rows, vocab), dtype=dz_dtype or student.dtype, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = lib().fq_qad_kl(teacher.data_ptr(), student.data_ptr(), _dtype_code(teacher), rows,
                         vocab, float(temperature), float(grad_scale), loss_rows.data_ptr(),
                         loss_mean.data_ptr(), _ptr(dz),
                         _dtype_code(dz) if dz is not None else F32, err.data_ptr(),
                         _stream(stream))
    _check(st, "fq_qad_kl")
    return loss_rows, loss_mean, dz, err


# --------------------------------------------------------------------------
# block-scaled FP4 GEMM
# --------------------------------------------------------------------------
def fq_gemm_workspace_size(m: int, n: int, k: int) -> int:
    return lib().fq_gemm_workspace_size(m, n, k)


def fq_gemm(a: QTensor, b: QTensor, m: int, n: int, k: int, cfg: Optional[Config] = None,
            c: Optional[torch.Tensor] = None, c_dtype=torch.float32,
            ws: Optional[torch.Tensor] = None, err: Optional[torch.Tensor] = None, stream=None):
    """C[m, n] = deq(A) deq(B)^T for row-wise NVFP4 or MXFP4 (cfg.format) A
    [m, k] and B [n, k] on the tensor cores.  Returns (C, err); err is a device int32 that is
    non-zero if a pipeline wait timed out (read it after synchronising)."""
    cfg = cfg or Config(NVFP4)
    dev = a.codes.device
    if c is None:
        c = torch.empty((m, n), dtype=c_dtype, device=dev)
    if ws is None:
        ws = torch.empty(max(fq_gemm_workspace_size(m, n, k), 16), dtype=torch.uint8, device=dev)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = lib().fq_gemm(ctypes.byref(cfg), ctypes.byref(a._c()), ctypes.byref(b._c()), m, n, k,
                       c.data_ptr(), _dtype_code(c), ws.data_ptr(), ws.numel(), err.data_ptr(),
                       _stream(stream))
    _check(st, "fq_gemm")
    return c, err
