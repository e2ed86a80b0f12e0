"""Oracle for block-scaled FP4 fake-quantization -- TEST INFRASTRUCTURE ONLY.

The oracle is a plain, slow, scalar C implementation (``fq_oracle.c``) of
what the CUDA library computes, plus this ctypes wrapper that moves numpy
arrays in and out (and, for the block-scaled GEMM, numpy's float64 matmul of
the dequantized operands).  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the library never does, and the
two share no code.  Nothing here performs any of the method's arithmetic
except through ``fq_oracle.c``; the wrapper only allocates arrays, widens
bfloat16 bit patterns to float32 (exact) and transposes (for the column-wise
pass, which is the row-wise definition applied to the transpose).

Parity status: pinned.  See tests/test_oracle_*.py: exact-rational format
tables, torch's float8/bfloat16 casts, cuRAND's host Philox4x32-10 generator,
hand-worked blocks and invariants; for the distillation loss, the Bernoulli
closed form, scipy's relative entropy, finite differences and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

NVFP4, MXFP4, NVFP4_2LEVEL = 0, 1, 2
RNE, SR = 0, 1
ROW, COL, ROWCOL = 1, 2, 3
BLOCK = {NVFP4: 16, MXFP4: 32, NVFP4_2LEVEL: 16}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fq_oracle.c with gcc: strict IEEE binary32, no FMA contraction."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fno-unsafe-math-optimizations", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        f32, i32, i64, u32, u64 = (ctypes.c_float, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_uint32, ctypes.c_uint64)
        vp = ctypes.c_void_p
        lib.fqo_e2m1_value.argtypes = [i32]; lib.fqo_e2m1_value.restype = f32
        lib.fqo_e2m1_round_nearest.argtypes = [f32]; lib.fqo_e2m1_round_nearest.restype = i32
        lib.fqo_e2m1_round_stochastic.argtypes = [f32, ctypes.c_uint]
        lib.fqo_e2m1_round_stochastic.restype = i32
        lib.fqo_e4m3_value.argtypes = [i32]; lib.fqo_e4m3_value.restype = f32
        lib.fqo_e4m3_encode.argtypes = [f32]; lib.fqo_e4m3_encode.restype = i32
        lib.fqo_e8m0_value.argtypes = [i32]; lib.fqo_e8m0_value.restype = f32
        lib.fqo_e8m0_for_amax.argtypes = [f32]; lib.fqo_e8m0_for_amax.restype = i32
        lib.fqo_bf16_from_f32.argtypes = [f32]; lib.fqo_bf16_from_f32.restype = ctypes.c_uint16
        lib.fqo_bf16_from_f32_array.argtypes = [vp, i64, vp]
        lib.fqo_bf16_from_f32_array.restype = None
        lib.fqo_philox4x32_10.argtypes = [vp, vp, vp]; lib.fqo_philox4x32_10.restype = None
        lib.fqo_sr_draw.argtypes = [u64, u64, u32, u32]; lib.fqo_sr_draw.restype = ctypes.c_uint
        lib.fqo_amax.argtypes = [vp, i64]; lib.fqo_amax.restype = f32
        lib.fqo_rht_signs.argtypes = [u32, u32]; lib.fqo_rht_signs.restype = ctypes.c_uint
        lib.fqo_rht16.argtypes = [vp, ctypes.c_uint]; lib.fqo_rht16.restype = None
        lib.fqo_rht_rows.argtypes = [vp, i64, i64, u32, u32]; lib.fqo_rht_rows.restype = None
        lib.fqo_quantize_rows.argtypes = [i32, i32, u64, u32, u32, vp, i64, i64, f32,
                                          vp, vp, vp, vp, vp]
        lib.fqo_quantize_rows.restype = i32
        lib.fqo_dequantize_rows.argtypes = [i32, vp, vp, vp, i64, i64, vp]
        lib.fqo_dequantize_rows.restype = i32
        lib.fqo_ste_backward.argtypes = [vp, vp, i64, i32, vp]
        lib.fqo_ste_backward.restype = None
        lib.fqo_channel_amax.argtypes = [vp, i64, i64, vp]; lib.fqo_channel_amax.restype = None
        lib.fqo_select_channels.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.fqo_select_channels.restype = i32
        lib.fqo_quantize_outliers.argtypes = [i32, i32, u64, u32, vp, i64, i64, vp, i64, vp, vp,
                                              vp, vp, vp, vp, vp, vp]
        lib.fqo_quantize_outliers.restype = i32
        lib.fqo_osci_step.argtypes = [i32, i32, u64, u32, vp, vp, vp, vp, vp, vp, vp,
                                      vp, vp, vp, i64, i64, vp, vp, vp]
        lib.fqo_osci_step.restype = i32
        lib.fqo_osci_reset.argtypes = [i32, vp, vp, vp, vp, vp, vp, i64, i64, f32, vp]
        lib.fqo_osci_reset.restype = i64
        lib.fqo_qad_kl.argtypes = [vp, vp, i64, i64, ctypes.c_double, ctypes.c_double, vp, vp,
                                   vp, vp]
        lib.fqo_qad_kl.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(st, what):
    if st != 0:
        raise ValueError(f"oracle {what}: status {st}")


# --------------------------------------------------------------------------
# scalar primitives
# --------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return _load().fqo_e2m1_value(code)


def e2m1_round_nearest(y: float) -> int:
    return _load().fqo_e2m1_round_nearest(y)


def e2m1_round_stochastic(y: float, u: int) -> int:
    return _load().fqo_e2m1_round_stochastic(y, u)


def e4m3_value(code: int) -> float:
    return _load().fqo_e4m3_value(code)


def e4m3_encode(s: float) -> int:
    return _load().fqo_e4m3_encode(s)


def e8m0_value(code: int) -> float:
    return _load().fqo_e8m0_value(code)


def e8m0_for_amax(amax: float) -> int:
    return _load().fqo_e8m0_for_amax(amax)


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().fqo_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return [int(v) for v in out]


def sr_draw(seed: int, idx: int, stream: int = 0, offset: int = 0) -> int:
    return _load().fqo_sr_draw(seed, idx, stream, offset)


# --------------------------------------------------------------------------
# array helpers (exact conversions only)
# --------------------------------------------------------------------------
def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    u16 = np.ascontiguousarray(u16, dtype=np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, nearest-even, via the oracle's C routine."""
    flat = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    _load().fqo_bf16_from_f32_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(np.shape(x))


def rht_signs(rht_seed: int, offset: int = 0) -> int:
    return _load().fqo_rht_signs(rht_seed, offset)


def rht16(block, signs: int) -> np.ndarray:
    z = np.ascontiguousarray(block, dtype=np.float32).copy()
    assert z.size == 16
    _load().fqo_rht16(_ptr(z), signs)
    return z


def rht_rows(x: np.ndarray, rht_seed: int, offset: int = 0) -> np.ndarray:
    """The 16-point randomized Hadamard transform of every 1x16 block (a copy)."""
    z = np.ascontiguousarray(x, dtype=np.float32).copy()
    rows, cols = z.shape
    _load().fqo_rht_rows(_ptr(z), rows, cols, rht_seed, offset)
    return z


def amax(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return _load().fqo_amax(_ptr(x), x.size)


# --------------------------------------------------------------------------
# tensor operations
# --------------------------------------------------------------------------
def _quantize_rows(x, fmt, rounding, seed, offset, stream, tensor_amax,
                   want_xhat, want_mask):
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    B = BLOCK[fmt]
    n = rows * cols
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // B), dtype=np.uint8)
    if fmt == NVFP4:
        tscale = np.zeros(1, dtype=np.float32)
    elif fmt == NVFP4_2LEVEL:
        tscale = np.zeros((rows, max(cols // 128, 0)), dtype=np.float32)
    else:
        tscale = np.zeros(1, dtype=np.float32)
    xhat = np.zeros((rows, cols), dtype=np.float32) if want_xhat else None
    mask = np.zeros((n + 31) // 32, dtype=np.uint32) if want_mask else None
    st = lib.fqo_quantize_rows(fmt, rounding, seed, offset, stream, _ptr(x), rows, cols,
                               float(tensor_amax), _ptr(codes), _ptr(scales), _ptr(tscale),
                               _ptr(xhat), _ptr(mask))
    _check(st, "quantize_rows")
    out = {"codes": codes, "scales": scales}
    if fmt == NVFP4:
        out["tscale"] = tscale
    elif fmt == NVFP4_2LEVEL:
        out["tscale"] = tscale
    if want_xhat:
        out["xhat"] = xhat
    if want_mask:
        out["mask"] = mask
    return out


def quantize(x, fmt=NVFP4, rounding=RNE, seed=0, offset=0, orient=ROW,
             want_xhat=False, want_mask=False, amax_in=None, rht_seed=0):
    """Quantize a float32 [rows, cols] array.

    Row-wise outputs under "row"; for the column-wise orientation the row-wise
    definition is applied to the transpose (stream 1), with the same tensor
    amax (NVFP4), and returned under "col" (codes [cols, rows/2] etc.).
    xhat and mask are produced by the row-wise pass only.
    rht_seed != 0: each orientation first applies the 16-point randomized
    Hadamard transform to its own 1x16 blocks, and the NVFP4 tensor amax is
    that of the transformed tensor of the orientation.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    res = {}
    if orient & ROW:
        xr = rht_rows(x, rht_seed, offset) if rht_seed else x
        t_amax = amax(xr) if amax_in is None else float(amax_in)
        res["amax"] = np.float32(t_amax)
        res["row"] = _quantize_rows(xr, fmt, rounding, seed, offset, 0, t_amax,
                                    want_xhat, want_mask)
    if orient & COL:
        xt = np.ascontiguousarray(x.T)
        if rht_seed:
            xt = rht_rows(xt, rht_seed, offset)
        t_amax = amax(xt) if amax_in is None else float(amax_in)
        res.setdefault("amax", np.float32(t_amax))
        res["col_amax"] = np.float32(t_amax)
        res["col"] = _quantize_rows(xt, fmt, rounding, seed, offset, 1, t_amax, False, False)
    return res


def dequantize(q, rows, cols, fmt=NVFP4):
    lib = _load()
    codes = np.ascontiguousarray(q["codes"], dtype=np.uint8)
    scales = np.ascontiguousarray(q["scales"], dtype=np.uint8)
    tscale = np.ascontiguousarray(q.get("tscale", np.zeros(1, np.float32)), dtype=np.float32)
    xhat = np.zeros((rows, cols), dtype=np.float32)
    st = lib.fqo_dequantize_rows(fmt, _ptr(codes), _ptr(scales), _ptr(tscale), rows, cols,
                                 _ptr(xhat))
    _check(st, "dequantize_rows")
    return xhat


def ste_backward(dy: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """dy: uint16 (bf16 bits) or float32/uint32 array; returns the same dtype."""
    dy = np.ascontiguousarray(dy)
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    dx = np.empty_like(dy)
    _load().fqo_ste_backward(_ptr(dy), _ptr(mask), dy.size, dy.itemsize, _ptr(dx))
    return dx


def channel_amax(x: np.ndarray, amax_in=None) -> np.ndarray:
    """Running per-column max |x| (start from zeros when amax_in is None)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    a = (np.zeros(cols, np.float32) if amax_in is None
         else np.ascontiguousarray(amax_in, dtype=np.float32).copy())
    _load().fqo_channel_amax(_ptr(x), rows, cols, _ptr(a))
    return a


def select_channels(amax_c: np.ndarray, k: int):
    amax_c = np.ascontiguousarray(amax_c, dtype=np.float32)
    cols = amax_c.size
    idx = np.zeros(max(k, 1), np.int32)
    bitmap = np.zeros((cols + 31) // 32, np.uint32)
    scale = np.zeros(max(k, 1), np.float32)
    _check(_load().fqo_select_channels(_ptr(amax_c), cols, k, _ptr(idx), _ptr(bitmap),
                                       _ptr(scale)), "select_channels")
    return {"idx": idx[:k], "bitmap": bitmap, "fp8_scale": scale[:k]}


def quantize_outliers(x, idx, fp8_scale, fmt=NVFP4, rounding=RNE, seed=0, offset=0):
    """Split fake-quantization: FP4 for the tensor with the retained columns
    zeroed, FP8 E4M3 (static per-channel scales) for the retained columns."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    fp8_scale = np.ascontiguousarray(fp8_scale, dtype=np.float32)
    k = idx.size
    B = BLOCK[fmt]
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // B), np.uint8)
    tscale = (np.zeros((rows, max(cols // 128, 1)), np.float32) if fmt == NVFP4_2LEVEL
              else np.zeros(1, np.float32))
    fp8 = np.zeros((rows, max(k, 1)), np.uint8)
    xhat = np.zeros((rows, cols), np.float32)
    mask = np.zeros((rows * cols + 31) // 32, np.uint32)
    scratch = np.zeros_like(x)
    st = lib.fqo_quantize_outliers(fmt, rounding, seed, offset, _ptr(x), rows, cols,
                                   _ptr(idx), k, _ptr(fp8_scale), _ptr(scratch), _ptr(codes),
                                   _ptr(scales), _ptr(tscale), _ptr(fp8), _ptr(xhat), _ptr(mask))
    _check(st, "quantize_outliers")
    out = {"codes": codes, "scales": scales, "fp8": fp8[:, :k], "xhat": xhat, "mask": mask}
    if fmt != MXFP4:
        out["tscale"] = tscale
    return out


class OsciState:
    """Per-tensor OsciReset state: FP32 master, dist_Q, dist_M and the previous
    step's quantized tensor (codes, scales, tscale)."""

    def __init__(self, w0: np.ndarray, fmt=NVFP4, rounding=RNE, seed=0):
        self.fmt, self.rounding, self.seed = fmt, rounding, seed
        self.master = np.ascontiguousarray(w0, dtype=np.float32).copy()
        self.rows, self.cols = self.master.shape
        self.dist_q = np.zeros_like(self.master)
        self.dist_m = np.zeros_like(self.master)
        q = quantize(self.master, fmt, rounding, seed, 0, ROW)["row"]
        self.codes, self.scales = q["codes"], q["scales"]
        self.tscale = q.get("tscale", np.zeros(1, np.float32))

    def step(self, delta: np.ndarray, offset: int = 0):
        lib = _load()
        delta = np.ascontiguousarray(delta, dtype=np.float32)
        codes_new = np.zeros_like(self.codes)
        scales_new = np.zeros_like(self.scales)
        tscale_new = np.zeros_like(self.tscale)
        xhat = np.zeros_like(self.master)
        n = self.master.size
        mask = np.zeros((n + 31) // 32, dtype=np.uint32)
        scratch = np.zeros_like(self.master)
        st = lib.fqo_osci_step(self.fmt, self.rounding, self.seed, offset,
                               _ptr(self.master), _ptr(delta), _ptr(self.dist_q),
                               _ptr(self.dist_m), _ptr(self.codes), _ptr(self.scales),
                               _ptr(self.tscale), _ptr(codes_new), _ptr(scales_new),
                               _ptr(tscale_new), self.rows, self.cols, _ptr(xhat),
                               _ptr(mask), _ptr(scratch))
        _check(st, "osci_step")
        self.codes, self.scales, self.tscale = codes_new, scales_new, tscale_new
        return {"xhat": xhat, "mask": mask}

    def reset(self, threshold: float = 4.0) -> int:
        scratch = np.zeros_like(self.master)
        cnt = _load().fqo_osci_reset(self.fmt, _ptr(self.master), _ptr(self.dist_q),
                                     _ptr(self.dist_m), _ptr(self.codes), _ptr(self.scales),
                                     _ptr(self.tscale), self.rows, self.cols,
                                     float(threshold), _ptr(scratch))
        if cnt < 0:
            raise ValueError("oracle osci_reset failed")
        return int(cnt)


def qad_kl(zt: np.ndarray, zs: np.ndarray, temperature: float = 1.0, grad_scale=None,
           want_grad: bool = True):
    """QAD distillation loss of [rows, vocab] teacher / student logits (FP32
    values; widen BF16 first): per-row KL(softmax(zt/T) || softmax(zs/T)),
    their mean, and dz = g (q - p) / T with g = grad_scale (default 1/rows,
    the gradient of the mean).  All results in float64."""
    zt = np.ascontiguousarray(zt, dtype=np.float32)
    zs = np.ascontiguousarray(zs, dtype=np.float32)
    assert zt.shape == zs.shape and zt.ndim == 2
    rows, vocab = zt.shape
    g = (1.0 / rows if rows else 0.0) if grad_scale is None else float(grad_scale)
    loss = np.zeros(rows, np.float64)
    dz = np.zeros((rows, vocab), np.float64) if want_grad else None
    mean = np.zeros(1, np.float64)
    scratch = np.zeros(2 * vocab, np.float64)
    _check(_load().fqo_qad_kl(_ptr(zt), _ptr(zs), rows, vocab, float(temperature), g,
                              _ptr(loss), _ptr(mean), _ptr(dz) if want_grad else None,
                              _ptr(scratch)), "qad_kl")
    return {"loss_rows": loss, "loss_mean": float(mean[0]), "dz": dz}


def gemm(qa: dict, qb: dict, m: int, n: int, k: int, fmt=NVFP4) -> np.ndarray:
    """Block-scaled FP4 GEMM by its plain definition: C = deq(A) deq(B)^T for
    row-wise quantized A [m, k] and B [n, k] (both quantized along the shared
    reduction dimension k, as the forward GEMM of a QAT linear layer takes
    them), deq being `dequantize`.  The product is numpy's float64 matmul of
    the exactly widened dequantized operands."""
    a = dequantize(qa, m, k, fmt).astype(np.float64)
    b = dequantize(qb, n, k, fmt).astype(np.float64)
    return a @ b.T
