"""Host-side checks of the C ABI (no GPU): the library builds, loads and
exports every entry point include/fq.h declares, and argument errors come back
as the documented status codes before anything is launched."""
import ctypes
import os
import re

import pytest

from fp4_quantization_aware_fq_gb300 import build as fqbuild
from fp4_quantization_aware_fq_gb300 import fq


@pytest.fixture(scope="module")
def L():
    fqbuild.build()
    return fq.lib()


def test_header_declares_the_boundary():
    names = set(fq.declared_symbols())
    for n in ("fq_quantize", "fq_dequantize", "fq_fakequant_ste", "fq_osci_update",
              "fq_osci_reset", "fq_ste_backward", "fq_amax", "fq_workspace_size",
              "fq_osci_workspace_size", "fq_status_string", "fq_channel_amax",
              "fq_select_channels", "fq_quantize_outliers"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in fq.declared_symbols():
        assert hasattr(L, n), n


def test_status_strings(L):
    assert fq.fq_status_string(0) == "ok"
    for s in range(1, 7):
        assert fq.fq_status_string(s) not in ("ok", "unknown status")
    assert fq.fq_status_string(99) == "unknown status"


def test_workspace_sizes(L):
    assert fq.fq_workspace_size(fq.Config(fq.NVFP4), 256, 1024) >= 4
    assert fq.fq_workspace_size(fq.Config(fq.MXFP4), 256, 1024) == 0
    assert fq.fq_workspace_size(fq.Config(fq.NVFP4_2LEVEL), 256, 1024) == 0
    assert fq.fq_osci_workspace_size(64) >= 64 * 4
    assert fq.fq_osci_workspace_size(0) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails validation first


def _qt(codes=FAKE, scales=FAKE, tscale=FAKE):
    return fq._QT(codes, scales, tscale)


def _quant(L, cfg, x=FAKE, dtype=fq.BF16, rows=64, cols=64, orient=fq.ROW, row=None, col=None,
           ws=FAKE, wsb=256, ld=None):
    r = ctypes.byref(row) if row is not None else None
    c = ctypes.byref(col) if col is not None else None
    return L.fq_quantize(ctypes.byref(cfg), x, dtype, rows, cols, cols if ld is None else ld,
                         orient, r, c, None, ws, wsb, None)


def test_quantize_argument_errors(L):
    ok = fq.Config(fq.NVFP4)
    assert _quant(L, fq.Config(7)) == 1                                    # unknown format
    assert _quant(L, fq.Config(fq.NVFP4, 5)) == 1                          # unknown rounding
    assert _quant(L, ok, dtype=9, row=_qt()) == 1                          # unknown dtype
    assert _quant(L, ok, x=0, row=_qt()) == 1                              # NULL input
    assert _quant(L, ok, orient=0, row=_qt()) == 1                         # bad orientation
    assert _quant(L, ok, orient=fq.ROW, row=None) == 1                     # missing output
    assert _quant(L, ok, cols=40, row=_qt()) == 2                          # cols % 16
    assert _quant(L, fq.Config(fq.MXFP4), cols=48, row=_qt()) == 2         # cols % 32
    assert _quant(L, fq.Config(fq.NVFP4_2LEVEL), cols=64, row=_qt()) == 2  # cols % 128
    assert _quant(L, ok, rows=40, orient=fq.COL, col=_qt()) == 2           # rows % 16
    assert _quant(L, fq.Config(fq.NVFP4_2LEVEL), rows=64, cols=128, orient=fq.COL,
                  col=_qt()) == 2                                          # rows % 128
    assert _quant(L, ok, rows=-1, row=_qt()) == 2
    assert _quant(L, ok, x=FAKE + 8, row=_qt()) == 3                       # misaligned input
    assert _quant(L, ok, row=_qt(codes=FAKE + 4)) == 3                     # misaligned codes
    assert _quant(L, ok, row=_qt(tscale=0)) == 1                           # NVFP4 needs tscale
    assert _quant(L, ok, row=_qt(), ws=0) == 4                             # no workspace
    assert _quant(L, ok, row=_qt(), wsb=2) == 4                            # workspace too small
    # the row pitch: at least cols, a multiple of 16 bytes, addressable
    assert _quant(L, ok, ld=48, row=_qt()) == 2                            # ld < cols
    assert _quant(L, ok, ld=68, row=_qt()) == 3                            # 136-byte BF16 rows
    assert _quant(L, ok, dtype=fq.F32, rows=0, ld=68, row=_qt()) == 0      # 272-byte FP32 rows
    assert _quant(L, ok, rows=1 << 40, ld=1 << 40, row=_qt()) == 2         # extent overflows
    assert _quant(L, ok, rows=0, ld=72, row=_qt()) == 0                    # padded, empty


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_empty_tensors_succeed_without_touching_the_device(L, fmt):
    """rows * cols == 0 is a valid call that does nothing: FQ_OK, returned before
    any CUDA call (on a machine without a GPU any call would come back as
    FQ_ERR_CUDA, so these also show that nothing was launched)."""
    cfg = fq.Config(fmt)
    c = ctypes.byref(cfg)
    q, q2 = _qt(), _qt()
    assert _quant(L, cfg, rows=0, cols=128, row=q) == 0
    assert _quant(L, cfg, rows=0, cols=128, orient=fq.ROWCOL, row=q, col=q2) == 0
    assert _quant(L, cfg, rows=128, cols=0, row=q) == 0
    assert L.fq_fakequant_ste(c, FAKE, fq.BF16, 0, 128, 128, FAKE, fq.BF16, FAKE,
                              ctypes.byref(q), None, None, FAKE, 256, None) == 0
    assert L.fq_dequantize(c, ctypes.byref(q), 0, 128, FAKE, fq.F32, 128, None) == 0
    assert L.fq_ste_backward(FAKE, fq.BF16, FAKE, 0, FAKE, None) == 0


def test_hadamard_transform_needs_block_local_scales(L):
    cfg = fq.Config(fq.NVFP4, fq.SR, 1, 0, rht_seed=7)
    assert _quant(L, cfg, row=_qt()) == 5                                  # unsupported
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows, cols = (i64 * 1)(64), (i64 * 1)(64)
    ptrs = (vp * 1)(FAKE)
    qs = (fq._QT * 1)(_qt())
    assert L.fq_osci_update(ctypes.byref(cfg), 1, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs,
                            None, fq.BF16, None, FAKE, 256, None) == 5


def test_fakequant_dequant_ste_amax_errors(L):
    cfg = fq.Config(fq.NVFP4)
    f = L.fq_fakequant_ste
    assert f(ctypes.byref(cfg), FAKE, fq.BF16, 64, 64, 64, None, fq.BF16, None, None, None, None,
             FAKE, 256, None) == 1                                         # xhat required
    assert f(ctypes.byref(cfg), FAKE, fq.BF16, 64, 64, 64, FAKE + 2, fq.BF16, None, None, None,
             None, FAKE, 256, None) == 3
    assert f(ctypes.byref(cfg), FAKE, fq.BF16, 64, 64, 64, FAKE, 5, None, None, None, None,
             FAKE, 256, None) == 1
    assert f(ctypes.byref(cfg), FAKE, fq.BF16, 64, 64, 32, FAKE, fq.BF16, None, None, None, None,
             FAKE, 256, None) == 2                                         # ld < cols
    assert f(ctypes.byref(cfg), FAKE, fq.BF16, 64, 64, 100, FAKE, fq.BF16, None, None, None,
             None, FAKE, 256, None) == 3                                   # 200-byte rows
    q = _qt()
    d = L.fq_dequantize
    assert d(ctypes.byref(cfg), ctypes.byref(q), 64, 24, FAKE, fq.F32, 24, None) == 2
    assert d(ctypes.byref(cfg), None, 64, 64, FAKE, fq.F32, 64, None) == 1
    assert d(ctypes.byref(cfg), ctypes.byref(q), 64, 64, FAKE + 1, fq.F32, 64, None) == 3
    assert d(ctypes.byref(cfg), ctypes.byref(q), 64, 64, FAKE, fq.F32, 60, None) == 2  # ldy < cols
    assert d(ctypes.byref(cfg), ctypes.byref(q), 64, 64, FAKE, fq.F32, 66, None) == 3  # 264 B rows
    assert d(ctypes.byref(cfg), ctypes.byref(q), 64, 64, FAKE, fq.BF16, 68, None) == 3  # 136 B rows
    assert L.fq_ste_backward(FAKE, fq.BF16, FAKE, 12, FAKE, None) == 2
    assert L.fq_ste_backward(FAKE, fq.BF16, None, 16, FAKE, None) == 1
    assert L.fq_ste_backward(FAKE + 2, fq.BF16, FAKE, 16, FAKE, None) == 3
    assert L.fq_amax(FAKE, fq.F32, 12, FAKE, None) == 2
    assert L.fq_amax(FAKE, fq.F32, 16, None, None) == 1


def test_osci_argument_errors(L):
    cfg = fq.Config(fq.NVFP4)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = (i64 * 2)(64, 64)
    cols = (i64 * 2)(64, 40)
    ptrs = (vp * 2)(FAKE, FAKE)
    qs = (fq._QT * 2)(_qt(), _qt())
    u = L.fq_osci_update
    assert u(ctypes.byref(cfg), 2, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16,
             None, FAKE, 256, None) == 2                                   # 40 % 16 != 0
    cols[1] = 64
    assert u(ctypes.byref(cfg), 2, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16,
             None, None, 0, None) == 4                                     # no workspace
    assert u(ctypes.byref(cfg), 2, rows, cols, None, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16,
             None, FAKE, 256, None) == 1
    bad = (vp * 2)(FAKE, FAKE + 4)
    assert u(ctypes.byref(cfg), 2, rows, cols, bad, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16,
             None, FAKE, 256, None) == 3
    assert u(ctypes.byref(cfg), -1, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16,
             None, FAKE, 256, None) == 1
    r = L.fq_osci_reset
    assert r(ctypes.byref(cfg), 2, rows, cols, ptrs, ptrs, ptrs, None, 4.0, None, None) == 1
    assert r(ctypes.byref(cfg), 2, rows, cols, ptrs, ptrs, ptrs, qs, 4.0, FAKE + 4, None) == 3


def test_osci_update_reset_and_noalloc_argument_errors(L):
    cfg = fq.Config(fq.NVFP4)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    rows = (i64 * 2)(64, 64)
    cols = (i64 * 2)(64, 40)
    ptrs = (vp * 2)(FAKE, FAKE)
    qs = (fq._QT * 2)(_qt(), _qt())
    ur = L.fq_osci_update_reset
    c = ctypes.byref(cfg)
    assert ur(c, 2, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None, 4.0,
              None, FAKE, 256, None) == 2                                  # 40 % 16 != 0
    cols[1] = 64
    assert ur(c, 2, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None, 4.0,
              None, None, 0, None) == 4                                    # no workspace
    assert ur(c, 2, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None, 4.0,
              FAKE + 4, FAKE, 256, None) == 3                              # n_reset not 8-aligned
    assert ur(c, 2, rows, cols, ptrs, None, ptrs, ptrs, qs, qs, None, fq.BF16, None, 4.0,
              None, FAKE, 256, None) == 1                                  # no delta
    assert ur(c, -1, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None, 4.0,
              None, FAKE, 256, None) == 1
    na = L.fq_osci_update_noalloc
    header = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                               "include", "fq.h")).read()
    cap = int(re.search(r"#define FQ_NOALLOC_MAX_TENSORS (\d+)", header).group(1))
    assert na(c, cap + 1, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None,
              None) == 4                                                   # beyond its scratch
    assert na(c, -1, rows, cols, ptrs, ptrs, ptrs, ptrs, qs, qs, None, fq.BF16, None,
              None) == 1
    assert na(c, 0, None, None, None, None, None, None, None, None, None, fq.BF16, None,
              None) == 0                                                   # nothing to do


def test_outlier_argument_errors(L):
    # channel amax
    assert L.fq_channel_amax(FAKE, 9, 64, 64, FAKE, None) == 1             # unknown dtype
    assert L.fq_channel_amax(FAKE, fq.F32, 64, 64, 0, None) == 1           # NULL amax
    assert L.fq_channel_amax(FAKE, fq.F32, 64, 40, FAKE, None) == 2        # cols % 16
    assert L.fq_channel_amax(FAKE + 4, fq.F32, 64, 64, FAKE, None) == 3    # misaligned
    # selection
    sel = L.fq_select_channels
    assert sel(0, 64, 4, FAKE, FAKE, FAKE, None) == 1                      # NULL amax
    assert sel(FAKE, 64, 4, 0, FAKE, FAKE, None) == 1                      # NULL idx, k > 0
    assert sel(FAKE, 64, 65, FAKE, FAKE, FAKE, None) == 1                  # k > cols
    assert sel(FAKE, 64, -1, FAKE, FAKE, FAKE, None) == 1                  # k < 0
    assert sel(FAKE, fq.MAX_CHANNELS + 32, 4, FAKE, FAKE, FAKE, None) == 2  # too many channels
    assert sel(FAKE, 64, 4, FAKE + 4, FAKE, FAKE, None) == 3               # misaligned idx
    assert sel(FAKE, 0, 0, 0, FAKE, 0, None) == 0                          # nothing to select

    # split quantization
    def q(cfg=fq.Config(fq.NVFP4), x=FAKE, rows=64, cols=64, bm=FAKE, k=4, sc=FAKE, out=None,
          fp8=FAKE, ws=FAKE, wsb=256):
        o = ctypes.byref(out) if out is not None else None
        return L.fq_quantize_outliers(ctypes.byref(cfg), x, fq.F32, rows, cols, bm, k, sc, o,
                                      fp8, None, fq.F32, None, ws, wsb, None)
    assert q(cfg=fq.Config(7)) == 1                                        # unknown format
    assert q(bm=0) == 1                                                    # NULL bitmap
    assert q(sc=0) == 1                                                    # NULL scales, k > 0
    assert q(k=65) == 1                                                    # k > cols
    assert q(cols=40) == 2                                                 # cols % 16
    assert q(cfg=fq.Config(fq.NVFP4_2LEVEL), cols=64) == 2                 # cols % 128
    assert q(cols=fq.MAX_CHANNELS + 16) == 2                               # too many channels
    assert q(cfg=fq.Config(fq.MXFP4, fq.SR, 1, 0, rht_seed=3)) == 5        # no transform here
    assert q(x=FAKE + 8) == 3                                              # misaligned input
    assert q(out=_qt(scales=FAKE + 1)) == 3                                # misaligned scales
    assert q(out=_qt(tscale=0)) == 1                                       # NVFP4 needs tscale
    assert q(ws=0) == 4                                                    # no workspace
    assert q(cfg=fq.Config(fq.MXFP4), ws=0, wsb=0, rows=0) == 0            # empty: nothing runs


def test_qad_kl_argument_errors(L):
    def k(zt=FAKE, zs=FAKE, dtype=fq.BF16, rows=4, vocab=64, T=1.0, g=1.0, lr=FAKE, lm=FAKE,
          dz=FAKE, dzt=fq.BF16, err=FAKE):
        return L.fq_qad_kl(zt, zs, dtype, rows, vocab, T, g, lr, lm, dz, dzt, err, None)
    assert k(dtype=7) == 1                       # unknown dtype
    assert k(zs=0) == 1                          # NULL student
    assert k(lr=0) == 1                          # NULL per-row losses
    assert k(dzt=9) == 1                         # unknown gradient dtype
    assert k(T=0.0) == 1                         # temperature must be > 0
    assert k(T=float("inf")) == 1
    assert k(g=float("nan")) == 1
    assert k(vocab=60) == 2                      # vocab % 8
    assert k(vocab=0) == 2
    assert k(rows=-1) == 2
    assert k(zt=FAKE + 8) == 3                   # misaligned logits
    assert k(dz=FAKE + 4) == 3                   # misaligned gradient
    assert k(vocab=460000) == 5                  # a BF16 row no longer fits one cluster
    assert k(dtype=fq.F32, vocab=230000) == 5    # nor an FP32 one


def test_gemm_argument_errors(L):
    def g(cfg=fq.Config(fq.NVFP4), a=None, b=None, m=128, n=128, k=256, c=FAKE, ct=fq.F32,
          ws=FAKE, wsb=1 << 20, err=FAKE):
        qa = a if a is not None else _qt()
        qb = b if b is not None else _qt()
        return L.fq_gemm(ctypes.byref(cfg), ctypes.byref(qa), ctypes.byref(qb), m, n, k, c, ct,
                         ws, wsb, err, None)
    assert fq.fq_gemm_workspace_size(256, 128, 512) == (256 + 128) * 512 // 16
    assert fq.fq_gemm_workspace_size(200, 96, 2880) == (256 + 128) * 3072 // 16  # padded
    assert g(cfg=fq.Config(9)) == 1                       # unknown format
    assert g(c=0) == 1                                    # NULL output
    assert g(ct=5) == 1                                   # unknown output dtype
    assert g(cfg=fq.Config(fq.NVFP4_2LEVEL)) == 5          # NVFP4 and MXFP4 only
    assert g(cfg=fq.Config(fq.MXFP4, rht_seed=3)) == 5
    assert g(a=_qt(tscale=0)) == 1                        # NVFP4 needs the tensor scale
    assert g(b=_qt(codes=FAKE + 4)) == 3                  # misaligned codes
    assert g(n=48) == 2                                   # n % 32
    assert g(k=48) == 2                                   # k % 32
    assert g(c=FAKE + 8) == 3                             # misaligned output
    assert g(ws=0) == 4                                   # no workspace
    assert g(wsb=100) == 4                                # workspace too small
    assert g(ws=FAKE + 8) == 3                            # misaligned workspace
    assert g(m=0) == 0                                    # empty: nothing runs
