"""Bounds checks without a sanitizer: every output of every entry point is
placed inside a larger buffer with a guard band of 0xA5 bytes on each side,
the call runs on small shapes whose tiles, blocks and chunks have ragged
edges, and the guard bands must come back untouched.  A write past either
end of an output (a tile edge store, a scattered 1- or 2-byte store, a GEMM
epilogue chunk, an OsciReset tail) changes a guard byte.  The outputs are
also compared with the oracle, so a write that lands in the wrong place
inside an output fails too.

The column-only MXFP4 case with cols % 32 == 16 is the shape in which the
tile loader once fetched a whole 1x32 row block past the end of each row; it
is run here on inputs of exactly that size.
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
GUARD = 4096
PAT = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` inside a buffer with GUARD bytes
    of PAT before and after it."""

    def __init__(self, shape, dtype, fill=PAT):
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        body = (self.nbytes + 15) // 16 * 16
        self.buf = torch.full((GUARD + body + GUARD,), PAT, dtype=torch.uint8, device=DEV)
        self.buf[GUARD:GUARD + self.nbytes] = fill
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self) -> bool:
        b = npy(self.buf)
        return bool((b[:GUARD] == PAT).all() and (b[GUARD + self.nbytes:] == PAT).all())


def guarded_q(rows, cols, fmt):
    """A quantized-tensor descriptor whose codes, scales and tensor scales are
    each guarded and sized exactly as the header states."""
    B = fq.BLOCK[fmt]
    parts = {"codes": Guarded((rows, cols // 2), torch.uint8),
             "scales": Guarded((rows, cols // B), torch.uint8)}
    if fmt == fq.NVFP4:
        parts["tscale"] = Guarded((1,), torch.float32)
    elif fmt == fq.NVFP4_2LEVEL:
        parts["tscale"] = Guarded((rows, cols // 128), torch.float32)
    q = fq.QTensor(parts["codes"].t, parts["scales"].t,
                   parts["tscale"].t if "tscale" in parts else None)
    return q, parts


def assert_intact(named):
    for name, g in named.items():
        assert g.intact(), f"write outside {name}"


# ------------------------------------------------------------------ quantizers
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols", [48, 80])
def test_mxfp4_col_only_half_row_block(dtype, cols):
    """MXFP4 column-wise with cols % 32 == 16 (allowed: the row pass is not
    run), on an input of exactly [rows, cols]."""
    rows = 96
    x = W.nvfp4_act(shape=(rows, cols), seed=cols, n_outlier_cols=2).to(dtype).to(DEV)
    cq, parts = guarded_q(cols, rows, fq.MXFP4)
    fq.fq_quantize(x, fq.Config(fq.MXFP4), orient=fq.COL, col_out=cq)
    torch.cuda.synchronize()
    assert_intact(parts)
    ref = oracle.quantize(as_oracle_input(x), oracle.MXFP4, orient=oracle.COL)
    check_q("col", cq, ref["col"], fq.MXFP4)


@pytest.mark.parametrize("fmt,rows,cols", [(fq.NVFP4, 144, 80), (fq.MXFP4, 96, 160),
                                           (fq.NVFP4_2LEVEL, 256, 384)])
@pytest.mark.parametrize("rnd", [fq.RNE, fq.SR])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fakequant_rowcol_guards(fmt, rows, cols, rnd, dtype):
    """Row + column tiles with ragged edges in both directions: codes, scales,
    tensor scales, xhat and mask of both orientations stay inside their
    buffers."""
    x = W.nvfp4_act(shape=(rows, cols), seed=rows + cols, n_outlier_cols=3).to(dtype).to(DEV)
    rq, rparts = guarded_q(rows, cols, fmt)
    cq, cparts = guarded_q(cols, rows, fmt)
    xhat = Guarded((rows, cols), dtype)
    mask = Guarded(((rows * cols + 7) // 8,), torch.uint8)
    cfg = fq.Config(fmt, rnd, 0x1234, 5)
    fq.fq_fakequant_ste(x, cfg, xhat=xhat.t, mask=mask.t, row_out=rq, col_out=cq)
    torch.cuda.synchronize()
    assert_intact({**{"row." + k: v for k, v in rparts.items()},
                   **{"col." + k: v for k, v in cparts.items()}, "xhat": xhat, "mask": mask})
    ref = oracle.quantize(as_oracle_input(x), FMT_O[fmt], rnd, 0x1234, 5, orient=oracle.ROWCOL,
                          want_xhat=True, want_mask=True)
    check_q("row", rq, ref["row"], fmt)
    check_q("col", cq, ref["col"], fmt)
    want = (oracle.f32_to_bf16_bits(ref["row"]["xhat"]) if dtype == torch.bfloat16
            else ref["row"]["xhat"].view(np.uint32))
    assert_eq("xhat", bits(xhat.t), want)
    assert_eq("mask", npy(mask.t), ref["row"]["mask"].view(np.uint8)[:mask.nbytes])


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
def test_row_only_and_hadamard_guards(fmt):
    """Row-wise only, on a row count that leaves the last CTA partly idle;
    MXFP4 and the double block also with the Hadamard transform."""
    rows, cols = 37, 384
    x = W.grad_2level(shape=(rows, cols), seed=9).to(DEV)
    for rht in ((0, 0xB00F) if fmt != fq.NVFP4 else (0,)):
        rq, parts = guarded_q(rows, cols, fmt)
        cfg = fq.Config(fmt, fq.SR, 7, 1, rht)
        fq.fq_quantize(x, cfg, row_out=rq)
        torch.cuda.synchronize()
        assert_intact(parts)
        ref = oracle.quantize(as_oracle_input(x), FMT_O[fmt], fq.SR, 7, 1, rht_seed=rht)
        check_q("row", rq, ref["row"], fmt)


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4, fq.NVFP4_2LEVEL])
@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_dequantize_and_ste_guards(fmt, ydt):
    rows, cols = 24, 256
    x = W.grad_2level(shape=(rows, cols), seed=4).to(DEV)
    cfg = fq.Config(fmt)
    rq, _ = fq.fq_quantize(x, cfg)
    y = Guarded((rows, cols), ydt)
    fq.fq_dequantize(rq, rows, cols, cfg, y=y.t)
    _, mask, _, _ = fq.fq_fakequant_ste(x, cfg, want_mask=True)
    dy = W.normal((rows, cols), 1.0, seed=3).to(ydt).to(DEV)
    dx = Guarded((rows, cols), ydt)
    fq.fq_ste_backward(dy, mask, dx=dx.t)
    torch.cuda.synchronize()
    assert_intact({"y": y, "dx": dx})
    q = {"codes": npy(rq.codes), "scales": npy(rq.scales)}
    if rq.tscale is not None:
        q["tscale"] = npy(rq.tscale)
    ref = oracle.dequantize(q, rows, cols, FMT_O[fmt])
    assert_eq("y", bits(y.t), oracle.f32_to_bf16_bits(ref) if ydt == torch.bfloat16
              else ref.view(np.uint32))
    want = oracle.ste_backward(bits(dy).reshape(-1), npy(mask).view(np.uint8)[:rows * cols // 8]
                               .copy().view(np.uint32))
    assert_eq("dx", bits(dx.t).reshape(-1), want)


# ------------------------------------------------------------------ OsciReset
@pytest.mark.parametrize("fused", [False, True])
def test_osci_tail_guards(fused):
    """Grouped OsciReset update (and the fused window-end reset) on tensors
    whose sizes end inside a tile of 16-byte chunks: every per-weight output
    and the ping-pong quantized buffers stay inside their buffers."""
    shapes = [(3, 16), (17, 48), (129, 32), (5, 2064)]
    fmt = fq.NVFP4
    cfg = fq.Config(fmt, fq.SR, 11, 1)
    master0 = [W.normal(s, 0.02, seed=70 + i) for i, s in enumerate(shapes)]
    deltas = [W.master_update(s, 1, std=3e-3) for s in shapes]
    g = {}
    master, dq, dm, xh, mk, nxt = [], [], [], [], [], []
    for i, s in enumerate(shapes):
        n = s[0] * s[1]
        g[f"master{i}"] = Guarded(s, torch.float32)
        g[f"master{i}"].t.copy_(master0[i].to(DEV))
        g[f"dq{i}"] = Guarded(s, torch.float32)
        g[f"dq{i}"].t.zero_()
        g[f"dm{i}"] = Guarded(s, torch.float32)
        g[f"dm{i}"].t.zero_()
        g[f"xhat{i}"] = Guarded(s, torch.bfloat16)
        g[f"mask{i}"] = Guarded(((n + 7) // 8,), torch.uint8)
        q, parts = guarded_q(s[0], s[1], fmt)
        for k, v in parts.items():
            g[f"next{i}.{k}"] = v
        master.append(g[f"master{i}"].t)
        dq.append(g[f"dq{i}"].t)
        dm.append(g[f"dm{i}"].t)
        xh.append(g[f"xhat{i}"].t)
        mk.append(g[f"mask{i}"].t)
        nxt.append(q)
    prev = [fq.fq_quantize(m, fq.Config(fmt, fq.SR, 11, 0))[0] for m in master]
    dd = [d.to(DEV) for d in deltas]
    cnt = Guarded((1,), torch.int64)
    cnt.t.zero_()
    if fused:
        fq.fq_osci_update_reset(cfg, master, dd, dq, dm, prev, nxt, 4.0, n_reset=cnt.t,
                                xhat=xh, mask=mk)
        g["n_reset"] = cnt
    else:
        fq.fq_osci_update(cfg, master, dd, dq, dm, prev, nxt, xhat=xh, mask=mk)
    torch.cuda.synchronize()
    assert_intact(g)
    for i, s in enumerate(shapes):
        st = oracle.OsciState(master0[i].numpy(), oracle.NVFP4, fq.SR, seed=11)
        out = st.step(deltas[i].numpy(), offset=1)
        if fused:
            st.reset(4.0)
        assert_eq(f"master{i}", bits(master[i]), st.master.view(np.uint32))
        assert_eq(f"dq{i}", bits(dq[i]), st.dist_q.view(np.uint32))
        assert_eq(f"xhat{i}", bits(xh[i]), oracle.f32_to_bf16_bits(out["xhat"]))
        assert_eq(f"dm{i}", bits(dm[i]), st.dist_m.view(np.uint32))
        assert_eq(f"codes{i}", npy(nxt[i].codes), st.codes)
        assert_eq(f"scales{i}", npy(nxt[i].scales), st.scales)
        n = s[0] * s[1]
        assert_eq(f"mask{i}", npy(mk[i]), out["mask"].view(np.uint8)[:(n + 7) // 8])


# ------------------------------------------------------------------ outlier retention
@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4])
def test_outlier_guards(fmt):
    """Split FP4 / FP8 quantization: the FP8 columns, the FP4 tensor, xhat and
    mask (scattered 1- and 2-byte stores of the kept elements) stay inside
    their buffers; selection outputs too."""
    rows, cols, k = 48, 96, 7
    x = W.channel_act((rows, cols), seed=5, n_outlier_cols=6).to(DEV)
    amax = Guarded((cols,), torch.float32, fill=0)
    fq.fq_channel_amax(x, amax.t)
    idx = Guarded((k,), torch.int32)
    bitmap = Guarded(((cols + 31) // 32,), torch.int32)
    scl = Guarded((k,), torch.float32)
    st = fq.lib().fq_select_channels(amax.t.data_ptr(), cols, k, idx.t.data_ptr(),
                                     bitmap.t.data_ptr(), scl.t.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == 0
    sel = fq.Outliers(idx.t, bitmap.t, scl.t)
    out, parts = guarded_q(rows, cols, fmt)
    fp8 = Guarded((rows, k), torch.uint8)
    xhat = Guarded((rows, cols), torch.bfloat16)
    mask = Guarded(((rows * cols + 7) // 8,), torch.uint8)
    cfg = fq.Config(fmt)
    fq.fq_quantize_outliers(x, cfg, sel, out=out, fp8=fp8.t, xhat=xhat.t, mask=mask.t)
    torch.cuda.synchronize()
    assert_intact({"amax": amax, "idx": idx, "bitmap": bitmap, "fp8_scale": scl, "fp8": fp8,
                   "xhat": xhat, "mask": mask, **parts})
    xo = as_oracle_input(x)
    rsel = oracle.select_channels(oracle.channel_amax(xo), k)
    assert_eq("idx", npy(idx.t), rsel["idx"])
    ref = oracle.quantize_outliers(xo, rsel["idx"], rsel["fp8_scale"], FMT_O[fmt])
    check_q("fp4", out, ref, fmt)
    assert_eq("fp8", npy(fp8.t), ref["fp8"][:, :k])
    assert_eq("xhat", bits(xhat.t), oracle.f32_to_bf16_bits(ref["xhat"]))
    assert_eq("mask", npy(mask.t), ref["mask"].view(np.uint8)[:mask.nbytes])


# ------------------------------------------------------------------ QAD loss and GEMM
def test_qad_guards():
    rows, vocab = 5, 1000
    zt, zs = W.qad_logits((rows, vocab), seed=3)
    zt, zs = zt.to(DEV), zs.to(DEV)
    loss = Guarded((rows,), torch.float32)
    mean = Guarded((1,), torch.float32)
    dz = Guarded((rows, vocab), torch.bfloat16)
    err = Guarded((1,), torch.int32, fill=0)
    fq.fq_qad_kl(zt, zs, loss_rows=loss.t, loss_mean=mean.t, dz=dz.t, err=err.t)
    torch.cuda.synchronize()
    assert int(err.t.item()) == 0
    assert_intact({"loss_rows": loss, "loss_mean": mean, "dz": dz, "err": err})
    ref = oracle.qad_kl(as_oracle_input(zt), as_oracle_input(zs))
    got = npy(loss.t).astype(np.float64)
    assert np.all(np.abs(got - ref["loss_rows"]) <= 2e-5 + 1e-4 * np.abs(ref["loss_rows"]))


@pytest.mark.parametrize("fmt", [fq.NVFP4, fq.MXFP4])
@pytest.mark.parametrize("cdt", [torch.float32, torch.bfloat16])
def test_gemm_guards(fmt, cdt):
    """m, n and k off the 128 x 128 x 256 tile grid: the guarded epilogue and
    the scale-layout workspace stay inside their buffers."""
    m, n, k = 130, 96, 96
    a = W.normal((m, k), 1.0, seed=31).to(DEV)
    b = W.normal((n, k), 0.02, seed=32).to(DEV)
    cfg = fq.Config(fmt)
    qa, _ = fq.fq_quantize(a, cfg)
    qb, _ = fq.fq_quantize(b, cfg)
    c = Guarded((m, n), cdt)
    ws = Guarded((fq.fq_gemm_workspace_size(m, n, k),), torch.uint8)
    err = Guarded((1,), torch.int32, fill=0)
    fq.fq_gemm(qa, qb, m, n, k, cfg, c=c.t, ws=ws.t, err=err.t)
    torch.cuda.synchronize()
    assert int(err.t.item()) == 0
    assert_intact({"c": c, "ws": ws, "err": err})

    def qd(q):
        d = {"codes": npy(q.codes), "scales": npy(q.scales)}
        if q.tscale is not None:
            d["tscale"] = npy(q.tscale)[:1]
        return d
    da = oracle.dequantize(qd(qa), m, k, FMT_O[fmt]).astype(np.float64)
    db = oracle.dequantize(qd(qb), n, k, FMT_O[fmt]).astype(np.float64)
    ref = da @ db.T
    bound = 2.0 ** -16 * (np.abs(da) @ np.abs(db).T)
    if cdt == torch.bfloat16:
        bound = bound + 2.0 ** -8 * np.abs(ref)
    got = npy(c.t.float()).astype(np.float64)
    assert np.all(np.abs(got - ref) <= bound)
