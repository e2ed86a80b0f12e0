"""OsciReset update / reset on the GPU vs the oracle, bit for bit."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W
from gpu_common import FMT_O, assert_eq, bits, npy

pytestmark = pytest.mark.gpu
DEV = "cuda"


class GpuOsci:
    """Device-side state of a group of tensors (ping-pong quantized buffers)."""

    def __init__(self, ws_bf16, cfg):
        self.cfg = cfg
        self.master = [w.float().to(DEV).contiguous() for w in ws_bf16]
        self.dq = [torch.zeros_like(m) for m in self.master]
        self.dm = [torch.zeros_like(m) for m in self.master]
        init_cfg = fq.Config(cfg.format, cfg.rounding, cfg.seed, 0)
        self.prev = [fq.fq_quantize(m, init_cfg)[0] for m in self.master]
        self.next = [fq.alloc_qtensor(*m.shape, cfg.format, DEV) for m in self.master]
        self.xhat = [torch.empty(m.shape, dtype=torch.bfloat16, device=DEV) for m in self.master]
        self.mask = [torch.empty(((m.numel() + 7) // 8 + 15) // 16 * 16, dtype=torch.uint8,
                                 device=DEV) for m in self.master]

    def step(self, deltas, t):
        cfg = fq.Config(self.cfg.format, self.cfg.rounding, self.cfg.seed, t)
        fq.fq_osci_update(cfg, self.master, deltas, self.dq, self.dm, self.prev, self.next,
                          xhat=self.xhat, mask=self.mask)
        self.prev, self.next = self.next, self.prev

    def reset(self, thr):
        cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
        fq.fq_osci_reset(self.cfg, self.master, self.dq, self.dm, self.prev, thr, n_reset=cnt)
        return cnt


def _compare(name, g: GpuOsci, i, st: oracle.OsciState, out=None):
    assert_eq(f"{name}.master", bits(g.master[i]), st.master.view(np.uint32))
    assert_eq(f"{name}.dist_q", bits(g.dq[i]), st.dist_q.view(np.uint32))
    assert_eq(f"{name}.dist_m", bits(g.dm[i]), st.dist_m.view(np.uint32))
    assert_eq(f"{name}.codes", npy(g.prev[i].codes), st.codes)
    assert_eq(f"{name}.scales", npy(g.prev[i].scales), st.scales)
    if g.cfg.format == fq.NVFP4:
        assert_eq(f"{name}.tscale", npy(g.prev[i].tscale)[:1].view(np.uint32),
                  st.tscale.reshape(-1)[:1].view(np.uint32))
    if out is not None:
        assert_eq(f"{name}.xhat", bits(g.xhat[i]), oracle.f32_to_bf16_bits(out["xhat"]))
        n = g.master[i].numel()
        assert_eq(f"{name}.mask", npy(g.mask[i])[: (n + 7) // 8],
                  out["mask"].view(np.uint8)[: (n + 7) // 8])


@pytest.mark.parametrize("fmt,rnd", [(fq.NVFP4, fq.RNE), (fq.NVFP4, fq.SR), (fq.MXFP4, fq.RNE),
                                     (fq.NVFP4_2LEVEL, fq.SR)])
def test_osci_group_matches_oracle(fmt, rnd):
    shapes = [(96, 256), (256, 128), (48, 384), (128, 128)]
    ws = [W.normal(s, 0.02, seed=40 + i).to(torch.bfloat16) for i, s in enumerate(shapes)]
    cfg = fq.Config(fmt, rnd, seed=77)
    g = GpuOsci(ws, cfg)
    sts = [oracle.OsciState(w.float().numpy(), FMT_O[fmt], rnd, seed=77) for w in ws]
    for t in range(1, 4):
        deltas = [W.master_update(s, t, std=3e-3) for s in shapes]   # large enough to flip bins
        g.step([d.to(DEV) for d in deltas], t)
        torch.cuda.synchronize()
        for i, (st, d) in enumerate(zip(sts, deltas)):
            out = st.step(d.numpy(), offset=t)
            _compare(f"t{t}.{i}", g, i, st, out)
    cnt = g.reset(4.0)
    torch.cuda.synchronize()
    total = sum(st.reset(4.0) for st in sts)
    assert int(cnt.item()) == total
    assert total > 0
    for i, st in enumerate(sts):
        _compare(f"reset.{i}", g, i, st)


@pytest.mark.parametrize("fmt,rnd", [(fq.NVFP4, fq.RNE), (fq.NVFP4_2LEVEL, fq.SR),
                                     (fq.MXFP4, fq.RNE)])
def test_fused_window_end_reset_matches_update_then_reset(fmt, rnd):
    """fq_osci_update_reset == fq_osci_update followed by fq_osci_reset, and
    both equal the oracle's step + reset."""
    shapes = [(64, 256), (128, 384), (32, 128)]
    ws = [W.normal(s, 0.02, seed=80 + i).to(torch.bfloat16) for i, s in enumerate(shapes)]
    cfg = fq.Config(fmt, rnd, seed=5)
    g = GpuOsci(ws, cfg)
    sts = [oracle.OsciState(w.float().numpy(), FMT_O[fmt], rnd, seed=5) for w in ws]
    for t in range(1, 4):
        deltas = [W.master_update(s, t, std=3e-3) for s in shapes]
        c = fq.Config(fmt, rnd, 5, t)
        if t < 3:
            g.step([d.to(DEV) for d in deltas], t)
        else:
            cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
            fq.fq_osci_update_reset(c, g.master, [d.to(DEV) for d in deltas], g.dq, g.dm,
                                    g.prev, g.next, 4.0, n_reset=cnt, xhat=g.xhat, mask=g.mask)
            g.prev, g.next = g.next, g.prev
        torch.cuda.synchronize()
        outs = [st.step(d.numpy(), offset=t) for st, d in zip(sts, deltas)]
    total = sum(st.reset(4.0) for st in sts)
    assert int(cnt.item()) == total and total > 0
    for i, st in enumerate(sts):
        _compare(f"fused.{i}", g, i, st, outs[i])


def test_osci_flip_example():
    with open(os.path.join(os.path.dirname(__file__), "golden", "osci_flip_e4.json")) as f:
        gd = json.load(f)
    w0 = torch.zeros((gd["rows"], gd["cols"]), dtype=torch.float32)
    for k, v in gd["w0"].items():
        w0[0, int(k)] = v
    g = GpuOsci([w0], fq.Config(fq.NVFP4))
    for t in range(1, gd["steps"] + 1):
        d = torch.zeros_like(w0)
        d[0, 1] = gd["delta_watched"] if t % 2 == 1 else -gd["delta_watched"]
        d[0, 2] = gd["delta_control"]
        g.step([d.to(DEV)], t)
    torch.cuda.synchronize()
    assert float(g.dq[0][0, 1]) == gd["expected_dist_q_watched"]
    assert abs(float(g.dm[0][0, 1]) - gd["expected_dist_m_watched_approx"]) < 1e-5
    assert float(g.dq[0][0, 2]) == gd["expected_dist_q_control"]
    cnt = g.reset(gd["threshold"])
    torch.cuda.synchronize()
    assert int(cnt.item()) == gd["expected_resets"]
    assert float(g.master[0][0, 1]) == gd["expected_master_watched_after_reset"]
    assert float(g.master[0][0, 16]) == 2688.0


def _full_moe_group(checked_idx, seed=1234):
    """The 32-expert MoE workload at full size (64 matrices, 1.06 G weights):
    the matrices in checked_idx come from the CPU generator (so the oracle can
    take them), the rest from a device generator."""
    spec = W.WORKLOADS["moe_qat"]
    E, up, down = spec["experts"], spec["up_shape"], spec["down_shape"]
    shapes = [up, down] * E
    gen = torch.Generator(device=DEV)
    gen.manual_seed(seed)
    ws, host = [], {}
    for i, s in enumerate(shapes):
        if i in checked_idx:
            w = W.normal(s, 0.02, seed=500 + i).to(torch.bfloat16)
            host[i] = w
            ws.append(w)
        else:
            ws.append((torch.randn(s, generator=gen, device=DEV) * 0.02).to(torch.bfloat16))
    return shapes, ws, host, gen


def _full_moe_deltas(shapes, checked_idx, t, gen):
    deltas, host = [], {}
    for i, s in enumerate(shapes):
        if i in checked_idx:
            d = W.master_update(s, t)
            host[i] = d
            deltas.append(d.to(DEV))
        else:
            deltas.append(torch.randn(s, generator=gen, device=DEV) * 1e-4)
    return deltas, host


@pytest.mark.slow
def test_osci_full_moe_two_steps():
    """Two update steps through the grouped launch on the full MoE group;
    eight matrices spread over the group (both shapes, first and last) are
    checked against the oracle bit for bit after each step, every matrix for
    invariants."""
    checked = (0, 9, 18, 27, 36, 45, 54, 63)
    shapes, ws, host_w, gen = _full_moe_group(checked)
    cfg = fq.Config(fq.NVFP4, fq.RNE)
    g = GpuOsci(ws, cfg)
    del ws
    sts = {i: oracle.OsciState(w.float().numpy(), oracle.NVFP4) for i, w in host_w.items()}
    for t in (1, 2):
        deltas, host = _full_moe_deltas(shapes, checked, t, gen)
        g.step(deltas, t)
        torch.cuda.synchronize()
        del deltas
        for i, st in sts.items():
            out = st.step(host[i].numpy(), offset=t)
            _compare(f"t{t}.{i}", g, i, st, out)
    for i in range(len(shapes)):
        assert torch.isfinite(g.dq[i]).all() and (g.dq[i] >= 0).all()
        assert (g.dm[i] > 0).float().mean() > 0.99


@pytest.mark.slow
def test_osci_full_moe_fused_reset():
    """The benchmark's dominant call, fq_osci_update_reset, on the full MoE
    group after one ordinary update.  The first, a middle and the last matrix
    are checked against the oracle's step + reset bit for bit.  Every matrix
    is checked against the unfused path (fq_osci_update then fq_osci_reset on
    a copy of the state), and the fused call's reset count equals the number
    of weights with dist_Q > 4 dist_M after the update, summed over all 64
    matrices; over the checked matrices that number equals the oracle's."""
    checked = (0, 31, 63)
    shapes, ws, host_w, gen = _full_moe_group(checked, seed=4321)
    cfg = fq.Config(fq.NVFP4, fq.RNE)
    g = GpuOsci(ws, cfg)
    del ws
    sts = {i: oracle.OsciState(w.float().numpy(), oracle.NVFP4) for i, w in host_w.items()}
    # step 1: ordinary update, large enough to move some weights across bins
    deltas, host = _full_moe_deltas(shapes, checked, 1, gen)
    deltas = [d * 30 for d in deltas]
    host = {i: d * 30 for i, d in host.items()}
    g.step(deltas, 1)
    for i, st in sts.items():
        st.step(host[i].numpy(), offset=1)
    del deltas
    # step 2: the window-end step, fused and unfused (on a copy)
    deltas, host = _full_moe_deltas(shapes, checked, 2, gen)
    u = GpuOsci.__new__(GpuOsci)
    u.cfg = cfg
    u.master = [m.clone() for m in g.master]
    u.dq = [d.clone() for d in g.dq]
    u.dm = [d.clone() for d in g.dm]
    u.prev = [fq.QTensor(q.codes.clone(), q.scales.clone(), q.tscale.clone()) for q in g.prev]
    u.next = [fq.alloc_qtensor(*m.shape, fq.NVFP4, DEV) for m in g.master]
    u.xhat = [torch.empty_like(x) for x in g.xhat]
    u.mask = [torch.empty_like(x) for x in g.mask]
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    fq.fq_osci_update_reset(fq.Config(fq.NVFP4, fq.RNE, 0, 2), g.master, deltas, g.dq, g.dm,
                            g.prev, g.next, 4.0, n_reset=cnt, xhat=g.xhat, mask=g.mask)
    g.prev, g.next = g.next, g.prev
    u.step(deltas, 2)
    torch.cuda.synchronize()
    del deltas
    per = [int((dq > 4.0 * dm).sum().item()) for dq, dm in zip(u.dq, u.dm)]
    ucnt = u.reset(4.0)
    torch.cuda.synchronize()
    assert int(cnt.item()) == int(ucnt.item()) == sum(per)
    assert sum(per) > 0
    for i in range(len(shapes)):
        for name, a, b in (("master", g.master[i], u.master[i]), ("dq", g.dq[i], u.dq[i]),
                           ("dm", g.dm[i], u.dm[i]), ("xhat", g.xhat[i], u.xhat[i]),
                           ("codes", g.prev[i].codes, u.prev[i].codes),
                           ("scales", g.prev[i].scales, u.prev[i].scales)):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (i, name)
    for i, st in sts.items():
        out = st.step(host[i].numpy(), offset=2)
        n = st.reset(4.0)
        assert n == per[i], (i, n, per[i])
        _compare(f"fused.{i}", g, i, st, out)
