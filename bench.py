#!/usr/bin/env python
"""Benchmark: block-scaled FP4 fake-quantization on GB300.

One step = one pass of the whole hot path over the synthetic workloads:
  nvfp4_small   NVFP4 fake-quant (RNE), FP32 [256, 1024]: codes, scales, s_g, FP32 xhat, mask
  mxfp4_weight  MXFP4 quantize + dequantize (RNE), BF16 [4096, 4096] weight with 0.1% x100
  nvfp4_act     NVFP4 row 1x16 + column 16x1 on the transpose in one call, BF16 [8192, 8192]
                activation with 8 outlier channels: both codes/scales, BF16 xhat, STE mask;
                then the STE backward of a BF16 gradient of the same shape
  grad_2level   double-block NVFP4 with stochastic rounding, BF16 [16384, 4096] Laplace gradient
  grad_rht_rowcol  the same kind of gradient as a backward-GEMM operand: 16-point random
                Hadamard transform + double-block SR, row 1x16 and column 16x1 in one call
  act_outliers  static outlier retention: BF16 [8192, 8192] activation with 64 outlier
                channels x50; the 10% of channels (819) with the largest calibration amax
                (two earlier batches, selected once before timing) go to FP8 E4M3, the rest
                to NVFP4: codes, scales, s_g, FP8 columns, BF16 xhat, STE mask
  qad_kl        QAD distillation loss: BF16 teacher and student logits [4096, 201088]
                (gpt-oss's vocabulary size), per-row KL(teacher || student) at T = 1, its
                mean, and the BF16 gradient with respect to the student logits
  osci_update   one ordinary QAT step over 32 MoE experts (64 FP32 master matrices
                [2880, 5760] and [5760, 2880], 1.06 G weights): update + NVFP4
                fake-quant + OsciReset statistics (what 99 of every 100 steps of an
                OsciReset window run)
  osci_update_reset  the window's last step over the same weights: the same update
                with the OsciReset reset fused into its second pass
The metric is algorithmic HBM bytes / device time (GB/s); elements/s are
reported per workload, with fractions of the measured copy bandwidth and of
the ~8 TB/s HBM3e spec.  Inputs live in HBM before the timed region; the step's
working set (about 26 GB) is far larger than L2, so every workload starts cold.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fake-quant HBM GB/s and % of GB300 HBM peak; Gelem/s per format"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0   # GB300 HBM3e peak as specified (~8 TB/s)

# Bytes per element each workload must move (reads + writes of its definition;
# the NVFP4 tensor amax is a second read of x).
BYTES_PER_ELEM = {
    "nvfp4_small": 4 + 4 + 0.5 + 1 / 16 + 4 + 1 / 8,
    "mxfp4_weight": 2 + 0.5 + 1 / 32 + 2 + 1 / 8,
    "nvfp4_act": 2 + 2 + 0.5 + 1 / 16 + 0.5 + 1 / 16 + 2 + 1 / 8,
    "ste_backward": 2 + 1 / 8 + 2,
    "grad_2level": 2 + 0.5 + 1 / 16 + 4 / 128,
    "grad_rht_rowcol": 2 + 2 * (0.5 + 1 / 16 + 4 / 128),
    "act_outliers": 2 + 2 + 0.5 + 1 / 16 + 819 / 8192 + 2 + 1 / 8,
    "qad_kl": 2 + 2 + 2,
    "osci_update": 20 + (4 + 0.5 + 1 / 16 + 8 + 0.5 + 1 / 16 + 2 + 1 / 8),
    "osci_update_reset": 20 + (4 + 0.5 + 1 / 16 + 8 + 8 + 0.5 + 1 / 16 + 2 + 1 / 8),
}
# Our kernels launched per step (memsets not counted).
LAUNCHES_PER_STEP = {"nvfp4_small": 2, "mxfp4_weight": 1, "nvfp4_act": 2, "ste_backward": 1,
                     "grad_2level": 1, "grad_rht_rowcol": 1, "act_outliers": 2,
                     "qad_kl": 2, "osci_update": 2, "osci_update_reset": 2}
# DRAM traffic per call of the OsciReset steps from an ncu capture, valid only
# for the kernel sources it was taken on (sha256 of the OsciReset sources).
# Captured on the 2-expert case (66.4 M weights; pass A + pass B read + write:
# 2227.5 MB for the ordinary step, 2824.0 MB for the window-end step) and
# scaled by the weights processed to the 32-expert call (traffic is linear in
# the number of weights).
_OSCI_SCALE = 1061683200 / 66355200
NCU_TRAFFIC = {"osci_update": {"bytes": int((1270458368 + 957048576) * _OSCI_SCALE),
                               "src_sha256": "c05d65f721f01046713f95db6ee83ed6f99794b57a90bc688d6f2dad1c5ac5d7"},
               "osci_update_reset": {"bytes": int((1267530752 + 1556487168) * _OSCI_SCALE),
                                     "src_sha256": "c05d65f721f01046713f95db6ee83ed6f99794b57a90bc688d6f2dad1c5ac5d7"}}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def src_sha(*names):
    """SHA-256 over the named csrc files, in order (a kernel's source and the
    headers it includes)."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "fp4_quantization_aware_fq_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# the sources the OsciReset kernels are compiled from
OSCI_SOURCES = ("k_osci.cu", "fq_device.cuh", "fq_internal.h")


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- workloads
class Suite:
    """The workloads' inputs and outputs, resident on one GPU.  `only` limits
    the suite to some workloads; `experts` scales the MoE workload down and
    `qad_rows` the logits (for profiling a smaller case of the same kernels);
    `mxfp4_rows` sets the rows of the MXFP4 weight (a larger case shows that
    kernel's DRAM traffic, which at 4096 rows still sits in L2 when it ends)."""

    ORDER = ("nvfp4_small", "mxfp4_weight", "nvfp4_act", "ste_backward", "grad_2level",
             "grad_rht_rowcol", "act_outliers", "qad_kl", "osci_update", "osci_update_reset")

    def __init__(self, dev, only=None, experts=None, qad_rows=None, mxfp4_rows=None):
        import torch
        from fp4_quantization_aware_fq_gb300 import fq
        from fp4_quantization_aware_fq_gb300 import workloads as W
        self.fq, self.torch, self.W, self.dev = fq, torch, W, dev
        self.names = [n for n in self.ORDER if not only or n in only]
        self.elems = {}
        self.step_no = 0
        want = set(self.names)
        if "nvfp4_small" in want:
            self.x1 = W.nvfp4_small(device=dev)
            self.cfg1 = fq.Config(fq.NVFP4)
            self.q1 = fq.alloc_qtensor(*self.x1.shape, fq.NVFP4, dev)
            self.xh1 = torch.empty(self.x1.shape, dtype=torch.float32, device=dev)
            self.m1 = self._mask(self.x1)
            self.ws1 = torch.empty(256, dtype=torch.uint8, device=dev)
            self.elems["nvfp4_small"] = self.x1.numel()
        if "mxfp4_weight" in want:
            self.x2 = W.mxfp4_weight(shape=(mxfp4_rows or 4096, 4096), device=dev)
            self.cfg2 = fq.Config(fq.MXFP4)
            self.q2 = fq.alloc_qtensor(*self.x2.shape, fq.MXFP4, dev)
            self.xh2 = torch.empty(self.x2.shape, dtype=torch.bfloat16, device=dev)
            self.m2 = self._mask(self.x2)
            self.elems["mxfp4_weight"] = self.x2.numel()
        if want & {"nvfp4_act", "ste_backward"}:
            self.x3 = W.nvfp4_act(device=dev)
            self.cfg3 = fq.Config(fq.NVFP4)
            r3, c3 = self.x3.shape
            self.rq3 = fq.alloc_qtensor(r3, c3, fq.NVFP4, dev)
            self.cq3 = fq.alloc_qtensor(c3, r3, fq.NVFP4, dev)
            self.xh3 = torch.empty(self.x3.shape, dtype=torch.bfloat16, device=dev)
            self.m3 = self._mask(self.x3)
            self.ws3 = torch.empty(256, dtype=torch.uint8, device=dev)
            self.elems["nvfp4_act"] = self.x3.numel()
            if "ste_backward" in want:
                self.nvfp4_act()          # the backward consumes this call's mask
                self.dy3 = W.normal(self.x3.shape, 1.0, seed=12, dtype=torch.bfloat16,
                                    device=dev)
                self.dx3 = torch.empty_like(self.dy3)
                self.elems["ste_backward"] = self.dy3.numel()
        if "grad_2level" in want:
            self.x4 = W.grad_2level(device=dev)
            self.cfg4 = fq.Config(fq.NVFP4_2LEVEL, fq.SR, 0x5EED, 0)
            self.q4 = fq.alloc_qtensor(*self.x4.shape, fq.NVFP4_2LEVEL, dev)
            self.elems["grad_2level"] = self.x4.numel()
        if "grad_rht_rowcol" in want:
            self.x6 = W.grad_2level(seed=6, device=dev)
            self.cfg6 = fq.Config(fq.NVFP4_2LEVEL, fq.SR, 0x5EED, 0, rht_seed=0xB00F)
            r6, c6 = self.x6.shape
            self.rq6 = fq.alloc_qtensor(r6, c6, fq.NVFP4_2LEVEL, dev)
            self.cq6 = fq.alloc_qtensor(c6, r6, fq.NVFP4_2LEVEL, dev)
            self.elems["grad_rht_rowcol"] = self.x6.numel()
        if "act_outliers" in want:
            c = W.WORKLOADS["channel_act"]
            self.x7 = W.channel_act(device=dev)
            r7, c7 = self.x7.shape
            amax = torch.zeros(c7, dtype=torch.float32, device=dev)
            for t in (1, 2):       # calibration window: two earlier batches
                fq.fq_channel_amax(W.channel_act(seed=c["seed"] + t, device=dev), amax)
            self.sel7 = fq.fq_select_channels(amax, c7 // 10)
            self.cfg7 = fq.Config(fq.NVFP4)
            self.q7 = fq.alloc_qtensor(r7, c7, fq.NVFP4, dev)
            self.fp87 = torch.empty((r7, c7 // 10), dtype=torch.uint8, device=dev)
            self.xh7 = torch.empty(self.x7.shape, dtype=torch.bfloat16, device=dev)
            self.m7 = self._mask(self.x7)
            self.ws7 = torch.empty(256, dtype=torch.uint8, device=dev)
            self.elems["act_outliers"] = self.x7.numel()
        if "qad_kl" in want:
            c = W.WORKLOADS["qad_logits"]
            r8 = qad_rows or c["shape"][0]
            self.zt8, self.zs8 = W.qad_logits((r8, c["shape"][1]), seed=c["seed"], device=dev)
            self.loss8 = torch.empty(r8, dtype=torch.float32, device=dev)
            self.mean8 = torch.empty(1, dtype=torch.float32, device=dev)
            self.dz8 = torch.empty_like(self.zs8)
            self.err8 = torch.zeros(1, dtype=torch.int32, device=dev)
            self.elems["qad_kl"] = self.zt8.numel()
        if want & {"osci_update", "osci_update_reset"}:
            m = W.WORKLOADS["moe_qat"]
            ws = W.moe_weights(experts or m["experts"], m["up_shape"], m["down_shape"],
                               seed=4, device=dev)
            self.cfg5 = fq.Config(fq.NVFP4)
            self.master = [w.float() for w in ws]
            del ws
            # one update per step call; each step reuses its update tensors: the
            # work (every weight read and written) does not depend on their values
            self.delta = [W.master_update(t.shape, 1, device=dev) for t in self.master]
            self.delta_u = ([W.master_update(t.shape, 2, device=dev) for t in self.master]
                            if "osci_update" in want else None)
            self.dq = [torch.zeros_like(t) for t in self.master]
            self.dm = [torch.zeros_like(t) for t in self.master]
            self.prev = [fq.fq_quantize(t, self.cfg5)[0] for t in self.master]
            self.next = [fq.alloc_qtensor(*t.shape, fq.NVFP4, dev) for t in self.master]
            self.xh5 = [torch.empty(t.shape, dtype=torch.bfloat16, device=dev)
                        for t in self.master]
            self.m5 = [self._mask(t) for t in self.master]
            self.ws5 = torch.empty(fq.fq_osci_workspace_size(len(self.master)),
                                   dtype=torch.uint8, device=dev)
            self.nreset = torch.zeros(1, dtype=torch.int64, device=dev)
            nw = sum(t.numel() for t in self.master)
            self.elems.update({"osci_update": nw, "osci_update_reset": nw})
        self.elems = {k: v for k, v in self.elems.items() if k in want}
        torch.cuda.synchronize()

    def _mask(self, x):
        return self.torch.empty(((x.numel() + 7) // 8 + 15) // 16 * 16, dtype=self.torch.uint8,
                                device=self.dev)

    def check(self):
        """Device-side error words of the calls that have them."""
        if "qad_kl" in self.names and int(self.err8.item()) != 0:
            raise RuntimeError("fq_qad_kl reported a shared-memory copy timeout")

    def step(self):
        for name in self.names:
            getattr(self, name)()
        self.step_no += 1

    # each call is one C-ABI entry point; all run on the current stream
    def nvfp4_small(self):
        self.fq.fq_fakequant_ste(self.x1, self.cfg1, xhat=self.xh1, mask=self.m1,
                                 row_out=self.q1, ws=self.ws1)

    def mxfp4_weight(self):
        self.fq.fq_fakequant_ste(self.x2, self.cfg2, xhat=self.xh2, mask=self.m2,
                                 row_out=self.q2)

    def nvfp4_act(self):
        self.fq.fq_fakequant_ste(self.x3, self.cfg3, xhat=self.xh3, mask=self.m3,
                                 row_out=self.rq3, col_out=self.cq3, ws=self.ws3)

    def ste_backward(self):
        self.fq.fq_ste_backward(self.dy3, self.m3, self.dx3)

    def grad_2level(self):
        self.cfg4.offset = self.step_no
        self.fq.fq_quantize(self.x4, self.cfg4, row_out=self.q4)

    def grad_rht_rowcol(self):
        # backward operand: Hadamard transform + double-block SR, both orientations
        self.cfg6.offset = self.step_no
        self.fq.fq_quantize(self.x6, self.cfg6, orient=self.fq.ROWCOL, row_out=self.rq6,
                            col_out=self.cq6)

    def act_outliers(self):
        self.fq.fq_quantize_outliers(self.x7, self.cfg7, self.sel7, out=self.q7, fp8=self.fp87,
                                     xhat=self.xh7, mask=self.m7, ws=self.ws7)

    def qad_kl(self):
        self.fq.fq_qad_kl(self.zt8, self.zs8, loss_rows=self.loss8, loss_mean=self.mean8,
                          dz=self.dz8, err=self.err8)

    def osci_update(self):
        # an ordinary QAT step of the OsciReset window
        self.fq.fq_osci_update(self.cfg5, self.master, self.delta_u, self.dq, self.dm,
                               self.prev, self.next, xhat=self.xh5, mask=self.m5, ws=self.ws5)
        self.prev, self.next = self.next, self.prev

    def osci_update_reset(self):
        # one QAT step that also ends the OsciReset window (reset fused in)
        self.fq.fq_osci_update_reset(self.cfg5, self.master, self.delta, self.dq, self.dm,
                                     self.prev, self.next, 4.0, n_reset=self.nreset,
                                     xhat=self.xh5, mask=self.m5, ws=self.ws5)
        self.prev, self.next = self.next, self.prev


def bytes_per_step(elems):
    return {k: BYTES_PER_ELEM[k] * elems[k] for k in elems}


# --------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, dist, device) -> float:
    """The largest value over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_step: float, steps: int, ms: float) -> float:
    """Whole-job GB/s: every rank moves bytes_per_step per step (weak scaling)."""
    return world * bytes_per_step * steps / (ms / 1e3) / 1e9


# --------------------------------------------------------------------------- device timing
def run_ours(args, rank, world, dist):
    import torch
    dev = torch.device("cuda", torch.cuda.current_device())
    suite = Suite(dev, only=args.only, experts=args.experts, qad_rows=args.qad_rows,
                  mxfp4_rows=args.mxfp4_rows)
    stream = torch.cuda.current_stream()
    bps = bytes_per_step(suite.elems)
    total_bytes = sum(bps.values())

    for _ in range(args.warmup):
        suite.step()
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        try:
            graph = capture_step(suite)
        except Exception as e:  # capture is an optimisation of the launches only
            log(f"CUDA graph capture failed ({e!r}); timing eager launches")
            graph = None
            torch.cuda.synchronize()
    if graph is not None:
        for _ in range(args.warmup):
            graph[0].replay()
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = {n: [] for n in suite.names}
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph[0].replay()
        else:
            for name in suite.names:
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                getattr(suite, name)()
                b.record(stream)
                ev[name].append((a, b))
            suite.step_no += 1
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    suite.check()
    ms = t0.elapsed_time(t1)
    if graph is not None:
        # per-workload times: the events the graph records between workloads,
        # read after each of a second series of replays
        g, evs = graph
        acc = [0.0] * len(suite.names)
        for _ in range(args.steps):
            g.replay()
            torch.cuda.synchronize()
            for i in range(len(suite.names)):
                acc[i] += evs[i].elapsed_time(evs[i + 1])
        per_ms = {n: acc[i] / args.steps for i, n in enumerate(suite.names)}
    else:
        per_ms = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / args.steps for n in suite.names}
    ms = max_over_ranks(ms, dist, dev)
    suite.launch_mode = "cuda_graph" if graph is not None else "eager"

    # end-to-end: pinned host inputs -> device, the same calls, results -> host
    e2e = run_e2e(args, suite, total_bytes) if not args.no_e2e else None
    if e2e is not None:
        e2e["ms_total"] = max_over_ranks(e2e["ms_total"], dist, dev)
    return suite, bps, total_bytes, ms, per_ms, clk, e2e


def capture_step(suite):
    """One step of the suite (every workload once) captured as a CUDA graph,
    with timing events that the graph itself records between the workloads.
    The step's two OsciReset calls swap the ping-pong quantized buffers twice,
    so every replay starts from the buffers the capture started from; the
    stochastic-rounding offsets are those of the captured step."""
    import torch
    names = suite.names
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        s = torch.cuda.current_stream()
        evs[0].record(s)
        for i, name in enumerate(names):
            getattr(suite, name)()
            evs[i + 1].record(s)
    suite.step_no += 1
    return g, evs


def e2e_buffers(suite):
    """Per workload (in step order): the device tensors that each step takes
    from the host (its inputs) and the results it hands back (packed codes and
    scales, losses, the reset count)."""
    io = {}
    if "nvfp4_small" in suite.names:
        io["nvfp4_small"] = ([suite.x1], [suite.q1.codes, suite.q1.scales, suite.q1.tscale])
    if "mxfp4_weight" in suite.names:
        io["mxfp4_weight"] = ([suite.x2], [suite.q2.codes, suite.q2.scales])
    if "nvfp4_act" in suite.names:
        io["nvfp4_act"] = ([suite.x3], [suite.rq3.codes, suite.rq3.scales, suite.cq3.codes,
                                        suite.cq3.scales])
    if "ste_backward" in suite.names:
        io["ste_backward"] = ([suite.dy3], [suite.dx3])
    if "grad_2level" in suite.names:
        io["grad_2level"] = ([suite.x4], [suite.q4.codes, suite.q4.scales, suite.q4.tscale])
    if "grad_rht_rowcol" in suite.names:
        io["grad_rht_rowcol"] = ([suite.x6], [suite.rq6.codes, suite.rq6.scales, suite.rq6.tscale,
                                              suite.cq6.codes, suite.cq6.scales, suite.cq6.tscale])
    if "act_outliers" in suite.names:
        io["act_outliers"] = ([suite.x7], [suite.q7.codes, suite.q7.scales, suite.q7.tscale,
                                           suite.fp87])
    if "qad_kl" in suite.names:
        io["qad_kl"] = ([suite.zt8, suite.zs8], [suite.loss8, suite.mean8])
    if "osci_update" in suite.names:
        io["osci_update"] = (list(suite.delta_u), [suite.dq[0][:1]])
    if "osci_update_reset" in suite.names:
        io["osci_update_reset"] = (list(suite.delta), [suite.nreset])
    return io


GEMM_SHAPE = (8192, 8192, 8192)   # M (tokens), N (output features), K (input features)
FP4_PER_BF16 = 6.0                 # nominal dense FP4 / BF16 tensor throughput (13.5 / 2.25 PF)
FALLBACK_BF16_TFLOPS = 1900.0


def bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("bf16_tflops", "bf16_TFLOPs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def run_gemm(steps=20, warmup=3, fmt_name="nvfp4"):
    """The forward GEMM of a QAT linear layer on NVFP4 (or MXFP4) operands: a
    BF16 activation [M, K] ~ N(0, 1) and a weight [N, K] ~ N(0, 0.02), both
    quantized with fq_quantize, then fq_gemm to a BF16 C, timed with CUDA
    events on the launching stream (the operands, about 70 MB of codes and
    scales, stay in L2 between launches: this measures the tensor-core path)."""
    import torch
    from fp4_quantization_aware_fq_gb300 import fq
    from fp4_quantization_aware_fq_gb300 import workloads as W
    dev = torch.device("cuda", torch.cuda.current_device())
    m, n, k = GEMM_SHAPE
    cfg = fq.Config(fq.MXFP4 if fmt_name == "mxfp4" else fq.NVFP4)
    a = W.normal((m, k), 1.0, seed=20, dtype=torch.bfloat16, device=dev)
    b = W.normal((n, k), 0.02, seed=21, dtype=torch.bfloat16, device=dev)
    qa, _ = fq.fq_quantize(a, cfg)
    qb, _ = fq.fq_quantize(b, cfg)
    del a, b
    c = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(fq.fq_gemm_workspace_size(m, n, k), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fq.fq_gemm(qa, qb, m, n, k, cfg, c=c, ws=ws, err=err)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        fq.fq_gemm(qa, qb, m, n, k, cfg, c=c, ws=ws, err=err)
    t1.record(stream)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("fq_gemm reported a pipeline wait timeout")
    ms = t0.elapsed_time(t1) / steps
    tflops = 2.0 * m * n * k / (ms * 1e-3) / 1e12
    peak, kind = bf16_peak()
    peak *= FP4_PER_BF16
    return {"shape_mnk": list(GEMM_SHAPE), "dtype": f"{fmt_name} x {fmt_name} -> bf16",
            "ms": round(ms, 4),
            "tflops": round(tflops, 1), "bound": "tensor", "peak_tflops": round(peak, 1),
            "peak_kind": kind + " bf16 x nominal FP4/BF16 ratio 6", "frac": round(tflops / peak, 3),
            "launches_per_call": 3, "note": "not part of the suite step; operands L2-resident"}


def run_small_at_scale(steps=20, warmup=3):
    """The nvfp4_small call (FP32 NVFP4 fake-quant with codes, scales, FP32 xhat
    and mask) on a [65536, 1024] tensor of the same recipe: at 256 x 1024 the
    workload is launch-bound, so the kernels' bandwidth shows only at size.
    Not part of the step; the input (256 MB) exceeds L2."""
    import torch
    from fp4_quantization_aware_fq_gb300 import fq
    from fp4_quantization_aware_fq_gb300 import workloads as W
    dev = torch.device("cuda", torch.cuda.current_device())
    x = W.normal((65536, 1024), 1.0, seed=0, device=dev)
    cfg = fq.Config(fq.NVFP4)
    q = fq.alloc_qtensor(*x.shape, fq.NVFP4, dev)
    xh = torch.empty_like(x)
    m = torch.empty(((x.numel() + 7) // 8 + 15) // 16 * 16, dtype=torch.uint8, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    call = lambda: fq.fq_fakequant_ste(x, cfg, xhat=xh, mask=m, row_out=q, ws=ws)  # noqa: E731
    for _ in range(warmup):
        call()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        call()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    gbs = BYTES_PER_ELEM["nvfp4_small"] * x.numel() / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"shape": [65536, 1024], "ms": round(ms, 4), "gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 3), "peak_kind": kind,
            "note": "nvfp4_small's two launches on a 64x larger tensor; not part of the step"}


def run_osci_window(suite, windows=2):
    """A whole OsciReset observation window on the MoE group: 99 ordinary QAT
    steps (fq_osci_update) and the window-end step with the reset fused in
    (fq_osci_update_reset), eager launches on the current stream, timed with
    CUDA events; each window's 100 steps move about 3.7 TB, far beyond L2.
    Not part of the suite step."""
    import torch
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(windows):
        for _ in range(99):
            suite.osci_update()
        suite.osci_update_reset()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / windows
    nbytes = (99 * BYTES_PER_ELEM["osci_update"] * suite.elems["osci_update"]
              + BYTES_PER_ELEM["osci_update_reset"] * suite.elems["osci_update_reset"])
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"steps_per_window": 100, "weights": suite.elems["osci_update"],
            "ms_per_window": round(ms, 2), "ms_per_step": round(ms / 100, 4),
            "bytes_per_window": int(nbytes), "gbs": round(gbs, 1),
            "frac_hbm": round(gbs / peak, 3), "frac_spec": round(gbs / SPEC_HBM_GBS, 3),
            "peak_kind": kind, "windows_timed": windows,
            "note": "99 ordinary steps + the window-end step with the reset; not part of the "
                    "suite step"}


def run_osci_reset(suite, reps=5):
    """The standalone window-end reset (fq_osci_reset) over the MoE group: each
    rep runs one ordinary QAT step (untimed, so the accumulators hold a step's
    statistics), then the reset alone between CUDA events.  20.5625
    algorithmic bytes per weight, the reset pass counted as if every weight
    were reset: dist_Q and dist_M read and written back as zero (16), the
    current codes and scales read (0.5625) and the master weight written (4).
    Not part of the suite step: the step fuses the reset into its last update
    (fq_osci_update_reset), at 8 more bytes per weight than an update."""
    import torch
    fq = suite.fq
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(reps):
        suite.osci_update()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        # after osci_update's swap, prev holds the step's codes: the current bin
        fq.fq_osci_reset(suite.cfg5, suite.master, suite.dq, suite.dm, suite.prev, 4.0,
                         n_reset=suite.nreset)
        t1.record(stream)
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1))
    times.sort()
    ms = times[len(times) // 2]
    nbytes = (16 + 0.5 + 1 / 16 + 4) * suite.elems["osci_update"]
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"weights": suite.elems["osci_update"], "ms_median": round(ms, 4),
            "ms_min": round(times[0], 4), "gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 3),
            "frac_spec": round(gbs / SPEC_HBM_GBS, 3), "peak_kind": kind, "reps": reps,
            "launches_per_call": 1,
            "note": "fq_osci_reset alone after an ordinary step; not part of the suite step"}


def run_osci_mxfp4(suite, steps=10, warmup=2):
    """The ordinary OsciReset step of the same 32-expert group with MXFP4 weight
    quantization (the format the gpt-oss QAT page trains back to): block-local
    E8M0 scales need no tensor amax, so the step is one pass over the weights.
    31.1875 algorithmic bytes per weight: master, delta, dist_M and dist_Q read
    (16), the previous codes and scales read (0.53125), master, dist_M and
    dist_Q written (12), the new codes and scales, BF16 xhat and mask written
    (2.65625).  Runs after the suite's own measurements, on its master weights
    and accumulators.  Not part of the suite step."""
    import torch
    fq = suite.fq
    cfg = fq.Config(fq.MXFP4)
    dev = suite.master[0].device
    prev = [fq.alloc_qtensor(*m.shape, fq.MXFP4, dev) for m in suite.master]
    nxt = [fq.alloc_qtensor(*m.shape, fq.MXFP4, dev) for m in suite.master]
    for m, q in zip(suite.master, prev):
        fq.fq_quantize(m, cfg, row_out=q)

    def step():
        nonlocal prev, nxt
        fq.fq_osci_update(cfg, suite.master, suite.delta_u, suite.dq, suite.dm, prev, nxt,
                          xhat=suite.xh5, mask=suite.m5, ws=suite.ws5)
        prev, nxt = nxt, prev

    for _ in range(warmup):
        step()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    nbytes = (16 + 0.5 + 1 / 32 + 12 + 0.5 + 1 / 32 + 2 + 1 / 8) * suite.elems["osci_update"]
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"weights": suite.elems["osci_update"], "ms_per_step": round(ms, 4),
            "gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 3),
            "frac_spec": round(gbs / SPEC_HBM_GBS, 3), "peak_kind": kind, "steps": steps,
            "launches_per_step": 1,
            "note": "ordinary OsciReset step with MXFP4 weights, one pass; not part of the suite "
                    "step"}


def run_quant_dequant(reps=20, warmup=3):
    """The MXFP4 weight workload as two separate calls, fq_quantize (codes and
    E8M0 scales) then fq_dequantize (BF16), on the same [4096, 4096] BF16
    weight.  The input fits in L2, so each rep first writes a 512 MB buffer
    (outside the timed events) to flush it.  Not part of the suite step."""
    import torch
    from fp4_quantization_aware_fq_gb300 import fq
    from fp4_quantization_aware_fq_gb300 import workloads as W
    dev = torch.device("cuda", torch.cuda.current_device())
    x = W.mxfp4_weight(device=dev)
    rows, cols = x.shape
    cfg = fq.Config(fq.MXFP4)
    q = fq.alloc_qtensor(rows, cols, fq.MXFP4, dev)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        fq.fq_quantize(x, cfg, row_out=q)
        fq.fq_dequantize(q, rows, cols, cfg, y=y)

    for _ in range(warmup):
        call()
    times = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        call()
        t1.record(stream)
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1))
    times.sort()
    ms = times[len(times) // 2]
    nbytes = (2 + 0.5 + 1 / 32 + 0.5 + 1 / 32 + 2) * x.numel()
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, kind = measured_peaks()
    return {"shape": [rows, cols], "ms_median": round(ms, 4), "ms_min": round(times[0], 4),
            "gbs": round(gbs, 1), "frac_hbm": round(gbs / peak, 3), "peak_kind": kind,
            "launches_per_call": 2, "l2": "flushed before each rep (512 MB write)",
            "note": "mxfp4_weight as quantize then dequantize; not part of the step"}


def quant_diagnostics(suite):
    """Quantization error of the workloads' last outputs, for monitoring (not
    timed): the relative squared error sum (x - xhat)^2 / sum x^2 and the
    signal-to-quantization-noise ratio in dB, the share of elements the STE
    mask marks as clipped, and for the stochastically rounded gradient the
    mean error relative to the mean magnitude (unbiasedness).  xhat is the
    fake-quantized output of the call, or fq_dequantize of its codes."""
    import math
    import torch
    fq = suite.fq
    pop = torch.tensor([bin(i).count("1") for i in range(256)], dtype=torch.int64,
                       device=suite.dev)

    def stats(x, xhat, mask=None):
        xf, hf = x.double(), xhat.double()
        err = (hf - xf).pow(2).sum().item()
        sig = xf.pow(2).sum().item()
        rel = err / sig if sig > 0 else 0.0
        d = {"rel_sq_error": float(f"{rel:.4e}"),
             "sqnr_db": round(-10.0 * math.log10(rel), 2) if rel > 0 else None}
        if mask is not None:
            n = x.numel()
            kept = int(pop[mask[:n // 8].long()].sum().item())
            d["clipped_share"] = float(f"{1.0 - kept / n:.4e}")
        return d

    out = {}
    if "nvfp4_small" in suite.names:
        out["nvfp4_small"] = stats(suite.x1, suite.xh1, suite.m1)
    if "mxfp4_weight" in suite.names:
        out["mxfp4_weight"] = stats(suite.x2, suite.xh2, suite.m2)
    if "nvfp4_act" in suite.names:
        out["nvfp4_act"] = stats(suite.x3, suite.xh3, suite.m3)
    if "act_outliers" in suite.names:
        out["act_outliers"] = stats(suite.x7, suite.xh7, suite.m7)
    if "grad_2level" in suite.names:
        r, c = suite.x4.shape
        y = fq.fq_dequantize(suite.q4, r, c, suite.cfg4, y_dtype=torch.float32)
        d = stats(suite.x4, y)
        x = suite.x4.double()
        d["rel_bias"] = float(f"{((y.double() - x).mean() / x.abs().mean()).item():.3e}")
        out["grad_2level"] = d
    torch.cuda.synchronize()
    return out


def run_e2e(args, suite, total_bytes):
    """The suite end to end: every step copies each workload's inputs from
    pinned host memory to the device (copy stream), runs the workload's calls
    (the current stream) and reads its results back to pinned host memory
    (read-back stream).  Events order each workload's copy-in before its calls
    and its read-back after them, and keep the next step's copy-in (or calls)
    from overwriting a buffer that this step still reads: the copies of later
    workloads overlap the calls of earlier ones, as in a training loop that
    streams its batches in."""
    import torch
    stream = torch.cuda.current_stream()
    cs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    io = e2e_buffers(suite)
    names = [n for n in suite.names if n in io]
    h_in = {n: [(d, d.cpu().pin_memory()) for d in io[n][0]] for n in names}
    h_out = {n: [(o, torch.empty(o.shape, dtype=o.dtype).pin_memory()) for o in io[n][1]]
             for n in names}
    h2d = sum(h.numel() * h.element_size() for n in names for _, h in h_in[n])
    d2h = sum(h.numel() * h.element_size() for n in names for _, h in h_out[n])
    ev_in = {n: torch.cuda.Event() for n in names}    # inputs are on the device
    ev_used = {n: torch.cuda.Event() for n in names}  # the calls are done (inputs read, outputs written)
    ev_out = {n: torch.cuda.Event() for n in names}   # outputs are back on the host
    recorded = set()

    def step():
        for n in names:
            if n in recorded:
                cs.wait_event(ev_used[n])
            with torch.cuda.stream(cs):
                for d, h in h_in[n]:
                    d.copy_(h, non_blocking=True)
            ev_in[n].record(cs)
        for n in names:
            stream.wait_event(ev_in[n])
            if n in recorded:
                stream.wait_event(ev_out[n])
            getattr(suite, n)()
            ev_used[n].record(stream)
            ds.wait_event(ev_used[n])
            with torch.cuda.stream(ds):
                for o, h in h_out[n]:
                    h.copy_(o, non_blocking=True)
            ev_out[n].record(ds)
            recorded.add(n)
        suite.step_no += 1

    for _ in range(max(1, min(args.warmup, 2))):
        step()
    torch.cuda.synchronize()
    k = max(1, min(args.steps, 10))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    cs.wait_event(a)
    ds.wait_event(a)
    for _ in range(k):
        step()
    stream.wait_stream(cs)
    stream.wait_stream(ds)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"ms_total": ms, "steps": k, "h2d": h2d, "d2h": d2h, "bytes": total_bytes}


# --------------------------------------------------------------------------- oracle timing
_ORACLE_INPUTS = {}


def _oracle_inputs(div):
    """The oracle's sample inputs, with every sample's rows divided by div
    (built once per div: the generators are not what is timed)."""
    if div in _ORACLE_INPUTS:
        return _ORACLE_INPUTS[div]
    import torch
    import oracle
    from fp4_quantization_aware_fq_gb300 import workloads as W
    oracle.build()
    f32 = lambda t: oracle.bf16_bits_to_f32(W.bf16_bits(t)).reshape(t.shape)  # noqa: E731
    d = {}
    d["x1"] = W.nvfp4_small(shape=(256 // div, 1024)).numpy()
    d["x2"] = f32(W.mxfp4_weight(shape=(4096 // div, 4096), seed=1))
    d["x3"] = f32(W.nvfp4_act(shape=(4096 // div, 8192), seed=2))
    d["dy"] = W.bf16_bits(W.normal(d["x3"].shape, 1.0, seed=12, dtype=torch.bfloat16))
    d["x4"] = f32(W.grad_2level(shape=(8192 // div, 4096), seed=3))
    d["x6"] = f32(W.grad_2level(shape=(2048 // div, 4096), seed=6))
    d["x7"] = f32(W.channel_act(shape=(2048 // div, 8192)))
    d["sel7"] = oracle.select_channels(
        oracle.channel_amax(f32(W.channel_act(shape=(2048 // div, 8192), seed=501))), 819)
    zt8, zs8 = W.qad_logits((max(16 // div, 1), 201088), seed=6)
    d["zt8"], d["zs8"] = f32(zt8), f32(zs8)
    d["w5"] = f32(W.normal((5760 // div, 5760), 0.02, seed=4).to(torch.bfloat16))
    d["d5"] = W.master_update((5760 // div, 5760), 1).numpy()
    d["d5b"] = W.master_update((5760 // div, 5760), 2).numpy()
    _ORACLE_INPUTS[div] = d
    return d


def _oracle_run(d):
    """One pass of the oracle over every workload's sample: {workload:
    (elements, seconds)}.  The OsciReset state is built before the clock
    starts."""
    import oracle
    res = {}

    def timed(fn):
        t = time.perf_counter()
        fn()
        return time.perf_counter() - t

    st = oracle.OsciState(d["w5"], oracle.NVFP4)
    res["nvfp4_small"] = (d["x1"].size, timed(lambda: oracle.quantize(
        d["x1"], oracle.NVFP4, want_xhat=True, want_mask=True)))
    res["mxfp4_weight"] = (d["x2"].size, timed(lambda: oracle.quantize(
        d["x2"], oracle.MXFP4, want_xhat=True, want_mask=True)))

    def c3():
        q = oracle.quantize(d["x3"], oracle.NVFP4, orient=oracle.ROWCOL, want_xhat=True,
                            want_mask=True)
        oracle.f32_to_bf16_bits(q["row"]["xhat"])
        return q
    t = time.perf_counter()
    q3 = c3()
    res["nvfp4_act"] = (d["x3"].size, time.perf_counter() - t)
    res["ste_backward"] = (d["dy"].size, timed(lambda: oracle.ste_backward(
        d["dy"], q3["row"]["mask"])))
    res["grad_2level"] = (d["x4"].size, timed(lambda: oracle.quantize(
        d["x4"], oracle.NVFP4_2LEVEL, oracle.SR, 0x5EED)))
    res["grad_rht_rowcol"] = (d["x6"].size, timed(lambda: oracle.quantize(
        d["x6"], oracle.NVFP4_2LEVEL, oracle.SR, 0x5EED, orient=oracle.ROWCOL, rht_seed=0xB00F)))

    def c7():
        q = oracle.quantize_outliers(d["x7"], d["sel7"]["idx"], d["sel7"]["fp8_scale"],
                                     oracle.NVFP4)
        oracle.f32_to_bf16_bits(q["xhat"])
    res["act_outliers"] = (d["x7"].size, timed(c7))
    res["qad_kl"] = (d["zt8"].size, timed(lambda: oracle.qad_kl(d["zt8"], d["zs8"])))

    def upd(delta, offset):
        out = st.step(delta, offset=offset)
        oracle.f32_to_bf16_bits(out["xhat"])
    res["osci_update"] = (d["w5"].size, timed(lambda: upd(d["d5"], 1)))
    res["osci_update_reset"] = (d["w5"].size, timed(lambda: upd(d["d5b"], 2))
                                + timed(lambda: st.reset(4.0)))
    return res


def host_cores():
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(div=1, threads=1):
    """Time the oracle on a bounded sample of every workload (row counts of the
    samples divided by div).  With threads > 1, that many threads each run the
    whole sample at once (the oracle's C code runs without the interpreter
    lock), so the per-element times are those of all cores working together:
    each thread's time divided by the number of threads.  Returns ({workload:
    (elements, seconds per element-equivalent run)}, description, wall
    seconds)."""
    import threading
    d = _oracle_inputs(div)
    if threads <= 1:
        t0 = time.perf_counter()
        res = _oracle_run(d)
        wall = time.perf_counter() - t0
    else:
        outs = [None] * threads
        go = threading.Barrier(threads + 1)

        def work(i):
            go.wait()
            outs[i] = _oracle_run(d)
        ths = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
        for th in ths:
            th.start()
        go.wait()
        t0 = time.perf_counter()
        for th in ths:
            th.join()
        wall = time.perf_counter() - t0
        res = {k: (outs[0][k][0], sum(o[k][1] for o in outs) / threads / threads)
               for k in outs[0]}
    r = lambda n: n // div  # noqa: E731
    desc = (f"oracle (scalar C) on {threads} host thread(s), each running: nvfp4_small "
            f"{r(256)} rows; mxfp4_weight {r(4096)} rows; nvfp4_act {r(4096)} rows row+col; "
            f"ste_backward {r(4096)}x8192; grad_2level {r(8192)} rows SR; grad_rht_rowcol "
            f"{r(2048)} rows; act_outliers {r(2048)} rows; qad_kl {max(16 // div, 1)} rows; "
            f"osci update, then update+reset, on a [{r(5760)}, 5760] matrix; per-element rates "
            f"scaled to the full step's elements")
    return res, desc, wall


def oracle_gbs(sample, elems_full):
    """Suite GB/s of the oracle: full-step bytes / (sum of full-size times at
    the sampled per-element rates)."""
    secs = 0.0
    for k, (n, t) in sample.items():
        if k in elems_full:
            secs += elems_full[k] * (t / n)
    total = sum(BYTES_PER_ELEM[k] * elems_full[k] for k in elems_full)
    return total / secs / 1e9, secs


FULL_ELEMS = {"nvfp4_small": 256 * 1024, "mxfp4_weight": 4096 * 4096,
              "nvfp4_act": 8192 * 8192, "ste_backward": 8192 * 8192,
              "grad_2level": 16384 * 4096, "grad_rht_rowcol": 16384 * 4096,
              "act_outliers": 8192 * 8192, "qad_kl": 4096 * 201088,
              "osci_update": 32 * 2 * 2880 * 5760,
              "osci_update_reset": 32 * 2 * 2880 * 5760}


def config_block(names=None, experts=None, qad_rows=None, mxfp4_rows=None):
    if names is not None and (list(names) != list(Suite.ORDER) or experts or qad_rows
                              or mxfp4_rows):
        return {"workload": "subset: " + ",".join(names) + (f"; moe experts={experts}"
                                                           if experts else "")
                + (f"; qad rows={qad_rows}" if qad_rows else "")
                + (f"; mxfp4 rows={mxfp4_rows}" if mxfp4_rows else ""),
                "l2": "no flush between steps", "bytes": "algorithmic"}
    return {"workload": "fake-quant suite over the synthetic workloads (one pass each per "
                        "step): nvfp4_small fp32 256x1024 NVFP4 RNE; mxfp4_weight bf16 "
                        "4096x4096 MXFP4 RNE quant+dequant; nvfp4_act bf16 8192x8192 NVFP4 "
                        "row 1x16 + col 16x1 + xhat + STE mask, then STE backward; grad_2level "
                        "bf16 16384x4096 double-block NVFP4 SR; grad_rht_rowcol the same "
                        "gradient with the 16-point Hadamard transform, both orientations; "
                        "act_outliers bf16 8192x8192 activation, 819 channels kept in FP8 "
                        "E4M3 by calibration amax, the rest NVFP4 RNE with xhat + STE mask; "
                        "qad_kl bf16 teacher/student logits 4096x201088: per-row KL at T=1, "
                        "mean, bf16 student gradient; "
                        "osci_update: 32 MoE experts x (2880x5760 + 5760x2880) FP32 master, one "
                        "ordinary QAT step with OsciReset statistics; osci_update_reset: the "
                        "window's last step on the same weights, the reset fused in",
            "elements_per_step": sum(FULL_ELEMS.values()),
            "l2": "no flush: the step's working set (~30 GB) exceeds L2, inputs are cold",
            "bytes": "algorithmic (definition reads + writes; NVFP4 amax is a second read)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of a CUDA graph of the step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", nargs="*", choices=Suite.ORDER, default=None,
                    help="run only these workloads (profiling a single kernel)")
    ap.add_argument("--experts", type=int, default=None,
                    help="MoE experts in moe_qat (default: the full 32)")
    ap.add_argument("--qad-rows", type=int, default=None,
                    help="rows of the qad_kl logits (default: the full 4096)")
    ap.add_argument("--mxfp4-rows", type=int, default=None,
                    help="rows of the mxfp4_weight tensor (default: the full 4096)")
    ap.add_argument("--gemm-only", choices=["nvfp4", "mxfp4"], default=None,
                    help="time only the tensor-core GEMM of this format (one JSON object)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return main_reference(args, rank, world)

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if args.gemm_only:
        print(json.dumps(run_gemm(args.steps, args.warmup, args.gemm_only)), flush=True)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from fp4_quantization_aware_fq_gb300 import build as fqbuild
    fqbuild.build()

    suite, bps, total_bytes, ms, per_ms, clk, e2e = run_ours(args, rank, world, dist)
    if rank == 0:
        peak, peak_kind = measured_peaks()
        ms_step = ms / args.steps
        value = job_throughput(world, total_bytes, args.steps, ms)
        per = {}
        for n in suite.names:
            t = per_ms[n] / 1e3
            per[n] = {"gbs": round(bps[n] / t / 1e9, 1),
                      "gelem_s": round(suite.elems[n] / t / 1e9, 3),
                      "ms": round(per_ms[n], 4),
                      "frac_hbm": round(bps[n] / t / 1e9 / peak, 3),
                      "frac_spec": round(bps[n] / t / 1e9 / SPEC_HBM_GBS, 3)}
        dom = max(suite.names, key=lambda n: per_ms[n])
        achieved = bps[dom] / (per_ms[dom] / 1e3) / 1e9
        tr = NCU_TRAFFIC.get(dom, {})
        traffic = tr.get("bytes") if tr.get("src_sha256") == src_sha(*OSCI_SOURCES) else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded torch generators, shapes/distributions of the "
                    "workloads)",
            "config": {**config_block(suite.names, args.experts, args.qad_rows, args.mxfp4_rows),
                       "launch": suite.launch_mode},
            "per_workload": per,
            "roofline": {"bound": "hbm", "kernel": dom + (" (osci_pass_a + osci_pass_b<reset>)"
                                                           if dom == "osci_update_reset" else ""),
                         "achieved": round(achieved, 1), "peak": peak,
                         "peak_kind": f"{peak_kind} copy bandwidth",
                         "unit": "GB/s", "frac": round(achieved / peak, 3),
                         "frac_spec": round(achieved / SPEC_HBM_GBS, 3),
                         "spec_peak": SPEC_HBM_GBS,
                         "traffic": traffic,
                         "algorithmic_bytes_per_launch": int(bps[dom])},
            "gpu_launches": sum(LAUNCHES_PER_STEP[n] for n in suite.names) * args.steps,
            "clocks": clk,
        }
        if e2e is not None:
            line["e2e"] = {"value": round(job_throughput(world, e2e["bytes"], e2e["steps"],
                                                         e2e["ms_total"]), 1),
                           "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                           "d2h_bytes_per_step": e2e["d2h"], "steps": e2e["steps"],
                           "ms_per_step": round(e2e["ms_total"] / e2e["steps"], 3)}
        reduced = bool(args.only or args.experts or args.qad_rows or args.mxfp4_rows)
        if world == 1 and not reduced:
            line["nvfp4_small_at_scale"] = run_small_at_scale()
            line["gemm_nvfp4"] = run_gemm(fmt_name="nvfp4")
            line["gemm_mxfp4"] = run_gemm(fmt_name="mxfp4")
            line["osci_window"] = run_osci_window(suite)
            line["osci_reset"] = run_osci_reset(suite)
            line["osci_update_mxfp4"] = run_osci_mxfp4(suite)
            line["mxfp4_quant_dequant"] = run_quant_dequant()
            line["quant_diagnostics"] = quant_diagnostics(suite)
        if not args.no_cpu_baseline and world == 1 and not reduced:
            # all host cores (one sample per thread, at once), then one core
            cores = host_cores()
            sample, desc, wall = oracle_sample(threads=cores)
            gbs, secs = oracle_gbs(sample, suite.elems)
            sample1, desc1, wall1 = oracle_sample(threads=1)
            gbs1, secs1 = oracle_gbs(sample1, suite.elems)
            line["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": cores,
                                    "kind": "oracle", "sample": desc,
                                    "sample_wall_seconds": round(wall, 2),
                                    "est_seconds_per_step": round(secs, 2),
                                    "single_thread": {"value": round(gbs1, 4), "cores": 1,
                                                      "sample_wall_seconds": round(wall1, 2),
                                                      "est_seconds_per_step": round(secs1, 1)}}
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def main_reference(args, rank, world):
    """The oracle as it stands, on all host cores: each step has every core run
    a bounded sample of every workload at once; value = the suite's bytes at
    the sampled per-element rates.  ms_per_step is the measured wall time of
    one such sampled step; the time the oracle would take for the full-size
    step is reported beside it as an estimate."""
    if rank != 0:
        return
    cores = host_cores()
    # each thread's sample is an eighth the size of the cpu_baseline's (about
    # a second of oracle work), so that the whole run stays within minutes
    for _ in range(args.warmup):
        oracle_sample(div=8, threads=cores)
    vals, walls, ests = [], [], []
    desc = ""
    for _ in range(args.steps):
        sample, desc, wall = oracle_sample(div=8, threads=cores)
        v, s = oracle_gbs(sample, FULL_ELEMS)
        vals.append(v)
        walls.append(wall)
        ests.append(s)
    value = statistics.median(vals)
    ms = statistics.median(walls) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 1),
            "ms_per_step_basis": "measured wall time of one sampled step (every core runs an "
                                 "eighth-size sample of each workload); value is the suite's "
                                 "bytes at the per-element rates measured there",
            "ms_per_step_full_size_estimate": round(statistics.median(ests) * 1e3, 1),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded torch generators)", "config": config_block(),
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": desc,
                             "value": round(value, 4), "unit": UNIT,
                             "sample_wall_seconds_per_step": round(ms / 1e3, 2)},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
