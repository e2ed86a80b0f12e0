"""CPU checks of the benchmark's output contract: the reference arm (the
oracle timed on the host cores) prints one JSON line with the keys the
benchmark's consumers read, and the config block names the workload that a
reduced profiling run measured."""
import json
import os
import subprocess
import sys
import time

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    t0 = time.monotonic()
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2",
                        "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    run_s = time.monotonic() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 2 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # ms_per_step is a measured time: the timed steps fit inside the run
    assert d["steps"] * d["ms_per_step"] / 1e3 < run_s
    assert d["ms_per_step_full_size_estimate"] > d["ms_per_step"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_every_workload_has_bytes_launches_and_full_size():
    names = set(bench.Suite.ORDER)
    assert names == set(bench.BYTES_PER_ELEM) == set(bench.LAUNCHES_PER_STEP)
    assert names == set(bench.FULL_ELEMS)
    # the plain OsciReset step moves 20 + 15.25 bytes per weight; the fused
    # window-end step also reads dist_M and zeroes both accumulators
    assert bench.BYTES_PER_ELEM["osci_update"] == 35.25
    assert bench.BYTES_PER_ELEM["osci_update_reset"] == 43.25


def test_config_block_names_reduced_runs():
    full = bench.config_block()
    assert "workload" in full and full["elements_per_step"] > 0
    sub = bench.config_block(["mxfp4_weight"], None, None, 32768)
    assert sub["workload"].startswith("subset: mxfp4_weight") and "mxfp4 rows=32768" in sub["workload"]
    moe = bench.config_block(list(bench.Suite.ORDER), 2, None)
    assert "moe experts=2" in moe["workload"]
    assert bench.config_block(list(bench.Suite.ORDER)) == full


def test_stored_traffic_is_keyed_on_kernel_sources():
    tr = bench.NCU_TRAFFIC["osci_update_reset"]
    assert tr["bytes"] > 0 and len(tr["src_sha256"]) == 64
    # the key covers the kernel's source and every local header it includes,
    # directly or through another header
    csrc = os.path.join(ROOT, "fp4_quantization_aware_fq_gb300", "csrc")
    seen, todo = set(), ["k_osci.cu"]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        seen.add(name)
        for line in open(os.path.join(csrc, name)):
            if line.startswith('#include "'):
                todo.append(line.split('"')[1])
    assert seen == set(bench.OSCI_SOURCES)
