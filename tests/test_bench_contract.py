"""CPU checks of bench.py's contract: the reference arm's JSON line (the
oracle timed on the host, tiny workload), argument checks, and the lookup of
DRAM traffic in the committed ncu summaries."""
import hashlib
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_json_line():
    import time
    t0 = time.time()
    r = _run("--impl", "reference", "--workload", "tiny_fprop", "--steps", "3", "--warmup", "3")
    wall = time.time() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None
    assert d["data"] == "synthetic"
    assert d["config"]["workload"] == "tiny_fprop"
    assert d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the steps it reports were run, within the process's own wall time
    assert d["ms_per_step"] * d["steps"] / 1e3 < wall
    assert d["work_per_step"] > 0
    assert abs(d["work_per_step"] / (d["ms_per_step"] * 1e-3) / 1e12 - d["value"]) < \
        0.25 * d["value"]
    # the same config dict as our arm's line for this workload
    import bench
    import numpy as np
    wl = bench.make_workload("tiny_fprop")
    assert d["config"] == json.loads(json.dumps(
        bench.workload_config(wl, wl.in_bytes(wl.host_inputs()), 1)))


def test_warmup_below_three_is_rejected():
    r = _run("--impl", "reference", "--workload", "tiny_fprop", "--steps", "3", "--warmup", "2",
             timeout=120)
    assert r.returncode != 0
    assert "warmup" in (r.stderr + r.stdout)


def test_unknown_workload_is_rejected():
    r = _run("--impl", "reference", "--workload", "no_such_workload", "--steps", "3",
             "--warmup", "3", timeout=120)
    assert r.returncode != 0


@pytest.mark.parametrize("kernel,workload", [
    ("fp8q_gemm_kernel", "fprop_4096x7168x7168"),
    ("fp8q_gemm_mx_kernel", "fprop_pow2_4096x7168x7168"),
    ("no_such_kernel", "fprop_4096x7168x7168"),
])
def test_profile_traffic_follows_the_source_hash(kernel, workload):
    # the traffic of a committed summary is reported only while the kernel's
    # source still hashes to the value recorded with the counters
    import bench
    got = bench.profile_traffic(kernel, workload)
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        assert got is None
        return
    text = open(path).read()
    src = re.search(r"source_file:\s*(\S+)", text).group(1)
    recorded = re.search(r"source_sha256:\s*([0-9a-f]{64})", text).group(1)
    cur = hashlib.sha256(open(os.path.join(ROOT, "fp8_fine_grained_amax_gb300", "csrc", src),
                              "rb").read()).hexdigest()
    dram = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
    assert got == (dram if cur == recorded else None)


@pytest.mark.gpu
def test_our_arm_json_line_on_the_gpu():
    # our arm on the tiny workload: the JSON line carries the keys the
    # benchmark contract asks for, with the device-resident value, the
    # end-to-end value through host buffers, the roofline of the dominant
    # kernel and the launch count of our kernels in the timed region
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = _run("--workload", "tiny_fprop", "--steps", "20", "--warmup", "3", "--no-cpu-baseline")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["value"] > 0 and d["steps"] == 20 and d["warmup"] == 3
    # quant_act, quant_weight, GEMM per step; the 20-step loop repeated until
    # the timed region has lasted at least a second
    assert d["repeats"] >= 1 and d["gpu_launches"] == 3 * 20 * d["repeats"]
    assert d["timed_s"] >= 0.9
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["kernel"] == "fp8q_gemm_kernel"
    assert roof["peak"] > 0 and abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 2 * (256 * 512 + 256 * 512)   # X and W, BF16
    assert e2e["d2h_bytes_per_step"] == 2 * 256 * 256                 # C, BF16
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["clocks"]["samples"] >= 1, d["clocks"]
    assert "workloads" not in d                  # only the headline run measures them all
    # the timed loop is a replayed CUDA graph, and the per-kernel intervals
    # (timing events on a side stream at every kernel boundary) cover the step
    assert d["timing"]["mode"] == "cuda_graph", d["timing"]
    kms = sum(v["ms"] for v in d["kernels"].values() if isinstance(v, dict))
    assert 0.8 * d["ms_per_step"] <= kms <= 1.05 * d["ms_per_step"], (kms, d["ms_per_step"])


@pytest.mark.parametrize("name", [n for _, n in __import__("bench").CONFIG_WORKLOADS] +
                         ["fprop_4096x7168x7168", "quant_tensor_4096", "quant_weight_16x4096"])
def test_every_configured_workload_is_known(name):
    # every workload the headline run measures (and the older names) parses,
    # and its algorithmic work is positive
    import bench
    wl = bench.make_workload(name)
    assert wl.name == name
    assert wl.work() > 0


def test_buffer_copies_rotate_inputs_under_twice_the_l2():
    # one copy only when a step's inputs alone exceed twice the L2; otherwise
    # enough copies that the inputs read between two uses of a copy exceed
    # twice the L2 (the Fprop step's 161 MB needs three)
    import bench
    L2 = bench.L2_BYTES
    assert bench.buffer_copies(2 * L2 + 1) == 1
    assert bench.buffer_copies(161 << 20) == 3
    for n in (1 << 20, 58 << 20, L2, 2 * L2):
        c = bench.buffer_copies(n)
        assert c == min(bench.MAX_COPIES, -(-2 * L2 // n) + 1)
        assert (c - 1) * n >= 2 * L2 or c == bench.MAX_COPIES


def test_quant_weight_names():
    import bench
    a = bench.make_workload("quant_weight_7168x7168")
    assert (a.rows * a.groups, a.cols) == (7168, 7168)
    b = bench.make_workload("quant_weight_16x4096x7168")
    assert (b.rows, b.cols, b.groups) == (4096, 7168, 16)
    c = bench.make_workload("quant_weight_16x4096")
    assert (c.rows * c.groups, c.cols) == (65536, 7168)
