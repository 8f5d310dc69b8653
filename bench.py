"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = the whole hot path of one linear layer's forward pass on seeded
synthetic inputs already resident in HBM:
  quantise the activation X [M][K] (1x128 tiles), quantise the weight W [N][K]
  (128x128 blocks), FP8 GEMM with per-128-K-group scaling, BF16 output.
Default workload: M=4096, N=7168, K=7168 (the single Fprop linear).  Other
workloads (--workload) cover the backward pass and the MoE grouped GEMM.

Prints ONE JSON line (rank 0).  `value` is the step's algorithmic GEMM
FLOPs (2MNK, summed over ranks) per second of device time; the per-kernel
figures, the roofline of the dominant kernel, an end-to-end number through
host buffers, clocks seen during the timed region and the CPU oracle's
throughput on a bounded sample are added to the same line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
Multi-GPU runs (torchrun, one rank per GPU) are independent replicas of the
same step (weak scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "blockscaled FP8 GEMM TFLOP/s & % FP8 peak; quantize GB/s & % HBM"
L2_BYTES = 126 * 1024 * 1024
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor-core rate
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index, self.period_ms = gpu_index, period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def profile_traffic(kernel_tag: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel, or
    None if there is none or the kernel's source changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    src = os.path.join(ROOT, "fp8_fine_grained_amax_gb300", "csrc", "gemm.cu")
    if not m or not h:
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m.group(1)) if cur == h.group(1) else None


# ----------------------------------------------------------------- workloads
def make_inputs(workload: str):
    from fp8_fine_grained_amax_gb300 import synth
    if workload == "fprop_4096x7168x7168":
        M, N, K = 4096, 7168, 7168
        return dict(M=M, N=N, K=K, X=synth.activation(M, K, seed=0, name="fprop.X"),
                    W=synth.weight(N, K, seed=0, name="fprop.W"))
    if workload.startswith("square_"):
        n = int(workload.split("_")[1])
        return dict(M=n, N=n, K=n, X=synth.activation(n, n, seed=0, name=f"square{n}.X"),
                    W=synth.weight(n, n, seed=0, name=f"square{n}.W"))
    raise SystemExit(f"unknown workload {workload}")


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from fp8_fine_grained_amax_gb300 import binding as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        from fp8_fine_grained_amax_gb300.build import build_library
        build_library()
    if world > 1:
        dist.barrier()
    B.load_library()

    inp = make_inputs(args.workload)
    M, N, K = inp["M"], inp["N"], inp["K"]

    def to_pinned(bits):
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    X_h, W_h = to_pinned(inp["X"]), to_pinned(inp["W"])
    X, W = X_h.to(dev), W_h.to(dev)
    qa = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sa = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    qb = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sb = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    C_h = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        B.fp8q_quant_act(X, q=qa, sa=sa, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        B.fp8q_quant_weight(W, q=qb, sb=sb, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        B.fp8q_gemm(qa, sa, qb, sb, c=C, stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if B.fp8q_sync_status(stream) != 0:
        raise SystemExit("device status error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    status = B.fp8q_sync_status(stream)
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")
    k_act = [e[0].elapsed_time(e[1]) for e in evs]
    k_w = [e[1].elapsed_time(e[2]) for e in evs]
    k_gemm = [e[2].elapsed_time(e[3]) for e in evs]

    # end to end through host buffers: H2D of X and W from pinned memory,
    # the three kernels, D2H of C to pinned memory, every step
    e2e_steps = max(3, min(20, args.steps))
    for _ in range(2):
        X.copy_(X_h, non_blocking=True)
        W.copy_(W_h, non_blocking=True)
        step()
        C_h.copy_(C, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        X.copy_(X_h, non_blocking=True)
        W.copy_(W_h, non_blocking=True)
        step()
        C_h.copy_(C, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    ms_step = total_ms / args.steps
    times = torch.tensor([ms_step, e2e_ms], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    ms_step, e2e_ms = times.tolist()
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    flops = 2.0 * M * N * K
    hbm, bf16, bf16_sus, src = peaks()
    fp8_peak = bf16 * FP8_OVER_BF16
    gemm_ms = statistics.mean(k_gemm)
    act_ms, w_ms = statistics.mean(k_act), statistics.mean(k_w)
    act_bytes = M * K * 2 + M * K + (K // 128) * M * 4
    w_bytes = N * K * 2 + N * K + ((N + 127) // 128) * (K // 128) * 4
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(world * flops / (ms_step * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "step": "quant_act(X) + quant_weight(W) + fp8_gemm -> bf16",
                   "l2": f"inputs larger than L2 ({(M * K + N * K) * 2 / 1e6:.0f} MB BF16 "
                         f"read per step > {L2_BYTES / 1e6:.0f} MB); no flush",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": profile_traffic(f"gemm_fprop_{M}x{N}x{K}"),
                     "kernel": "fp8q_gemm_kernel",
                     "peak_source": f"{src}: bf16 burst {bf16} TFLOP/s x {FP8_OVER_BF16} "
                                    "(nominal fp8/bf16 ratio)"},
        "kernels": {
            "fp8q_gemm_kernel": {"ms": round(gemm_ms, 5), "tflops": round(gemm_tflops, 1),
                                 "frac_fp8_peak": round(gemm_tflops / fp8_peak, 4)},
            "quant_act_kernel": {"ms": round(act_ms, 5),
                                 "gbs": round(act_bytes / (act_ms * 1e-3) / 1e9, 1),
                                 "frac_hbm": round(act_bytes / (act_ms * 1e-3) / 1e9 / hbm, 4)},
            "quant_weight_kernel": {"ms": round(w_ms, 5),
                                    "gbs": round(w_bytes / (w_ms * 1e-3) / 1e9, 1),
                                    "frac_hbm": round(w_bytes / (w_ms * 1e-3) / 1e9 / hbm, 4)},
            "hbm_peak_gbs": hbm, "peak_source": src},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (M * K + N * K) * 2, "d2h_bytes_per_step": M * N * 2,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------- CPU oracle
def cpu_baseline(inp, target_s: float):
    """The oracle, as it stands, on a bounded sample of the step; extrapolated
    to the full step and reported in the metric's unit (TFLOP/s)."""
    import oracle
    M, N, K = inp["M"], inp["N"], inp["K"]
    X, W = inp["X"], inp["W"]
    qa, sa = oracle.quant_act(X)           # full quantisers (fast enough), timed below
    qb, sb = oracle.quant_weight(W)
    t0 = time.perf_counter()
    qa, sa = oracle.quant_act(X)
    t_act = time.perf_counter() - t0
    t0 = time.perf_counter()
    qb, sb = oracle.quant_weight(W)
    t_w = time.perf_counter() - t0
    rows = 8
    t0 = time.perf_counter()
    oracle.gemm_rows(qa, sa, qb, sb, oracle.BSCALE_BLOCK, np.arange(rows))
    t_probe = time.perf_counter() - t0
    budget = max(1.0, target_s - t_act - t_w - t_probe)
    rows = int(min(M, max(8, rows * budget / max(t_probe, 1e-3))))
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(M, size=rows, replace=False))
    t0 = time.perf_counter()
    oracle.gemm_rows(qa, sa, qb, sb, oracle.BSCALE_BLOCK, sample)
    t_gemm = time.perf_counter() - t0
    step_s = t_act + t_w + t_gemm * (M / rows)
    return {"value": round(2.0 * M * N * K / step_s / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"quant_act {M}x{K} and quant_weight {N}x{K} in full "
                      f"({t_act:.2f} s + {t_w:.2f} s); GEMM on {rows} of {M} rows "
                      f"({t_gemm:.2f} s), extrapolated linearly to {M} rows",
            "seconds": round(t_act + t_w + t_gemm, 2)}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle on the host cores, same metric and config."""
    if rank != 0:
        return None
    inp = make_inputs(args.workload)
    M, N, K = inp["M"], inp["N"], inp["K"]
    per_step = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(inp, per_step)
        if i >= args.warmup:
            vals.append(cb)
    value = statistics.median(v["value"] for v in vals)
    step_ms = 2.0 * M * N * K / (value * 1e12) * 1e3
    cb = dict(vals[-1])
    cb["value"] = value
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "step": "quant_act(X) + quant_weight(W) + scaled GEMM (CPU oracle)"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="fprop_4096x7168x7168")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
