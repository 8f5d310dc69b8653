"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = the whole hot path of one workload on seeded synthetic inputs that
are already resident in HBM.  The headline workload is the forward pass of one
linear layer, M=4096 tokens, N=7168 outputs, K=7168 inputs:
  quantise the activation X [M][K] (1x128 tiles), quantise the weight W [N][K]
  (128x128 blocks), FP8 GEMM with per-128-K-group scaling, BF16 output.
Other workloads (--workload, and all of them in the line's "workloads" key):
  tiny_fprop             256 x 256 x 512 Fprop (the small parity case)
  fprop_pow2_4096x7168x7168  the headline with power-of-two scales (block-scaled MMA)
  linear_bwd_T8192       Dgrad + Wgrad of a 7168->2048 linear over 8192 tokens,
                         with the 128x1 / fused 1x128 and 128x128 quantisers
  linear_bwd_pow2_T8192  the same with power-of-two scales
  linear_bwd_cached_T8192  the backward with X requantised from the FP8 cache
  moe_fprop_16x16384     MoE up- (7168->4096) and down-projection (2048->7168),
                         16 experts, Dirichlet(0.5) top-1 routing, grouped GEMMs
  moe_fprop_pow2_16x16384  the same with power-of-two scales
  square_<n>             n x n x n Fprop step (quantise both operands + GEMM)
  quant_act_<t>          1x128 quantisation of t x 7168 (GB/s)
  quant_act_pow2_<t>     same with power-of-two scales (GB/s)
  quant_act_T_<t>        128x1 transposed quantisation of t x 7168 (GB/s)
  quant_act_T_pow2_<t>   same with power-of-two scales (GB/s)
  quant_weight_<n>x<k>   128x128 quantisation of one n x k weight (GB/s)
  quant_weight_<g>x<n>x<k>  the same over g stacked n x k weights (GB/s)
  quant_tensor_<t>       per-tensor quantisation of t x 7168, for comparison (GB/s)

Prints ONE JSON line (rank 0).  `value` is the step's algorithmic work (GEMM
FLOPs 2MNK over real rows, or quantiser bytes) summed over ranks per second of
device time.  The timed region is the K-step loop, repeated until it has run
for at least --min-seconds (each repeat between a barrier and a device
synchronise); the median repeat gives `ms_per_step`.  The K-step loop is
captured once as a CUDA graph and replayed (--no-graph launches it from the
host instead), so that the device runs the kernels back to back rather than
waiting on host launch overhead; the per-kernel times come from timing events
between the kernels inside the graph.  The per-kernel times, the
roofline of the dominant kernel, an end-to-end number through host buffers,
the clocks sampled during the timed region, the error of the result against
the CPU oracle, the CPU oracle's own throughput, and (one GPU) the same
per-kernel measurement for every other workload are added.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
Multi-GPU runs (torchrun, one process per GPU) are independent replicas of the
same step (weak scaling): the path has no exchange step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
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
HEADLINE = "fprop_4096x7168x7168"
L2_BYTES = 126 * 1024 * 1024
FP8_OVER_BF16 = 2.0          # nominal dense FP8 / BF16 tensor-core rate
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CSRC = os.path.join(ROOT, "fp8_fine_grained_amax_gb300", "csrc")

# Every configuration's workloads (tiny Fprop; Fprop; linear backward; MoE;
# quantiser and square-GEMM sweep), each measured after the headline in the
# same run, with its own timed region.
CONFIG_WORKLOADS = [
    ("tiny", "tiny_fprop"),
    ("fprop", "fprop_pow2_4096x7168x7168"),
    ("linear_bwd", "linear_bwd_T8192"),
    ("linear_bwd", "linear_bwd_pow2_T8192"),
    ("linear_bwd", "linear_bwd_cached_T8192"),
    ("moe", "moe_fprop_16x16384"),
    ("moe", "moe_fprop_pow2_16x16384"),
    ("sweep", "quant_act_4096"),
    ("sweep", "quant_act_16384"),
    ("sweep", "quant_act_65536"),
    ("sweep", "quant_act_pow2_4096"),
    ("sweep", "quant_act_pow2_16384"),
    ("sweep", "quant_act_pow2_65536"),
    ("sweep", "quant_act_T_4096"),
    ("sweep", "quant_act_T_16384"),
    ("sweep", "quant_act_T_65536"),
    ("sweep", "quant_act_T_pow2_65536"),
    ("sweep", "quant_weight_7168x7168"),
    ("sweep", "quant_weight_16x4096x7168"),
    ("sweep", "square_2048"),
    ("sweep", "square_4096"),
    ("sweep", "square_8192"),
    ("sweep", "square_16384"),
]


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
    """nvidia-smi samples of SM clock and throttle reasons, each stamped with
    the host time it arrived, for the whole run; summary() picks the samples
    of one timed window.  Query only: it changes no setting of the GPU."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu_index, self.period_ms = gpu_index, period_ms
        self.proc = None
        self.samples = []           # (host time, sm MHz, max MHz, power W, active reasons)
        self.first = threading.Event()

    def start(self, wait_s: float = 5.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            self.first.wait(wait_s)      # the first sample is in before timing starts
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax, pw = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            act = [nm for nm, v in zip(self.REASONS, parts[5:9]) if v.lower() == "active"]
            self.samples.append((time.time(), sm, smax, pw, act))
            self.first.set()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)
            self.proc = None

    def summary(self, t0: float, t1: float):
        win = [s for s in list(self.samples) if t0 <= s[0] <= t1]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win),
                "power_w_max": max(s[3] for s in win),
                "reasons": sorted({r for s in win for r in s[4]}), "samples": len(win)}


def profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None if there is none or the kernel's source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    f = re.search(r"source_file:\s*(\S+)", text)
    if not m or not h or not f:
        return None
    src = os.path.join(CSRC, f.group(1))
    if not os.path.exists(src):
        return None
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m.group(1)) if cur == h.group(1) else None


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank values over all ranks (the slowest rank's
    times); the identity for a single process."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_value(work_per_rank, world, ms_step, scale):
    """Throughput of all ranks together: every rank does `work_per_rank` per
    step (weak scaling) and the job's step takes the slowest rank's time."""
    return world * work_per_rank / (ms_step * 1e-3) / scale


_HOST_CACHE = {}


def cached(key, make):
    """Host inputs drawn once per process (several workloads share a tensor)."""
    if key not in _HOST_CACHE:
        _HOST_CACHE[key] = make()
    return _HOST_CACHE[key]


def _host_tensor(bits, pin):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t


def _host_copies(inp, names, host, pin=True):
    """Host copies of the named BF16 inputs (shared with `host` if given);
    pinned for the end-to-end leg."""
    if host is not None:
        return {n + "_h": host[n + "_h"] for n in names}
    return {n + "_h": _host_tensor(inp[n], pin) for n in names}


def _host_out(host, name, shape, dtype, pin=True):
    """Host buffer for a result (shared with `host`'s if given)."""
    import torch
    if host is not None:
        return host["io_out"][name][0]
    t = torch.empty(shape, dtype=dtype)
    return t.pin_memory() if pin else t


def _row_sample(M, n, seed=0):
    return np.sort(np.random.default_rng(seed).choice(M, size=min(M, n), replace=False))


def _rows_for_budget(run, M, budget_s):
    """Rows of a seeded sample sized so that run(rows) takes about budget_s."""
    probe = np.arange(min(M, 8))
    t0 = time.perf_counter()
    run(probe)
    t_probe = max(time.perf_counter() - t0, 1e-3)
    return int(min(M, max(probe.size, probe.size * max(budget_s, 0.25) / t_probe)))


# ----------------------------------------------------------------- workloads
class Kernel:
    """One launch of the step: name, call, algorithmic work and its bound."""

    def __init__(self, name, fn, work, bound):
        self.name, self.fn, self.work, self.bound = name, fn, work, bound


class Workload:
    unit = "TFLOP/s"
    work_bound = "tensor"
    io_inputs = ()

    def host_inputs(self):            # name -> BF16 bits / int arrays
        raise NotImplementedError

    def setup(self, dev, inp, host=None, pin=True):   # device tensors; host copies
        raise NotImplementedError

    def kernels(self, st, stream):     # list of Kernel
        raise NotImplementedError

    def cpu_step(self, inp, budget_s, full=False):
        """The oracle on this step: every part in full when `full`, else a
        bounded sample.  Returns a dict: est_s (time of the whole step,
        extrapolated linearly where rows were sampled), spent (seconds
        actually run), work_done (the metric's work of what was run), sample
        (description), and the references kept for error reports."""
        raise NotImplementedError

    def work(self):
        """Algorithmic work of one step in the metric's unit (same formulas
        as kernels(); no GPU needed)."""
        raise NotImplementedError

    def in_bytes(self, inp):
        return sum(int(inp[n].nbytes) for n in self.io_inputs)

    def h2d(self, st):                  # copy the step's inputs host -> device
        for name, (host, dev) in st["io_in"].items():
            dev.copy_(host, non_blocking=True)

    def d2h(self, st):
        for name, (host, dev) in st["io_out"].items():
            host.copy_(dev, non_blocking=True)

    def io_bytes(self, st):
        bi = sum(h.numel() * h.element_size() for h, _ in st["io_in"].values())
        bo = sum(h.numel() * h.element_size() for h, _ in st["io_out"].values())
        return bi, bo


class Fprop(Workload):
    """quant_act(X) + quant_weight(W) + GEMM.  pow2: power-of-two scales, and the
    GEMM on the block-scaled MMA (fp8q_gemm_pow2)."""

    io_inputs = ("X", "W")

    def __init__(self, name, M, N, K, pow2=False):
        self.name, self.M, self.N, self.K, self.pow2 = name, M, N, K, pow2
        self.config = {"M": M, "N": N, "K": K,
                       "step": ("quant_act(X, pow2) + quant_weight(W, pow2) + fp8_gemm_pow2 "
                                "-> bf16") if pow2 else
                               "quant_act(X) + quant_weight(W) + fp8_gemm -> bf16"}

    def host_inputs(self):
        from fp8_fine_grained_amax_gb300 import synth
        tag = self.name.replace("_pow2", "")
        M, N, K = self.M, self.N, self.K
        return {"X": cached(("act", M, K, tag), lambda: synth.activation(M, K, 0, f"{tag}.X")),
                "W": cached(("w", N, K, tag), lambda: synth.weight(N, K, 0, f"{tag}.W"))}

    def setup(self, dev, inp, host=None, pin=True):
        import torch
        M, N, K = self.M, self.N, self.K
        st = _host_copies(inp, ("X", "W"), host, pin)
        st["X"], st["W"] = st["X_h"].to(dev), st["W_h"].to(dev)
        st["qa"] = torch.empty((M, K), dtype=torch.uint8, device=dev)
        st["sa"] = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
        st["qb"] = torch.empty((N, K), dtype=torch.uint8, device=dev)
        st["sb"] = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
        st["C"] = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        st["io_in"] = {"X": (st["X_h"], st["X"]), "W": (st["W_h"], st["W"])}
        st["io_out"] = {"C": (_host_out(host, "C", (M, N), torch.bfloat16, pin), st["C"])}
        return st

    def kernels(self, st, stream):
        from fp8_fine_grained_amax_gb300 import binding as B
        M, N, K = self.M, self.N, self.K
        mode = B.FP8Q_SCALE_POW2 if self.pow2 else B.FP8Q_SCALE_FP32
        gemm = B.fp8q_gemm_pow2 if self.pow2 else B.fp8q_gemm
        return [
            Kernel("quant_act_kernel",
                   lambda: B.fp8q_quant_act(st["X"], q=st["qa"], sa=st["sa"], scale_mode=mode,
                                            stream=stream),
                   M * K * 2 + M * K + (K // 128) * M * 4, "hbm"),
            Kernel("quant_weight_kernel",
                   lambda: B.fp8q_quant_weight(st["W"], q=st["qb"], sb=st["sb"], scale_mode=mode,
                                               stream=stream),
                   N * K * 3 + ((N + 127) // 128) * (K // 128) * 4, "hbm"),
            Kernel("fp8q_gemm_mx_kernel" if self.pow2 else "fp8q_gemm_kernel",
                   lambda: gemm(st["qa"], st["sa"], st["qb"], st["sb"], c=st["C"], stream=stream),
                   2.0 * M * N * K, "tensor"),
        ]

    def work(self):
        return 2.0 * self.M * self.N * self.K

    def cpu_step(self, inp, budget_s, full=False):
        import oracle
        M, N, K, p2 = self.M, self.N, self.K, self.pow2
        t0 = time.perf_counter()
        qb, sb = oracle.quant_weight(inp["W"], p2)
        t_w = time.perf_counter() - t0
        if full:
            rows = np.arange(M)
        else:
            def probe(r):
                qa_r, sa_r = oracle.quant_act(inp["X"][r], p2)
                oracle.gemm_rows(qa_r, sa_r, qb, sb, oracle.BSCALE_BLOCK)
            rows = _row_sample(M, _rows_for_budget(probe, M, budget_s - t_w))
        # the sampled rows' activations are quantised (1x128 tiles are per row)
        t0 = time.perf_counter()
        qa, sa = oracle.quant_act(np.ascontiguousarray(inp["X"][rows]), p2)
        t_a = time.perf_counter() - t0
        t0 = time.perf_counter()
        c_ref, absdot = oracle.gemm_rows(qa, sa, qb, sb, oracle.BSCALE_BLOCK)
        t_g = time.perf_counter() - t0
        r = rows.size
        est = t_w + (t_a + t_g) * M / r
        what = "in full" if r == M else f"on {r} of {M} rows, extrapolated linearly"
        return {"est_s": est, "spent": t_w + t_a + t_g, "work_done": 2.0 * r * N * K,
                "sample": (f"quant_weight {N}x{K} in full ({t_w:.2f} s); quant_act and GEMM "
                           f"{what} ({t_a:.2f} s + {t_g:.2f} s)"),
                "rows": rows, "c_ref": c_ref, "absdot": absdot}


class LinearBwd(Workload):
    """Backward of Y = X W^T with X [T][d_in], W [d_out][d_in], dY [T][d_out]."""

    io_inputs = ("dY", "X", "W")

    def __init__(self, T=8192, d_in=7168, d_out=2048, pow2=False):
        self.name = f"linear_bwd_pow2_T{T}" if pow2 else f"linear_bwd_T{T}"
        self.T, self.d_in, self.d_out, self.pow2 = T, d_in, d_out, pow2
        self.config = {"T": T, "d_in": d_in, "d_out": d_out,
                       "step": "quant_act_T(dY, fused 1x128) + quant_act_T(X) + "
                               "quant_weight(W, transposed) + Dgrad (bf16) + Wgrad (fp32)" +
                               (", power-of-two scales, GEMMs on the block-scaled MMA"
                                if pow2 else "")}

    def host_inputs(self):
        from fp8_fine_grained_amax_gb300 import synth
        T, di, do = self.T, self.d_in, self.d_out
        return {"dY": cached(("dY", T, do), lambda: synth.normal_bf16((T, do), 1e-3, 0, "bwd.dY")),
                "X": cached(("bX", T, di), lambda: synth.activation(T, di, 0, "bwd.X")),
                "W": cached(("bW", do, di), lambda: synth.weight(do, di, 0, "bwd.W"))}

    def setup(self, dev, inp, host=None, pin=True):
        import torch
        T, di, do = self.T, self.d_in, self.d_out
        u8, f32 = torch.uint8, torch.float32
        st = _host_copies(inp, self.io_inputs, host, pin)
        for k in self.io_inputs:
            st[k] = st[k + "_h"].to(dev)
        e = lambda *s, dt=u8: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        st.update(qdyT=e(do, T), sdyT=e(T // 128, do, dt=f32), qdy=e(T, do),
                  sdy=e(do // 128, T, dt=f32), qxT=e(di, T), sxT=e(T // 128, di, dt=f32),
                  qw=e(do, di), sw=e(do // 128, di // 128, dt=f32), qwT=e(di, do),
                  dX=e(T, di, dt=torch.bfloat16), dW=e(do, di, dt=f32))
        st["io_in"] = {k: (st[k + "_h"], st[k]) for k in self.io_inputs}
        st["io_out"] = {"dX": (_host_out(host, "dX", (T, di), torch.bfloat16, pin), st["dX"]),
                        "dW": (_host_out(host, "dW", (do, di), f32, pin), st["dW"])}
        return st

    def kernels(self, st, stream):
        from fp8_fine_grained_amax_gb300 import binding as B
        T, di, do = self.T, self.d_in, self.d_out
        mode = B.FP8Q_SCALE_POW2 if self.pow2 else B.FP8Q_SCALE_FP32
        gemm = B.fp8q_gemm_pow2 if self.pow2 else B.fp8q_gemm
        gname = "fp8q_gemm_mx_kernel" if self.pow2 else "fp8q_gemm_kernel"
        return [
            Kernel("quant_act_T_kernel(dY,rows)", lambda: B.fp8q_quant_act_T(
                st["dY"], with_rows=True, qT=st["qdyT"], sT=st["sdyT"], q_rows=st["qdy"],
                s_rows=st["sdy"], scale_mode=mode, stream=stream), T * do * 4 +
                (T // 128) * do * 4 + (do // 128) * T * 4, "hbm"),
            Kernel("quant_act_T_kernel(X)", lambda: B.fp8q_quant_act_T(
                st["X"], qT=st["qxT"], sT=st["sxT"], scale_mode=mode, stream=stream),
                T * di * 3 + (T // 128) * di * 4, "hbm"),
            Kernel("quant_weight_kernel(T)", lambda: B.fp8q_quant_weight(
                st["W"], with_transpose=True, q=st["qw"], qT=st["qwT"], sb=st["sw"],
                scale_mode=mode, stream=stream), do * di * 4 + (do // 128) * (di // 128) * 4,
                "hbm"),
            Kernel(gname + "(dgrad)", lambda: gemm(
                st["qdy"], st["sdy"], st["qwT"], st["sw"], bscale_kind=B.FP8Q_BSCALE_BLOCK_T,
                c=st["dX"], stream=stream), 2.0 * T * di * do, "tensor"),
            Kernel(gname + "(wgrad)", lambda: gemm(
                st["qdyT"], st["sdyT"], st["qxT"], st["sxT"], bscale_kind=B.FP8Q_BSCALE_ROW,
                out_dtype=B.FP8Q_OUT_FP32, c=st["dW"], stream=stream), 2.0 * do * di * T,
                "tensor"),
        ]

    def work(self):
        return 2 * 2.0 * self.T * self.d_in * self.d_out

    def _quantise(self, inp):
        import oracle
        p2 = self.pow2
        qdyT, sdyT = oracle.quant_act_T(inp["dY"], p2)
        qdy, sdy = oracle.quant_act(inp["dY"], p2)
        qxT, sxT = oracle.quant_act_T(inp["X"], p2)
        qw, sw = oracle.quant_weight(inp["W"], p2)
        return qdyT, sdyT, qdy, sdy, qxT, sxT, np.ascontiguousarray(qw.T), sw

    def cpu_step(self, inp, budget_s, full=False):
        import oracle
        T, di, do = self.T, self.d_in, self.d_out
        t0 = time.perf_counter()
        qdyT, sdyT, qdy, sdy, qxT, sxT, qwT, sw = self._quantise(inp)
        t_q = time.perf_counter() - t0
        dgrad = lambda r: oracle.gemm_rows(qdy, sdy, qwT, sw, oracle.BSCALE_BLOCK_T, r)  # noqa
        wgrad = lambda r: oracle.gemm_rows(qdyT, sdyT, qxT, sxT, oracle.BSCALE_ROW, r)  # noqa
        half = (budget_s - t_q) / 2
        rd = np.arange(T) if full else _row_sample(T, _rows_for_budget(dgrad, T, half))
        rw = np.arange(do) if full else _row_sample(do, _rows_for_budget(wgrad, do, half), 1)
        t0 = time.perf_counter()
        dgrad(rd)
        t_d = time.perf_counter() - t0
        t0 = time.perf_counter()
        wgrad(rw)
        t_w = time.perf_counter() - t0
        est = t_q + t_d * T / rd.size + t_w * do / rw.size
        what = "in full" if (rd.size == T and rw.size == do) else \
            f"on {rd.size} of {T} and {rw.size} of {do} rows, extrapolated linearly"
        return {"est_s": est, "spent": t_q + t_d + t_w,
                "work_done": 2.0 * di * (rd.size * do + rw.size * T),
                "sample": (f"all quantisers in full ({t_q:.2f} s); Dgrad and Wgrad {what} "
                           f"({t_d:.2f} s + {t_w:.2f} s)")}


class LinearBwdCached(LinearBwd):
    """The same backward, with X taken from the forward pass's FP8 cache (1x128
    codes and scales) and requantised 128x1 instead of read again as BF16."""

    def __init__(self, T=8192, d_in=7168, d_out=2048):
        super().__init__(T, d_in, d_out)
        self.name = f"linear_bwd_cached_T{T}"
        self.config = dict(self.config, step="quant_act_T(dY, fused 1x128) + requant_act_T(X "
                           "from FP8 cache) + quant_weight(W, transposed) + Dgrad + Wgrad")

    def setup(self, dev, inp, host=None, pin=True):
        from fp8_fine_grained_amax_gb300 import binding as B
        st = super().setup(dev, inp, host, pin)
        st["qx_cache"], st["sx_cache"] = B.fp8q_quant_act(st["X"])   # the forward pass's cache
        return st

    def kernels(self, st, stream):
        from fp8_fine_grained_amax_gb300 import binding as B
        ks = super().kernels(st, stream)
        T, di = self.T, self.d_in
        ks[1] = Kernel("requant_act_T_kernel(X)", lambda: B.fp8q_requant_act_T(
            st["qx_cache"], st["sx_cache"], qT=st["qxT"], sT=st["sxT"], stream=stream),
            T * di * 2 + (di // 128) * T * 4 + (T // 128) * di * 4, "hbm")
        return ks

    def _quantise(self, inp):
        import oracle
        qx, sx = oracle.quant_act(inp["X"])    # the forward pass's cache
        qdyT, sdyT = oracle.quant_act_T(inp["dY"])
        qdy, sdy = oracle.quant_act(inp["dY"])
        qxT, sxT = oracle.requant_act_T(qx, sx)
        qw, sw = oracle.quant_weight(inp["W"])
        return qdyT, sdyT, qdy, sdy, qxT, sxT, np.ascontiguousarray(qw.T), sw


class MoEFprop(Workload):
    io_inputs = ("X", "H", "Wup", "Wdown")

    def __init__(self, G=16, tokens=16384, d_model=7168, d_ff=4096, d_down_in=2048, pow2=False):
        self.name = f"moe_fprop_pow2_{G}x{tokens}" if pow2 else f"moe_fprop_{G}x{tokens}"
        self.pow2 = pow2
        self.G, self.T, self.dm, self.dff, self.ddi = G, tokens, d_model, d_ff, d_down_in
        self.config = {"experts": G, "tokens": tokens, "up": f"{d_model}->{d_ff}",
                       "down": f"{d_down_in}->{d_model}", "routing": "Dirichlet(0.5) top-1",
                       "step": "quant_act(X) + quant_weight(W_up, all experts) + grouped GEMM "
                               "up; quant_act(H) + quant_weight(W_down) + grouped GEMM down" +
                               ("; power-of-two scales, GEMMs on the block-scaled MMA"
                                if pow2 else "")}

    def host_inputs(self):
        from fp8_fine_grained_amax_gb300 import synth
        G, T, dm, dff, ddi = self.G, self.T, self.dm, self.dff, self.ddi
        return {"offs": synth.moe_offsets(T, G, 0.5, seed=0),
                "X": cached(("moeX", T, dm), lambda: synth.activation(T, dm, 0, "moe.X")),
                "H": cached(("moeH", T, ddi), lambda: synth.normal_bf16((T, ddi), 1.0, 0, "moe.H")),
                "Wup": cached(("moeWup", G, dff, dm),
                              lambda: synth.weight(G * dff, dm, 0, "moe.Wup")),
                "Wdown": cached(("moeWdn", G, dm, ddi),
                                lambda: synth.weight(G * dm, ddi, 0, "moe.Wdown"))}

    def setup(self, dev, inp, host=None, pin=True):
        import torch
        G, T, dm, dff, ddi = self.G, self.T, self.dm, self.dff, self.ddi
        u8, f32 = torch.uint8, torch.float32
        st = _host_copies(inp, self.io_inputs, host, pin)
        for k in self.io_inputs:
            st[k] = st[k + "_h"].to(dev)
        st["offs"] = torch.from_numpy(inp["offs"]).to(dev)
        e = lambda *s, dt=u8: torch.empty(s, dtype=dt, device=dev)  # noqa: E731
        st.update(qx=e(T, dm), sx=e(dm // 128, T, dt=f32), qh=e(T, ddi), sh=e(ddi // 128, T, dt=f32),
                  qup=e(G * dff, dm), sup=e(G * dff // 128, dm // 128, dt=f32),
                  qdn=e(G * dm, ddi), sdn=e(G * dm // 128, ddi // 128, dt=f32),
                  Yup=e(T, dff, dt=torch.bfloat16), Ydn=e(T, dm, dt=torch.bfloat16))
        st["io_in"] = {k: (st[k + "_h"], st[k]) for k in self.io_inputs}
        st["io_out"] = {"Yup": (_host_out(host, "Yup", (T, dff), torch.bfloat16, pin), st["Yup"]),
                        "Ydn": (_host_out(host, "Ydn", (T, dm), torch.bfloat16, pin), st["Ydn"])}
        return st

    def kernels(self, st, stream):
        from fp8_fine_grained_amax_gb300 import binding as B
        G, T, dm, dff, ddi = self.G, self.T, self.dm, self.dff, self.ddi
        mode = B.FP8Q_SCALE_POW2 if self.pow2 else B.FP8Q_SCALE_FP32
        ggemm = B.fp8q_grouped_gemm_pow2 if self.pow2 else B.fp8q_grouped_gemm
        gname = "fp8q_gemm_mx_kernel" if self.pow2 else "fp8q_gemm_kernel"
        return [
            Kernel("quant_act_kernel(X)", lambda: B.fp8q_quant_act(
                st["X"], q=st["qx"], sa=st["sx"], scale_mode=mode, stream=stream),
                T * dm * 3 + T * dm // 32, "hbm"),
            Kernel("quant_weight_kernel(Wup)", lambda: B.fp8q_quant_weight(
                st["Wup"], q=st["qup"], sb=st["sup"], scale_mode=mode, stream=stream),
                G * dff * dm * 3, "hbm"),
            Kernel(gname + "(grouped up)", lambda: ggemm(
                st["qx"], st["sx"], st["qup"].view(G, dff, dm),
                st["sup"].view(G, dff // 128, dm // 128), st["offs"], c=st["Yup"],
                stream=stream), 2.0 * T * dff * dm, "tensor"),
            Kernel("quant_act_kernel(H)", lambda: B.fp8q_quant_act(
                st["H"], q=st["qh"], sa=st["sh"], scale_mode=mode, stream=stream),
                T * ddi * 3 + T * ddi // 32, "hbm"),
            Kernel("quant_weight_kernel(Wdown)", lambda: B.fp8q_quant_weight(
                st["Wdown"], q=st["qdn"], sb=st["sdn"], scale_mode=mode, stream=stream),
                G * dm * ddi * 3, "hbm"),
            Kernel(gname + "(grouped down)", lambda: ggemm(
                st["qh"], st["sh"], st["qdn"].view(G, dm, ddi),
                st["sdn"].view(G, dm // 128, ddi // 128), st["offs"], c=st["Ydn"],
                stream=stream), 2.0 * T * dm * ddi, "tensor"),
        ]

    def work(self):
        return 2.0 * self.T * self.dff * self.dm + 2.0 * self.T * self.dm * self.ddi

    def cpu_step(self, inp, budget_s, full=False):
        import oracle
        G, T, dm, dff, ddi, p2 = self.G, self.T, self.dm, self.dff, self.ddi, self.pow2
        t0 = time.perf_counter()
        qup, sup = oracle.quant_weight(inp["Wup"], p2)
        qdn, sdn = oracle.quant_weight(inp["Wdown"], p2)
        t_w = time.perf_counter() - t0
        offs = inp["offs"]
        qup, sup = qup.reshape(G, dff, dm), sup.reshape(G, dff // 128, dm // 128)
        qdn, sdn = qdn.reshape(G, dm, ddi), sdn.reshape(G, dm // 128, ddi // 128)

        def part(x, qb, sb, rows):   # the listed tokens' 1x128 tiles and GEMM rows
            qa, sa = oracle.quant_act(np.ascontiguousarray(x[rows]), p2)
            # each sampled token keeps its expert: offsets of the sample
            g_of = np.searchsorted(offs, rows, side="right") - 1
            o = np.zeros(G + 1, np.int32)
            o[1:] = np.cumsum(np.bincount(g_of, minlength=G))
            oracle.grouped_gemm_rows(qa, sa, qb, sb, o)

        half = (budget_s - t_w) / 2
        ru = np.arange(T) if full else _row_sample(
            T, _rows_for_budget(lambda r: part(inp["X"], qup, sup, r), T, half))
        rd = np.arange(T) if full else _row_sample(
            T, _rows_for_budget(lambda r: part(inp["H"], qdn, sdn, r), T, half), 1)
        t0 = time.perf_counter()
        part(inp["X"], qup, sup, ru)
        t_u = time.perf_counter() - t0
        t0 = time.perf_counter()
        part(inp["H"], qdn, sdn, rd)
        t_d = time.perf_counter() - t0
        est = t_w + t_u * T / ru.size + t_d * T / rd.size
        what = "in full" if ru.size == T and rd.size == T else \
            f"on {ru.size} and {rd.size} of {T} tokens, extrapolated linearly"
        return {"est_s": est, "spent": t_w + t_u + t_d,
                "work_done": 2.0 * ru.size * dff * dm + 2.0 * rd.size * dm * ddi,
                "sample": (f"expert weights quantised in full ({t_w:.2f} s); token quantisation "
                           f"and grouped GEMMs {what} ({t_u:.2f} s + {t_d:.2f} s)")}


class QuantOnly(Workload):
    unit = "GB/s"
    work_bound = "hbm"
    io_inputs = ("X",)

    def __init__(self, name, kind, rows, cols=7168, groups=1):
        self.kind, self.rows, self.cols, self.groups = kind, rows, cols, groups
        self.name = name
        self.config = {"rows": rows * groups, "cols": cols, "step": kind}
        if groups > 1:
            self.config["weights"] = f"{groups} x {rows}x{cols}"

    def host_inputs(self):
        from fp8_fine_grained_amax_gb300 import synth
        R, C = self.rows * self.groups, self.cols
        if self.kind == "quant_weight":
            return {"X": cached(("sweepW", R, C), lambda: synth.weight(R, C, 0, f"sweep.W{R}"))}
        return {"X": cached(("sweepX", R, C),
                            lambda: synth.activation(R, C, 0, f"sweep.X{R}"))}

    def setup(self, dev, inp, host=None, pin=True):
        import torch
        R, C = self.rows * self.groups, self.cols
        st = _host_copies(inp, ("X",), host, pin)
        st["X"] = st["X_h"].to(dev)
        if self.kind.startswith("quant_act_T"):
            st["q"] = torch.empty((C, R), dtype=torch.uint8, device=dev)
            st["s"] = torch.empty((R // 128, C), dtype=torch.float32, device=dev)
        elif self.kind == "quant_weight":
            st["q"] = torch.empty((R, C), dtype=torch.uint8, device=dev)
            st["s"] = torch.empty(((R + 127) // 128, C // 128), dtype=torch.float32, device=dev)
        else:
            st["q"] = torch.empty((R, C), dtype=torch.uint8, device=dev)
            st["s"] = torch.empty((C // 128, R), dtype=torch.float32, device=dev)
        st["io_in"] = {"X": (st["X_h"], st["X"])}
        st["io_out"] = {"q": (_host_out(host, "q", tuple(st["q"].shape), torch.uint8, pin),
                              st["q"])}
        return st

    def kernels(self, st, stream):
        from fp8_fine_grained_amax_gb300 import binding as B
        R, C = self.rows * self.groups, self.cols
        if self.kind.startswith("quant_act_T"):
            mode = B.FP8Q_SCALE_POW2 if self.kind == "quant_act_T_pow2" else B.FP8Q_SCALE_FP32
            return [Kernel("quant_act_T_kernel", lambda: B.fp8q_quant_act_T(
                st["X"], qT=st["q"], sT=st["s"], scale_mode=mode, stream=stream),
                R * C * 3 + R * C // 32, "hbm")]
        if self.kind == "quant_weight":
            return [Kernel("quant_weight_kernel", lambda: B.fp8q_quant_weight(
                st["X"], q=st["q"], sb=st["s"], stream=stream), self.work(), "hbm")]
        if self.kind == "quant_tensor":
            if "ws" not in st:
                import torch
                st["ws"] = torch.empty((B.fp8q_quant_tensor_workspace_bytes(R, C),),
                                       dtype=torch.uint8, device=st["X"].device)
                st["s1"] = torch.empty((1,), dtype=torch.float32, device=st["X"].device)
            return [Kernel("tensor_amax+quant_kernels", lambda: B.fp8q_quant_tensor(
                st["X"], q=st["q"], s=st["s1"], workspace=st["ws"], stream=stream),
                R * C * 3, "hbm")]
        mode = B.FP8Q_SCALE_POW2 if self.kind == "quant_act_pow2" else B.FP8Q_SCALE_FP32
        return [Kernel("quant_act_kernel", lambda: B.fp8q_quant_act(
            st["X"], q=st["q"], sa=st["s"], scale_mode=mode, stream=stream),
            R * C * 3 + R * C // 32, "hbm")]

    def work(self):
        R, C = self.rows * self.groups, self.cols
        if self.kind == "quant_weight":
            return R * C * 3 + ((R + 127) // 128) * (C // 128) * 4
        return R * C * 3 + (0 if self.kind == "quant_tensor" else R * C // 32)

    def cpu_step(self, inp, budget_s, full=False):
        import oracle
        t0 = time.perf_counter()
        p2 = self.kind.endswith("_pow2")
        if self.kind.startswith("quant_act_T"):
            oracle.quant_act_T(inp["X"], p2)
        elif self.kind == "quant_tensor":
            oracle.quant_tensor(inp["X"])
        elif self.kind == "quant_weight":
            oracle.quant_weight(inp["X"])
        else:
            oracle.quant_act(inp["X"], p2)
        t = time.perf_counter() - t0
        return {"est_s": t, "spent": t, "work_done": self.work(),
                "sample": f"{self.kind} on the full {self.rows * self.groups}x{self.cols} "
                          f"input ({t:.2f} s)"}


def make_workload(name: str) -> Workload:
    if name == "fprop_4096x7168x7168":
        return Fprop(name, 4096, 7168, 7168)
    if name == "fprop_pow2_4096x7168x7168":
        return Fprop(name, 4096, 7168, 7168, pow2=True)
    if name == "tiny_fprop":
        return Fprop(name, 256, 256, 512)
    if name.startswith("square_"):
        n = int(name.split("_")[1])
        return Fprop(name, n, n, n)
    if name == "linear_bwd_T8192":
        return LinearBwd()
    if name == "linear_bwd_pow2_T8192":
        return LinearBwd(pow2=True)
    if name == "linear_bwd_cached_T8192":
        return LinearBwdCached()
    if name == "moe_fprop_16x16384":
        return MoEFprop()
    if name == "moe_fprop_pow2_16x16384":
        return MoEFprop(pow2=True)
    m = re.fullmatch(r"quant_weight_(\d+)x(\d+)(?:x(\d+))?", name)
    if m:
        a, b, c = int(m.group(1)), int(m.group(2)), m.group(3)
        if c is not None:                      # g stacked n x k weights
            return QuantOnly(name, "quant_weight", b, int(c), groups=a)
        if b == 4096:                          # g stacked 4096 x 7168 weights
            return QuantOnly(name, "quant_weight", 4096, 7168, groups=a)
        return QuantOnly(name, "quant_weight", a, b)
    for kind in ("quant_act_T_pow2", "quant_act_pow2", "quant_act_T", "quant_tensor", "quant_act"):
        m = re.fullmatch(kind + r"_(\d+)", name)
        if m:
            return QuantOnly(name, kind, int(m.group(1)))
    raise SystemExit(f"unknown workload {name}")


def workload_config(wl: Workload, in_bytes: int, world: int):
    """The line's `config`: the same dict for both arms of one workload."""
    n = buffer_copies(in_bytes)
    l2 = (f"inputs larger than twice the L2 ({in_bytes / 1e6:.0f} MB read per step > "
          f"2 x {L2_BYTES / 1e6:.0f} MB); no flush" if n == 1 else
          f"inputs {in_bytes / 1e6:.1f} MB, under twice the L2: steps cycle through {n} "
          f"copies of the step's buffers ({n * in_bytes / 1e6:.0f} MB of inputs); no flush")
    return dict(workload=wl.name, **wl.config, l2=l2, parallelism=f"replicas x{world}")


def cpu_baseline(wl: Workload, inp, budget_s: float, full: bool):
    """The oracle, as it stands, on one step (every part in full when `full`,
    else a bounded sample extrapolated to the full step), in the metric's unit."""
    import oracle
    r = wl.cpu_step(inp, budget_s, full)
    scale = 1e12 if wl.unit == "TFLOP/s" else 1e9
    return {"value": round(wl.work() / r["est_s"] / scale, 6), "unit": wl.unit,
            "cores": oracle.num_threads(), "kind": "oracle", "sample": r["sample"],
            "seconds": round(r["spent"], 2)}, r


def gemm_errors(wl: Fprop, inp, st, ref):
    """Error of the GPU result on the oracle's rows: the largest
    |C - C_ref| / tolerance, and (context) the relative Frobenius error
    against an unquantised BF16 GEMM on a 256-row sample of them."""
    import oracle
    rows = ref["rows"]
    c = st["C"].float().cpu().numpy().astype(np.float64)[rows]
    tol = oracle.gemm_tolerance(ref["c_ref"], ref["absdot"], True)
    ratio = float(np.max(np.abs(c - ref["c_ref"]) / tol))
    sub = np.arange(rows.size) if rows.size <= 256 else _row_sample(rows.size, 256, 2)
    c16 = oracle.bf16_gemm_rows(inp["X"], inp["W"], rows[sub])
    fro = float(np.linalg.norm(c[sub] - c16) / np.linalg.norm(c16))
    fro_q = float(np.linalg.norm(ref["c_ref"][sub] - c16) / np.linalg.norm(c16))
    return {"rows_checked": int(rows.size), "cols": int(c.shape[1]),
            "max_err_over_tol": round(ratio, 4),
            "tolerance": "|C - C_ref| <= 2e-4 * sum_k |a_k b_k| + 0.5 ulp_bf16",
            "rel_fro_err_vs_bf16_gemm": round(fro, 6),
            "rel_fro_err_vs_bf16_gemm_oracle": round(fro_q, 6),
            "bf16_rows": int(sub.size)}


# ----------------------------------------------------------------- our arm
def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _graph_events_supported():
    """CUDA events that a graph capture records as timing nodes (torch's
    `external` events) exist in this torch."""
    import inspect

    import torch
    try:
        return "external" in inspect.signature(torch.cuda.Event.__new__).parameters
    except (TypeError, ValueError):
        return False


class Timer:
    """The K-step loop of one workload, repeated `repeats` times; each repeat
    sits between a barrier and a device synchronise.  `ks_sets` holds one
    kernel list per copy of the step's buffers; step i runs on copy
    i % len(ks_sets), so that a workload whose inputs are under twice the L2 reads
    them from HBM (each copy has been evicted by the others by the time it
    comes round again).

    Per-kernel times come from timing events recorded at every kernel
    boundary on a side stream: the compute stream forks to it after each
    kernel, and the next kernel does not wait for the event.  An event
    recorded on the compute stream itself would sit between two kernels and
    hold the next one back (4-7 us per boundary on GB300).

    With `graph`, the K-step loop is captured once as a CUDA graph (one graph
    per starting copy, so that copies keep rotating across repeats) and each
    repeat replays it: the device runs the kernels back to back instead of
    waiting for the host to launch each one."""

    def __init__(self, ks_sets, stream, dev, steps, graph=True):
        import torch
        self.ks_sets, self.stream, self.dev, self.steps = ks_sets, stream, dev, steps
        self.ks = ks_sets[0]
        self.i = 0
        self.graph = bool(graph) and _graph_events_supported()
        kw = {"external": True} if self.graph else {}
        n = steps * len(self.ks) + 1
        self.bevs = [torch.cuda.Event(enable_timing=True, **kw) for _ in range(n)]
        self.forks = [torch.cuda.Event() for _ in range(n)]
        self.join = torch.cuda.Event()
        self.side = torch.cuda.Stream(dev)
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)
        self.graphs = []
        self.graph_error = None

    def step(self, at=None, mark=None):
        """One step's kernels on its buffer copy; `mark(j)` before kernel j."""
        if at is None:
            at = self.i
            self.i += 1
        for j, k in enumerate(self.ks_sets[at % len(self.ks_sets)]):
            if mark is not None:
                mark(j)
            k.fn()

    def _mark(self, n):
        self.forks[n].record(self.stream)
        self.side.wait_event(self.forks[n])
        self.bevs[n].record(self.side)

    def _timed_loop(self, first):
        nk = len(self.ks)
        for i in range(self.steps):
            self.step(first + i, lambda j, i=i: self._mark(i * nk + j))
        self._mark(self.steps * nk)
        self.join.record(self.side)
        self.stream.wait_event(self.join)

    def capture(self):
        """Capture the timed loop (after eager warm-up steps have run every
        kernel once).  Falls back to eager launches if capture fails."""
        import torch
        if not self.graph:
            return
        c = len(self.ks_sets)
        try:
            for j in range(c // math.gcd(self.steps, c)):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
                    self._timed_loop(j * self.steps)
                self.graphs.append(g)
        except RuntimeError as e:  # keep the eager loop
            self.graph_error = str(e).splitlines()[0][:200]
            self.graphs = []
            self.graph = False
            torch.cuda.synchronize(self.dev)

    def loop(self, r):
        """Repeat r of the K-step loop (graph replay or eager launches)."""
        import torch
        if self.graphs:
            with torch.cuda.stream(self.stream):
                self.graphs[r % len(self.graphs)].replay()
        else:
            self._timed_loop(self.i)
            self.i += self.steps

    def mode(self):
        out = {"mode": "cuda_graph" if self.graphs else "eager",
               "kernel_events": "recorded on a side stream at every kernel boundary"}
        if self.graphs:
            out["graphs"] = len(self.graphs)
        if self.graph_error:
            out["graph_error"] = self.graph_error
        return out

    def run(self, repeats, world):
        import torch
        nk = len(self.ks)
        rep_ms, ksum = [], [0.0] * nk
        t0 = time.time()
        for r in range(repeats):
            _barrier(world)
            torch.cuda.synchronize(self.dev)
            self.e0.record(self.stream)
            self.loop(r)
            self.e1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            _barrier(world)
            rep_ms.append(self.e0.elapsed_time(self.e1))
            for n in range(self.steps * nk):
                ksum[n % nk] += self.bevs[n].elapsed_time(self.bevs[n + 1])
        t1 = time.time()
        n = repeats * self.steps
        return {"ms_step": statistics.median(rep_ms) / self.steps,
                "kernel_ms": [s / n for s in ksum], "t0": t0, "t1": t1,
                "timed_s": sum(rep_ms) / 1e3}


MAX_COPIES = 16


def buffer_copies(in_bytes):
    """Copies of the step's buffers to cycle through: enough that the inputs
    read between two uses of one copy exceed twice the L2 (one copy when the
    inputs alone are larger than twice the L2; with inputs between one and
    two L2s, part of one step's inputs would still be in L2 when the next
    step reads them)."""
    if in_bytes > 2 * L2_BYTES:
        return 1
    return int(min(MAX_COPIES, math.ceil(2 * L2_BYTES / max(in_bytes, 1)) + 1))


def kernel_sets(wl, dev, inp, stream, first_st, pin):
    """The step's kernels on `first_st` and on the extra buffer copies."""
    sets = [wl.kernels(first_st, stream)]
    for _ in range(buffer_copies(wl.in_bytes(inp)) - 1):
        sets.append(wl.kernels(wl.setup(dev, inp, pin=pin), stream))
    return sets


def repeats_for(per_step_s, steps, min_s, world, dev):
    """Repeats of the K-step loop that make the timed region last min_s
    (the same on every rank)."""
    r = max(1, math.ceil(min_s / max(per_step_s * steps, 1e-6)))
    r = min(r, 100000)
    return int(max_over_ranks([r], world, device=dev)[0])


def warm_up(timer, warmup, dev):
    """W untimed steps (at least one per buffer copy), the capture of the
    timed loop and one replay of each graph, then three calibration passes;
    returns the fastest one's device time per step (what sizes the repeats of
    the timed region)."""
    import torch
    for _ in range(max(warmup, len(timer.ks_sets))):
        timer.step()
    torch.cuda.synchronize(dev)
    timer.capture()
    for r in range(len(timer.graphs)):  # the first launch of a graph uploads it
        timer.loop(r)
    torch.cuda.synchronize(dev)
    best = float("inf")
    for r in range(3):
        timer.e0.record(timer.stream)
        timer.loop(r)
        timer.e1.record(timer.stream)
        torch.cuda.synchronize(dev)
        best = min(best, timer.e0.elapsed_time(timer.e1))
    return best * 1e-3 / timer.steps


def kernel_table(ks, kms, hbm, fp8_peak):
    out = {}
    for k, ms in zip(ks, kms):
        if k.bound == "tensor":
            a = k.work / (ms * 1e-3) / 1e12
            out[k.name] = {"ms": round(ms, 5), "tflops": round(a, 1),
                           "frac_fp8_peak": round(a / fp8_peak, 4)}
        else:
            a = k.work / (ms * 1e-3) / 1e9
            out[k.name] = {"ms": round(ms, 5), "gbs": round(a, 1), "frac_hbm": round(a / hbm, 4)}
    return out


def measure_other(name, dev, stream, args, clk, hbm, fp8_peak):
    """One more workload on this GPU: per-kernel times over a timed region of
    at least --min-seconds, and the clocks seen during it."""
    import torch
    from fp8_fine_grained_amax_gb300 import binding as B
    wl = make_workload(name)
    inp = wl.host_inputs()
    st = wl.setup(dev, inp, pin=False)
    sets = kernel_sets(wl, dev, inp, stream, st, False)
    ks = sets[0]
    timer = Timer(sets, stream, dev, args.steps, graph=args.graph)
    per_step = warm_up(timer, args.warmup, dev)
    if B.fp8q_sync_status(stream) != 0:
        raise SystemExit(f"device status error in the warm-up of {name}")
    reps = repeats_for(per_step, args.steps, args.min_seconds, 1, dev)
    r = timer.run(reps, 1)
    if B.fp8q_sync_status(stream) != 0:
        raise SystemExit(f"device status error in {name}")
    scale = 1e12 if wl.unit == "TFLOP/s" else 1e9
    work = sum(k.work for k in ks if k.bound == wl.work_bound)
    res = {"value": round(work / (r["ms_step"] * 1e-3) / scale, 2), "unit": wl.unit,
           "ms_per_step": round(r["ms_step"], 5), "steps": args.steps, "repeats": reps,
           "timed_s": round(r["timed_s"], 3),
           "config": workload_config(wl, wl.in_bytes(inp), 1),
           "buffer_copies": len(sets),
           "timing": timer.mode(),
           "kernels": kernel_table(ks, r["kernel_ms"], hbm, fp8_peak),
           "clocks": clk.summary(r["t0"], r["t1"])}
    del st, sets, ks, timer
    torch.cuda.empty_cache()
    return res


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
    _barrier(world)
    B.load_library()

    clk = ClockSampler(local).start()
    wl = make_workload(args.workload)
    inp = wl.host_inputs()
    st = wl.setup(dev, inp)
    # a stream of its own: the legacy default stream cannot be captured
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    copies = kernel_sets(wl, dev, inp, stream, st, True)
    ks = copies[0]
    timer = Timer(copies, stream, dev, args.steps, graph=args.graph)

    per_step = warm_up(timer, args.warmup, dev)
    if B.fp8q_sync_status(stream) != 0:
        raise SystemExit("device status error during warm-up")
    reps = repeats_for(per_step, args.steps, args.min_seconds, world, dev)
    r = timer.run(reps, world)
    status = B.fp8q_sync_status(stream)
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")
    clocks = clk.summary(r["t0"], r["t1"])

    # end to end through host buffers: every step copies its inputs from pinned
    # host memory (H2D stream), runs its kernels (compute stream) and reads its
    # results back to pinned host memory (D2H stream).  Two device buffer sets
    # alternate so that step i+1's input copy and step i-1's result copy overlap
    # step i's kernels, as a pipeline of batches would run.
    st2 = wl.setup(dev, inp, host=st)
    sets = [(st, ks), (st2, wl.kernels(st2, stream))]
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cin.wait_event(e0)
        for i in range(n):
            b = i % 2
            sti, ksi = sets[b]
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(ev_comp[b])       # step i-2 done reading set b
                wl.h2d(sti)
                ev_in[b].record(cin)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])         # step i-2's results copied out
            for k in ksi:
                k.fn()
            ev_comp[b].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(ev_comp[b])
                wl.d2h(sti)
                ev_out[b].record(cout)
        stream.wait_event(ev_out[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(ev_out[(n - 2) % 2])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    e2e_steps = max(4, min(40, args.steps))
    e2e_run(4)
    e2e_ms = e2e_run(e2e_steps) / e2e_steps
    if B.fp8q_sync_status(stream) != 0:
        raise SystemExit("device status error in the end-to-end leg")
    # the timed steps ran on `st`; run one more step on it so that its output
    # is this step's result again (the end-to-end leg reused its buffers)
    timer.step(at=0)
    torch.cuda.synchronize(dev)

    ms_step, e2e_ms = max_over_ranks([r["ms_step"], e2e_ms], world, device=dev)
    if rank != 0:
        clk.stop()
        if world > 1:
            dist.destroy_process_group()
        return None

    hbm, bf16, bf16_sus, src = peaks()
    fp8_peak = bf16 * FP8_OVER_BF16
    scale = 1e12 if wl.unit == "TFLOP/s" else 1e9
    work = sum(k.work for k in ks if k.bound == wl.work_bound)
    kms = r["kernel_ms"]
    kernels = kernel_table(ks, kms, hbm, fp8_peak)
    dom_i = max(range(len(ks)), key=lambda i: kms[i])
    dom = ks[dom_i]
    base_name = dom.name.split("(")[0]
    if dom.bound == "tensor":
        ach = dom.work / (kms[dom_i] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4),
                "peak_source": f"{src}: bf16 burst {bf16} TFLOP/s x {FP8_OVER_BF16} "
                               "(nominal fp8/bf16 ratio)"}
    else:
        ach = dom.work / (kms[dom_i] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "peak_source": f"{src}: HBM copy bandwidth"}
    roof["traffic"] = profile_traffic(base_name, wl.name)
    roof["kernel"] = dom.name
    roof["work_per_launch"] = dom.work
    bi, bo = wl.io_bytes(st)
    line = {
        "metric": METRIC,
        "value": round(whole_job_value(work, world, ms_step, scale), 2),
        "unit": wl.unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "repeats": reps,
        "timed_s": round(r["timed_s"], 3),
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3 (fp32 accumulate)" if wl.unit == "TFLOP/s" else "bf16 -> e4m3",
        "data": "synthetic",
        "config": workload_config(wl, wl.in_bytes(inp), world),
        "roofline": roof,
        "timing": timer.mode(),
        "kernels": dict(kernels, hbm_peak_gbs=hbm, fp8_peak_tflops=round(fp8_peak, 1),
                        peak_source=src),
        "e2e": {"value": round(whole_job_value(work, world, e2e_ms, scale), 2), "unit": wl.unit,
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "pipeline": "H2D(i+1) and D2H(i-1) overlap kernels(i); 2 device buffer sets"},
        "gpu_launches": len(ks) * args.steps * reps,
        "buffer_copies": len(copies),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        full = isinstance(wl, (Fprop, LinearBwd)) and wl.work() <= 1e12
        cb, ref = cpu_baseline(wl, inp, args.cpu_seconds, full)
        line["cpu_baseline"] = cb
        if isinstance(wl, Fprop):
            line["errors"] = gemm_errors(wl, inp, st, ref)
    if world == 1 and args.all_workloads:
        del st, st2, sets, ks, timer, copies
        torch.cuda.empty_cache()
        others = {}
        for _, name in CONFIG_WORKLOADS:
            if name != wl.name:
                others[name] = measure_other(name, dev, stream, args, clk, hbm, fp8_peak)
        line["workloads"] = others
    clk.stop()
    if world > 1:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------- reference arm
def run_reference(args, rank, world):
    """Reference arm: the CPU oracle on the host cores, same metric and config.
    Each step is a bounded sample of the workload's step (rows of its GEMMs;
    quantisers whole or on the same rows); `value` is the work that sample did
    per second it ran, `ms_per_step` the time one sampled step took."""
    if rank != 0:
        return None
    import oracle
    wl = make_workload(args.workload)
    inp = wl.host_inputs()
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    runs = []
    for i in range(args.warmup + args.steps):
        r = wl.cpu_step(inp, per_step, full=False)
        if i >= args.warmup:
            runs.append(r)
    scale = 1e12 if wl.unit == "TFLOP/s" else 1e9
    rates = [r["work_done"] / r["spent"] / scale for r in runs]
    value = round(statistics.median(rates), 6)
    ms = statistics.median(r["spent"] for r in runs) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": wl.unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (oracle)", "data": "synthetic",
        "config": workload_config(wl, wl.in_bytes(inp), world),
        "work_per_step": runs[-1]["work_done"],
        "cpu_baseline": {"value": value, "unit": wl.unit, "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": "each step: " + runs[-1]["sample"]},
        "e2e": {"value": value, "unit": wl.unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="shortest timed region per workload (repeats of the K-step loop)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", dest="graph", action="store_false", default=True,
                    help="launch the timed loop eagerly instead of replaying it as a CUDA graph")
    ap.add_argument("--all-workloads", dest="all_workloads", action="store_true", default=None,
                    help="also measure every other configuration's workloads (default: on for "
                         "the headline workload on one GPU)")
    ap.add_argument("--no-all-workloads", dest="all_workloads", action="store_false")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.all_workloads is None:
        args.all_workloads = args.workload == HEADLINE
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
