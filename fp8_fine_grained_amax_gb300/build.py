"""Build libfp8q.so in-tree with nvcc for sm_103a.

Each .cu file is compiled separately (in parallel) and linked into one shared
library next to this file.  The CUDA runtime is linked statically, and the
driver's tensor-map encoder is looked up at run time, so loading the library
needs no GPU driver (the symbol check in the CPU tests relies on this).

The GEMM kernel gives registers from its control warpgroup to its epilogue
warpgroups with setmaxnreg; that split is only valid if ptxas builds the
kernel for exactly the launch register count the source assumes
(``kLaunchRegs`` in csrc/gemm.cu).  The build reads ptxas' report and refuses
to link a library that breaks this.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8q.so")
SOURCES = ["gemm.cu", "gemm_mx.cu", "quant.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "fp8q.h"))
    files.append(os.path.abspath(__file__))
    return files


def _up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xptxas", "-v", "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def launch_regs_of(gemm_src: str) -> int:
    """The per-thread launch register count the GEMM source is written for."""
    m = re.search(r"constexpr int kLaunchRegs = (\d+);", open(gemm_src).read())
    if not m:
        raise RuntimeError("kLaunchRegs not found in " + gemm_src)
    return int(m.group(1))


def check_gemm_registers(ptxas_log: str, expected: int, kernel: str = "fp8q_gemm_kernel") -> None:
    """Every instantiation of `kernel` must be built for `expected` registers."""
    entries = re.split(r"Compiling entry function", ptxas_log)
    found = 0
    for e in entries:
        if kernel not in e.split("\n", 1)[0]:
            continue
        m = re.search(r"Used (\d+) registers", e)
        if not m or int(m.group(1)) != expected:
            raise RuntimeError(
                "GEMM kernel not built for %d registers per thread (ptxas: %s); the "
                "setmaxnreg split would not balance" % (expected, m and m.group(0)))
        found += 1
    if found == 0:
        raise RuntimeError("ptxas report names no " + kernel)


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libfp8q.so."""
    if not force and _up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = dict(zip(SOURCES, ex.map(_compile, SOURCES)))
    check_gemm_registers(results["gemm.cu"][1], launch_regs_of(os.path.join(CSRC, "gemm.cu")))
    check_gemm_registers(results["gemm_mx.cu"][1], launch_regs_of(os.path.join(CSRC, "gemm_mx.cu")),
                         "fp8q_gemm_mx_kernel")
    if verbose:
        for src, (_, log) in results.items():
            print(f"== {src}\n{log}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[results[s][0] for s in SOURCES]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
