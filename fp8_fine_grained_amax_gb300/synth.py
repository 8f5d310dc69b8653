"""Seeded synthetic inputs shaped like the LLM tensors the method quantises.

This module draws random numbers and rounds them to BF16; it holds none of the
quantisation or GEMM arithmetic.  Both the CUDA path's tests/benchmark and the
CPU oracle take their inputs from here, so the two always see identical bytes.

Recipe (stated once, used everywhere):
  * Generator: numpy ``PCG64`` seeded by ``SeedSequence([seed, stream, chunk])``
    where ``stream`` is a fixed id per named tensor and the tensor is drawn in
    chunks of ``CHUNK`` elements (so any prefix of rows is reproducible and
    large tensors never need a full-size float temporary).
  * Values: ``std * standard_normal`` in float32; with outliers, each element
    independently (probability ``outlier_frac``, by a uniform draw from the same
    chunk's stream) is multiplied by ``outlier_mult``; then rounded to BF16,
    nearest-even.
  * MoE routing: expert probabilities ``p ~ Dirichlet(alpha * 1_G)``, token
    counts ``~ Multinomial(n_tokens, p)`` (top-1, tokens sorted by expert), as
    ``int32`` offsets ``[0, c0, c0+c1, ..., n_tokens]``.

BF16 tensors are returned as numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 20


def stream_id(name: str) -> int:
    """Stable 32-bit id of a named tensor (crc32 of its name)."""
    return zlib.crc32(name.encode("utf-8")) & 0xFFFFFFFF


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns, round to nearest even (finite inputs)."""
    u = x.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_bf16(shape, std: float, seed: int, name: str,
                outlier_frac: float = 0.0, outlier_mult: float = 100.0) -> np.ndarray:
    """BF16 tensor of ``std * N(0,1)`` with optional multiplied outliers."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, np.uint16)
    sid = stream_id(name)

    def fill(ci: int) -> None:
        lo = ci * CHUNK
        hi = min(n, lo + CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, sid, ci])))
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        v *= np.float32(std)
        if outlier_frac > 0.0:
            u = rng.random(hi - lo, dtype=np.float32)
            v[u < np.float32(outlier_frac)] *= np.float32(outlier_mult)
        out[lo:hi] = _round_bf16(v)

    # chunks are seeded independently, so drawing them on several threads
    # (numpy releases the GIL while it fills and rounds) gives the same bytes
    n_chunks = (n + CHUNK - 1) // CHUNK
    if n_chunks <= 2:
        for ci in range(n_chunks):
            fill(ci)
    else:
        with ThreadPoolExecutor(min(n_chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def moe_offsets(n_tokens: int, n_experts: int, alpha: float, seed: int,
                name: str = "moe.routing") -> np.ndarray:
    """Top-1 routing: int32 offsets [G+1] of tokens sorted by expert."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream_id(name)])))
    p = rng.dirichlet(np.full(n_experts, alpha))
    counts = rng.multinomial(n_tokens, p)
    offs = np.zeros(n_experts + 1, np.int32)
    offs[1:] = np.cumsum(counts)
    return offs


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------- workloads
# The five workloads the path is measured and checked on (tokens x channels,
# BF16 inputs, seed 0).  Activations ~N(0,1) with 0.1% entries x100; weights
# ~N(0,0.02); the backward's output gradient ~N(0,1e-3).
OUTLIER_FRAC = 1e-3
OUTLIER_MULT = 100.0

WORKLOADS = {
    "tiny_fprop": dict(M=256, N=256, K=512),
    "fprop_4096x7168x7168": dict(M=4096, N=7168, K=7168),
    "linear_bwd_T8192": dict(T=8192, d_in=7168, d_out=2048),
    "moe_fprop_16x16384": dict(G=16, tokens=16384, d_model=7168, d_ff=4096,
                               d_down_in=2048, alpha=0.5),
    "sweep": dict(act_T=(4096, 16384, 65536), act_C=7168,
                  gemm_sizes=(2048, 4096, 8192, 16384)),
}


def activation(M: int, K: int, seed: int = 0, name: str = "X") -> np.ndarray:
    return normal_bf16((M, K), 1.0, seed, name, OUTLIER_FRAC, OUTLIER_MULT)


def weight(N: int, K: int, seed: int = 0, name: str = "W") -> np.ndarray:
    return normal_bf16((N, K), 0.02, seed, name)
