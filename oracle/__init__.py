"""CPU oracle for fine-grained FP8 quantisation and the per-group-scaled GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``fp8_fine_grained_amax_gb300``) never imports it and shares no
code with it: the arithmetic lives in ``fp8q_oracle.c`` (plain C, IEEE single
and double precision, no FMA contraction), written from the pages' statement of
the method; this module only marshals numpy arrays in and out of it.

Arrays:
  * BF16 tensors are numpy ``uint16`` arrays of raw BF16 bit patterns.
  * E4M3 tensors are numpy ``uint8`` arrays of raw codes.
  * Scales are ``float32``; GEMM results are ``float64``.

Every function states the layout it returns; see the C file for the citations
and for the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8q_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCALE_FP32 = 0
SCALE_POW2 = 1

BSCALE_BLOCK = 0      # sb[nb][kb]
BSCALE_BLOCK_T = 1    # sb[kb][nb]
BSCALE_ROW = 2        # sb[kb][n]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            INT = ctypes.c_int
            L.oracle_e4m3_decode.restype = ctypes.c_double
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode_array.restype = None
            L.oracle_e4m3_encode_array.argtypes = [P, I64, P]
            L.oracle_group_scale.restype = None
            L.oracle_group_scale.argtypes = [ctypes.c_float, INT, P, P]
            L.oracle_quant_act.restype = None
            L.oracle_quant_act.argtypes = [P, I64, I64, I64, P, I64, P, I64, INT]
            L.oracle_quant_act_T.restype = None
            L.oracle_quant_act_T.argtypes = [P, I64, I64, I64, P, I64, P, I64, INT]
            L.oracle_quant_weight.restype = None
            L.oracle_quant_weight.argtypes = [P, I64, I64, I64, P, I64, P, INT]
            L.oracle_gemm_rows.restype = None
            L.oracle_gemm_rows.argtypes = [P, I64, P, I64, P, I64, P, INT, I64,
                                           I64, I64, P, I64, P, P]
            L.oracle_grouped_gemm_rows.restype = None
            L.oracle_grouped_gemm_rows.argtypes = [P, I64, P, I64, P, P, P, INT,
                                                   I64, I64, P, I64, P, P]
            L.oracle_bf16_gemm_rows.restype = None
            L.oracle_bf16_gemm_rows.argtypes = [P, I64, P, I64, I64, I64, P, I64, P]
            L.oracle_requant_act_T.restype = None
            L.oracle_requant_act_T.argtypes = [P, I64, I64, I64, P, I64, P, I64, P, I64, INT]
            L.oracle_quant_tensor.restype = None
            L.oracle_quant_tensor.argtypes = [P, I64, I64, I64, P, I64, P, INT]
            L.oracle_num_threads.restype = INT
            L.oracle_num_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    """Threads the oracle's parallel-for uses (ORACLE_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- E4M3 codec
def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    L = _load()
    c = np.asarray(codes, dtype=np.uint8)
    lut = np.array([L.oracle_e4m3_decode(v) for v in range(256)], dtype=np.float64)
    return lut[c]


def e4m3_encode_scalar(v: float) -> int:
    return int(_load().oracle_e4m3_encode(ctypes.c_float(v)))


def e4m3_encode(x) -> np.ndarray:
    """float32 array -> E4M3 codes (round to nearest even, saturate at 448)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(q))
    return q


def group_scale(amax: float, pow2: bool):
    """(s, inv) of one group with the given max-abs value, as float32."""
    s = np.zeros(1, np.float32)
    inv = np.zeros(1, np.float32)
    _load().oracle_group_scale(ctypes.c_float(amax), int(bool(pow2)), _ptr(s), _ptr(inv))
    return s[0], inv[0]


# ---------------------------------------------------------------- quantisers
def quant_act(x_bf16: np.ndarray, pow2: bool = False):
    """1x128 tiles.  x [M][K] (BF16 bits) -> q [M][K] uint8, sa [K/128][M] f32."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    assert K % 128 == 0
    q = np.empty((M, K), np.uint8)
    sa = np.empty((K // 128, M), np.float32)
    _load().oracle_quant_act(_ptr(x), M, K, K, _ptr(q), K, _ptr(sa), M, int(bool(pow2)))
    return q, sa


def quant_act_T(x_bf16: np.ndarray, pow2: bool = False):
    """128x1 tiles.  x [T][C] -> qT [C][T] uint8, sT [T/128][C] f32."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, C = x.shape
    assert T % 128 == 0
    qT = np.empty((C, T), np.uint8)
    sT = np.empty((T // 128, C), np.float32)
    _load().oracle_quant_act_T(_ptr(x), T, C, C, _ptr(qT), T, _ptr(sT), C, int(bool(pow2)))
    return qT, sT


def quant_weight(w_bf16: np.ndarray, pow2: bool = False):
    """128x128 blocks.  w [N][K] -> q [N][K] uint8, sb [ceil(N/128)][K/128] f32."""
    w = np.ascontiguousarray(w_bf16, dtype=np.uint16)
    N, K = w.shape
    assert K % 128 == 0
    q = np.empty((N, K), np.uint8)
    sb = np.empty(((N + 127) // 128, K // 128), np.float32)
    _load().oracle_quant_weight(_ptr(w), N, K, K, _ptr(q), K, _ptr(sb), int(bool(pow2)))
    return q, sb


def quant_tensor(x_bf16: np.ndarray, pow2: bool = False):
    """Per-tensor quantisation (comparison only): x [M][K] -> q [M][K], one f32 scale."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.zeros(1, np.float32)
    _load().oracle_quant_tensor(_ptr(x), M, K, K, _ptr(q), K, _ptr(s), int(bool(pow2)))
    return q, s[0]


def requant_act_T(q, s_rows, pow2: bool = False):
    """128x1 requantisation of FP8-cached 1x128 activations.

    q [T][C] E4M3 codes with 1x128 scales s_rows [C/128][T] -> qT [C][T],
    sT [T/128][C] (each value dequantised by one FP32 multiply first)."""
    q = np.ascontiguousarray(q, np.uint8)
    s_rows = np.ascontiguousarray(s_rows, np.float32)
    T, C = q.shape
    assert T % 128 == 0 and C % 128 == 0 and s_rows.shape == (C // 128, T)
    qT = np.empty((C, T), np.uint8)
    sT = np.empty((T // 128, C), np.float32)
    _load().oracle_requant_act_T(_ptr(q), T, C, C, _ptr(s_rows), T, _ptr(qT), T, _ptr(sT), C,
                                 int(bool(pow2)))
    return qT, sT


# ---------------------------------------------------------------- GEMMs
def gemm_rows(qa, sa, qb, sb, bkind: int, rows=None):
    """Dequantised product in double for the listed rows of A.

    qa [M][K] codes, sa [K/128][M]; qb [N][K] codes; sb laid out per ``bkind``
    (BSCALE_BLOCK: [ceil(N/128)][K/128]; BSCALE_BLOCK_T: [K/128][ceil(N/128)];
    BSCALE_ROW: [K/128][N]).  Returns (C [len(rows)][N], sum_k |a_k b_k|).
    """
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % 128 == 0 and sa.shape == (K // 128, M)
    if rows is None:
        rows = np.arange(M)
    rows = np.ascontiguousarray(rows, np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
    c = np.empty((rows.size, N), np.float64)
    ad = np.empty((rows.size, N), np.float64)
    _load().oracle_gemm_rows(_ptr(qa), K, _ptr(sa), M, _ptr(qb), K, _ptr(sb),
                             int(bkind), sb.shape[1], N, K, _ptr(rows), rows.size,
                             _ptr(c), _ptr(ad))
    return c, ad


def grouped_gemm_rows(qa, sa, qb, sb, offs, rows=None):
    """MoE grouped product: row m uses expert g with offs[g] <= m < offs[g+1].

    qa [M][K], sa [K/128][M]; qb [G][N][K]; sb [G][ceil(N/128)][K/128];
    offs int32 [G+1].  Returns (C [len(rows)][N], sum_k |a_k b_k|).
    """
    qa = np.ascontiguousarray(qa, np.uint8)
    qb = np.ascontiguousarray(qb, np.uint8)
    sa = np.ascontiguousarray(sa, np.float32)
    sb = np.ascontiguousarray(sb, np.float32)
    offs = np.ascontiguousarray(offs, np.int32)
    M, K = qa.shape
    G, N, K2 = qb.shape
    assert K == K2 and offs.shape == (G + 1,)
    assert sb.shape == (G, (N + 127) // 128, K // 128)
    if rows is None:
        rows = np.arange(M)
    rows = np.ascontiguousarray(rows, np.int64)
    c = np.empty((rows.size, N), np.float64)
    ad = np.empty((rows.size, N), np.float64)
    _load().oracle_grouped_gemm_rows(_ptr(qa), K, _ptr(sa), M, _ptr(qb), _ptr(sb),
                                     _ptr(offs), G, N, K, _ptr(rows), rows.size,
                                     _ptr(c), _ptr(ad))
    return c, ad


def bf16_gemm_rows(x_bf16, w_bf16, rows=None):
    """Context only: unquantised x @ w^T in double for the listed rows."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    w = np.ascontiguousarray(w_bf16, np.uint16)
    M, K = x.shape
    N, _ = w.shape
    if rows is None:
        rows = np.arange(M)
    rows = np.ascontiguousarray(rows, np.int64)
    c = np.empty((rows.size, N), np.float64)
    _load().oracle_bf16_gemm_rows(_ptr(x), K, _ptr(w), K, N, K, _ptr(rows), rows.size, _ptr(c))
    return c


# ---------------------------------------------------------------- tolerance
def gemm_tolerance(c_ref: np.ndarray, absdot: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Per-element bound |C - C_ref| <= 2e-4 * sum_k|a_k b_k| (+ half a BF16 ulp).

    The 2e-4 relative bound on the scaled dot-product magnitude is the
    acceptance criterion stated for this path; a BF16 result may in addition
    differ by the half unit in the last place that rounding FP32 to BF16 adds,
    taken at the largest magnitude the FP32 result can have (|C_ref| + bound),
    so that a result rounded across a power of two is still covered.
    """
    tol = 2e-4 * np.asarray(absdot, np.float64)
    if out_bf16:
        tol = tol + 0.5 * bf16_ulp(np.abs(c_ref) + tol)
    return tol


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |v| (8 significant bits; subnormal floor)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(np.int64))
