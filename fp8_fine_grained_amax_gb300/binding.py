"""Thin ctypes binding of libfp8q (include/fp8q.h), same names as the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of libfp8q.so.  Tensors are torch CUDA tensors (torch supplies device
memory and the current stream); outputs that are not passed in are allocated
with torch.  E4M3 tensors are torch.uint8 (raw codes; ``.view(torch.float8_e4m3fn)``
gives the FP8 dtype).  A failing call raises FP8QError; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8q.so")

FP8Q_OK = 0
FP8Q_ERR_INVALID = 1
FP8Q_ERR_SHAPE = 2
FP8Q_ERR_ALIGN = 3
FP8Q_ERR_UNSUPPORTED = 4
FP8Q_ERR_CUDA = 5
FP8Q_ERR_TIMEOUT = 6

FP8Q_SCALE_FP32 = 0
FP8Q_SCALE_POW2 = 1
FP8Q_OUT_BF16 = 0
FP8Q_OUT_FP32 = 1
FP8Q_BSCALE_BLOCK = 0
FP8Q_BSCALE_BLOCK_T = 1
FP8Q_BSCALE_ROW = 2

# name -> (restype, argtypes) for every entry point declared in include/fp8q.h
_P, _I64, _INT, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
SIGNATURES = {
    "fp8q_quant_act": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _INT, _P]),
    "fp8q_quant_act_T": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64,
                                _INT, _P]),
    "fp8q_quant_weight": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P]),
    "fp8q_requant_act_T": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P]),
    "fp8q_quant_tensor_workspace_bytes": (_I64, [_I64, _I64]),
    "fp8q_quant_tensor": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _P, _I64, _INT, _P]),
    "fp8q_quant_tensor_noalloc": (_INT, [_P, _I64, _I64, _I64, _P, _I64, _P, _INT, _P]),
    "fp8q_gemm": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P, _I64, _INT, _I64,
                         _I64, _I64, _P]),
    "fp8q_gemm_accumulate": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P, _I64, _I64,
                                    _I64, _I64, _P]),
    "fp8q_gemm_pow2": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P, _I64, _INT, _I64,
                         _I64, _I64, _P]),
    "fp8q_gemm_pow2_accumulate": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _I64, _INT, _P, _I64, _I64,
                                    _I64, _I64, _P]),
    "fp8q_grouped_gemm": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _INT, _P, _I64, _INT,
                                 _I64, _I64, _I64, _P]),
    "fp8q_grouped_gemm_pow2": (_INT, [_P, _I64, _P, _I64, _P, _I64, _P, _P, _INT, _P, _I64, _INT,
                                      _I64, _I64, _I64, _P]),
    "fp8q_cast_e4m3": (_INT, [_P, _I64, _P, _P]),
    "fp8q_sync_status": (_INT, [_P]),
    "fp8q_set_wait_timeout_ns": (None, [_U64]),
    "fp8q_selftest_wait_timeout": (_INT, [_U64, _P]),
    "fp8q_status_string": (ctypes.c_char_p, [_INT]),
    "fp8q_version": (_INT, []),
}

_lib = None
_lock = threading.Lock()


class FP8QError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_string(status)} (status {status})")


def load_library(path: str | None = None):
    """Load libfp8q.so (built by fp8_fine_grained_amax_gb300.build).  Raises if missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libfp8q.so not found at {p}: build it with "
                    "`python -m fp8_fine_grained_amax_gb300.build` (no CPU fallback exists)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().fp8q_status_string(int(status)).decode()


def _check(status: int, call: str) -> None:
    if status != FP8Q_OK:
        raise FP8QError(status, call)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# torch's handle of the current stream without building a Stream object (a
# few microseconds per call otherwise); torch.cuda.current_stream() if absent
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None:
            return ctypes.c_void_p(_raw_stream(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _rows_ld(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with a contiguous last dimension")
    return t.stride(0)


def fp8q_quant_act(x, *, scale_mode=FP8Q_SCALE_FP32, q=None, sa=None, stream=None):
    """1x128 quantisation of BF16 x [M][K] -> (q uint8 [M][K], sa f32 [K/128][M])."""
    M, K = x.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if sa is None:
        sa = torch.empty((K // 128, M), dtype=torch.float32, device=x.device)
    _check(load_library().fp8q_quant_act(
        _ptr(x), M, K, _rows_ld(x, "x"), _ptr(q), _rows_ld(q, "q"), _ptr(sa),
        _rows_ld(sa, "sa") if sa.numel() else M, scale_mode, _stream(stream)), "fp8q_quant_act")
    return q, sa


def fp8q_quant_act_T(x, *, scale_mode=FP8Q_SCALE_FP32, with_rows=False, qT=None, sT=None,
                     q_rows=None, s_rows=None, stream=None):
    """128x1 quantisation of BF16 x [T][C] -> (qT uint8 [C][T], sT f32 [T/128][C]),
    plus (q_rows [T][C], s_rows [C/128][T]) from the same read when with_rows."""
    T, C = x.shape
    dev = x.device
    if qT is None:
        qT = torch.empty((C, T), dtype=torch.uint8, device=dev)
    if sT is None:
        sT = torch.empty((T // 128, C), dtype=torch.float32, device=dev)
    if with_rows:
        if q_rows is None:
            q_rows = torch.empty((T, C), dtype=torch.uint8, device=dev)
        if s_rows is None:
            s_rows = torch.empty((C // 128, T), dtype=torch.float32, device=dev)
    _check(load_library().fp8q_quant_act_T(
        _ptr(x), T, C, _rows_ld(x, "x"), _ptr(qT), _rows_ld(qT, "qT") if qT.numel() else T,
        _ptr(sT), _rows_ld(sT, "sT") if sT.numel() else C,
        _ptr(q_rows) if with_rows else None, _rows_ld(q_rows, "q_rows") if with_rows else 0,
        _ptr(s_rows) if with_rows else None,
        (_rows_ld(s_rows, "s_rows") if s_rows.numel() else T) if with_rows else 0,
        scale_mode, _stream(stream)), "fp8q_quant_act_T")
    if with_rows:
        return qT, sT, q_rows, s_rows
    return qT, sT


def fp8q_requant_act_T(q, s_rows, *, scale_mode=FP8Q_SCALE_FP32, qT=None, sT=None, stream=None):
    """128x1 requantisation of FP8-cached 1x128 codes q uint8 [T][C] with scales
    s_rows f32 [C/128][T] -> (qT uint8 [C][T], sT f32 [T/128][C])."""
    T, C = q.shape
    if qT is None:
        qT = torch.empty((C, T), dtype=torch.uint8, device=q.device)
    if sT is None:
        sT = torch.empty((T // 128, C), dtype=torch.float32, device=q.device)
    _check(load_library().fp8q_requant_act_T(
        _ptr(q), T, C, _rows_ld(q, "q"), _ptr(s_rows),
        _rows_ld(s_rows, "s_rows") if s_rows.numel() else T, _ptr(qT),
        _rows_ld(qT, "qT") if qT.numel() else T, _ptr(sT), _rows_ld(sT, "sT") if sT.numel() else C,
        scale_mode, _stream(stream)), "fp8q_requant_act_T")
    return qT, sT


def fp8q_quant_weight(w, *, scale_mode=FP8Q_SCALE_FP32, with_transpose=False, q=None, qT=None,
                      sb=None, stream=None):
    """128x128 quantisation of BF16 w [N][K] -> (q uint8 [N][K], sb f32 [ceil(N/128)][K/128]),
    plus qT uint8 [K][N] when with_transpose (returned as a third item)."""
    N, K = w.shape
    dev = w.device
    if q is None:
        q = torch.empty((N, K), dtype=torch.uint8, device=dev)
    if sb is None:
        sb = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
    if with_transpose and qT is None:
        qT = torch.empty((K, N), dtype=torch.uint8, device=dev)
    _check(load_library().fp8q_quant_weight(
        _ptr(w), N, K, _rows_ld(w, "w"), _ptr(q), _rows_ld(q, "q"),
        _ptr(qT) if with_transpose else None,
        (_rows_ld(qT, "qT") if qT.numel() else N) if with_transpose else 0,
        _ptr(sb), _rows_ld(sb, "sb") if sb.numel() else K // 128, scale_mode, _stream(stream)),
        "fp8q_quant_weight")
    if with_transpose:
        return q, sb, qT
    return q, sb


def fp8q_quant_tensor_workspace_bytes(M: int, K: int) -> int:
    return int(load_library().fp8q_quant_tensor_workspace_bytes(M, K))


def fp8q_quant_tensor(x, *, scale_mode=FP8Q_SCALE_FP32, q=None, s=None, workspace=None,
                      stream=None):
    """Per-tensor quantisation (comparison path): x BF16 [M][K] -> (q uint8 [M][K],
    s f32 [1]).  A workspace tensor is allocated with torch when not given."""
    M, K = x.shape
    dev = x.device
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    if s is None:
        s = torch.empty((1,), dtype=torch.float32, device=dev)
    nbytes = fp8q_quant_tensor_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 4),), dtype=torch.uint8, device=dev)
    _check(load_library().fp8q_quant_tensor(
        _ptr(x), M, K, _rows_ld(x, "x"), _ptr(q), _rows_ld(q, "q"), _ptr(s), _ptr(workspace),
        workspace.numel() * workspace.element_size(), scale_mode, _stream(stream)),
        "fp8q_quant_tensor")
    return q, s


def fp8q_quant_tensor_noalloc(x, q, s, *, scale_mode=FP8Q_SCALE_FP32, stream=None):
    """fp8q_quant_tensor on the library's fixed per-device scratch: x BF16 [M][K]
    (M <= 65536) into the caller's q uint8 [M][K] and s f32 [1].  Allocates
    nothing; calls that overlap on the GPU share the scratch and race."""
    M, K = x.shape
    _check(load_library().fp8q_quant_tensor_noalloc(
        _ptr(x), M, K, _rows_ld(x, "x"), _ptr(q), _rows_ld(q, "q"), _ptr(s), scale_mode,
        _stream(stream)), "fp8q_quant_tensor_noalloc")
    return q, s


def fp8q_gemm(a, sa, b, sb, *, bscale_kind=FP8Q_BSCALE_BLOCK, out_dtype=FP8Q_OUT_BF16, c=None,
              stream=None, _entry="fp8q_gemm"):
    """C [M][N] = per-128-K-group scaled a [M][K] x b [N][K]^T (E4M3 codes)."""
    M, K = a.shape
    N = b.shape[0]
    if c is None:
        dt = torch.bfloat16 if out_dtype == FP8Q_OUT_BF16 else torch.float32
        c = torch.empty((M, N), dtype=dt, device=a.device)
    ld_sa = _rows_ld(sa, "sa") if sa.numel() else M
    ld_sb = _rows_ld(sb, "sb") if sb.numel() else 1
    _check(getattr(load_library(), _entry)(
        _ptr(a), _rows_ld(a, "a") if a.numel() else K, _ptr(sa), ld_sa, _ptr(b),
        _rows_ld(b, "b") if b.numel() else K, _ptr(sb), ld_sb, bscale_kind, _ptr(c),
        _rows_ld(c, "c"), out_dtype, M, N, K, _stream(stream)), _entry)
    return c


def fp8q_gemm_pow2(a, sa, b, sb, *, bscale_kind=FP8Q_BSCALE_BLOCK, out_dtype=FP8Q_OUT_BF16,
                   c=None, stream=None):
    """fp8q_gemm for power-of-two scales (FP8Q_SCALE_POW2 quantisers) on the
    block-scaled MMA; same arguments and result."""
    return fp8q_gemm(a, sa, b, sb, bscale_kind=bscale_kind, out_dtype=out_dtype, c=c,
                     stream=stream, _entry="fp8q_gemm_pow2")


def fp8q_gemm_accumulate(a, sa, b, sb, c, *, bscale_kind=FP8Q_BSCALE_BLOCK, stream=None,
                         _entry="fp8q_gemm_accumulate"):
    """c (FP32 [M][N]) += per-128-K-group scaled a [M][K] x b [N][K]^T."""
    M, K = a.shape
    N = b.shape[0]
    if c.dtype != torch.float32 or tuple(c.shape) != (M, N):
        raise ValueError("c must be an FP32 [M][N] tensor")
    ld_sa = _rows_ld(sa, "sa") if sa.numel() else M
    ld_sb = _rows_ld(sb, "sb") if sb.numel() else 1
    _check(getattr(load_library(), _entry)(
        _ptr(a), _rows_ld(a, "a") if a.numel() else K, _ptr(sa), ld_sa, _ptr(b),
        _rows_ld(b, "b") if b.numel() else K, _ptr(sb), ld_sb, bscale_kind, _ptr(c),
        _rows_ld(c, "c"), M, N, K, _stream(stream)), _entry)
    return c


def fp8q_gemm_pow2_accumulate(a, sa, b, sb, c, *, bscale_kind=FP8Q_BSCALE_BLOCK, stream=None):
    """c (FP32 [M][N]) += the fp8q_gemm_pow2 product."""
    return fp8q_gemm_accumulate(a, sa, b, sb, c, bscale_kind=bscale_kind, stream=stream,
                                _entry="fp8q_gemm_pow2_accumulate")


def fp8q_grouped_gemm(a, sa, b, sb, offs, *, out_dtype=FP8Q_OUT_BF16, c=None, stream=None,
                      _entry="fp8q_grouped_gemm"):
    """MoE grouped GEMM: a [M][K], b [G][N][K], sb [G][ceil(N/128)][K/128],
    offs int32 [G+1] on the device.  Rows outside [offs[0], offs[G]) are left as is."""
    M, K = a.shape
    G, N, _ = b.shape
    if c is None:
        dt = torch.bfloat16 if out_dtype == FP8Q_OUT_BF16 else torch.float32
        c = torch.empty((M, N), dtype=dt, device=a.device)
    if b.stride(2) != 1 or b.stride(0) != N * b.stride(1):
        raise ValueError("b must be [G][N][ldb] with experts packed back to back")
    _check(getattr(load_library(), _entry)(
        _ptr(a), _rows_ld(a, "a") if a.numel() else K, _ptr(sa),
        _rows_ld(sa, "sa") if sa.numel() else M, _ptr(b), b.stride(1), _ptr(sb), _ptr(offs), G,
        _ptr(c), _rows_ld(c, "c"), out_dtype, M, N, K, _stream(stream)), _entry)
    return c


def fp8q_grouped_gemm_pow2(a, sa, b, sb, offs, *, out_dtype=FP8Q_OUT_BF16, c=None, stream=None):
    """fp8q_grouped_gemm for power-of-two scales on the block-scaled MMA."""
    return fp8q_grouped_gemm(a, sa, b, sb, offs, out_dtype=out_dtype, c=c, stream=stream,
                             _entry="fp8q_grouped_gemm_pow2")


def fp8q_cast_e4m3(x, *, q=None, stream=None):
    """FP32 -> E4M3 codes (RNE, saturate), no scaling."""
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(load_library().fp8q_cast_e4m3(_ptr(x), x.numel(), _ptr(q), _stream(stream)),
           "fp8q_cast_e4m3")
    return q


def fp8q_sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load_library().fp8q_sync_status(_stream(stream)))


def fp8q_set_wait_timeout_ns(ns: int) -> None:
    load_library().fp8q_set_wait_timeout_ns(int(ns))


def fp8q_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(load_library().fp8q_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "fp8q_selftest_wait_timeout")


def fp8q_version() -> int:
    return int(load_library().fp8q_version())
