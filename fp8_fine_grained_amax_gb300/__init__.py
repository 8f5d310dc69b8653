"""GB300-native fine-grained FP8 quantisation and per-group-scaled FP8 GEMM.

The product path is libfp8q.so (C ABI in include/fp8q.h, CUDA kernels for
sm_103a in csrc/); ``binding`` exposes it to Python with the same names.
``synth`` generates the seeded synthetic workloads.  Importing the package
does not load the library; the first call does, and fails loudly if the
library has not been built (there is no CPU fallback).
"""
from .binding import (  # noqa: F401
    FP8Q_BSCALE_BLOCK, FP8Q_BSCALE_BLOCK_T, FP8Q_BSCALE_ROW, FP8Q_OUT_BF16, FP8Q_OUT_FP32,
    FP8Q_SCALE_FP32, FP8Q_SCALE_POW2, FP8QError, fp8q_cast_e4m3, fp8q_gemm, fp8q_gemm_accumulate, fp8q_gemm_pow2, fp8q_gemm_pow2_accumulate, fp8q_grouped_gemm, fp8q_grouped_gemm_pow2,
    fp8q_quant_act, fp8q_quant_act_T, fp8q_quant_tensor, fp8q_quant_tensor_noalloc, fp8q_quant_weight, fp8q_requant_act_T, fp8q_selftest_wait_timeout,
    fp8q_set_wait_timeout_ns, fp8q_sync_status, fp8q_version, load_library, status_string)
