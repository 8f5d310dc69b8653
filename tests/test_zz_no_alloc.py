"""GPU check of fp8q_quant_tensor_noalloc, the per-tensor quantiser that runs on
the library's fixed per-device scratch instead of a caller workspace.

It is called straight through the C ABI (ctypes on libfp8q) and compared with
fp8q_quant_tensor, the workspace form, on two calls in a row with different
inputs: the second call must not see anything the first left in the shared
scratch.  The file is named so that it is collected last; it also passes alone
in a fresh process (its fixture builds and loads the library itself).
"""
import ctypes

import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import assert_bytes_equal, assert_scales_equal, bf16_to_torch, f32, u8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
B = pytest.importorskip("fp8_fine_grained_amax_gb300.binding")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_fine_grained_amax_gb300.build import build_library
    build_library()
    lib = B.load_library()
    yield lib
    assert B.fp8q_sync_status() == 0


def _noalloc(lib, x, q, s, mode):
    M, K = x.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fp8q_quant_tensor_noalloc(
        ctypes.c_void_p(x.data_ptr()), M, K, x.stride(0), ctypes.c_void_p(q.data_ptr()),
        q.stride(0), ctypes.c_void_p(s.data_ptr()), mode, stream)


@pytest.mark.parametrize("mode", [0, 1])   # FP8Q_SCALE_FP32, FP8Q_SCALE_POW2
def test_noalloc_matches_workspace_form_twice(lib, mode):
    # two calls in a row on different inputs: a large one that fills most of
    # the scratch, then a small one that reads only its own partials
    for (M, K, seed) in [(4096, 7168, 701), (300, 1024, 702)]:
        x = bf16_to_torch(synth.activation(M, K, seed=seed))
        q = torch.full((M, K), 0xCD, dtype=torch.uint8, device="cuda")
        s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(lib, x, q, s, mode) == 0
        q_ref, s_ref = B.fp8q_quant_tensor(x, scale_mode=mode)
        torch.cuda.synchronize()
        assert_bytes_equal(u8(q), u8(q_ref), f"codes M={M}")
        assert_scales_equal(f32(s), f32(s_ref), f"scale M={M}")


def test_noalloc_row_limit(lib):
    K = 128
    s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    x = torch.zeros((65537, K), dtype=torch.bfloat16, device="cuda")
    q = torch.full((65537, K), 0xCD, dtype=torch.uint8, device="cuda")
    assert _noalloc(lib, x, q, s, 0) == B.FP8Q_ERR_SHAPE
    torch.cuda.synchronize()
    assert np.all(u8(q) == 0xCD) and f32(s)[0] == -1.0, "a rejected call wrote its outputs"
    # the largest accepted size: all-zero input quantises to zero codes
    assert _noalloc(lib, x[:65536], q[:65536], s, 0) == 0
    q_ref, s_ref = B.fp8q_quant_tensor(x[:65536], scale_mode=0)
    torch.cuda.synchronize()
    assert np.all(u8(q[:65536]) == 0)
    assert_bytes_equal(u8(q[:65536]), u8(q_ref), "codes M=65536")
    assert_scales_equal(f32(s), f32(s_ref), "scale M=65536")


@pytest.mark.parametrize("mode", [0, 1])   # FP8Q_SCALE_FP32, FP8Q_SCALE_POW2
@pytest.mark.parametrize("M,K", [(0, 256), (300, 0)])
def test_noalloc_empty_input_gives_the_zero_tensor_scale(lib, oracle, M, K, mode):
    # a call on real data first leaves nonzero partials in the shared scratch;
    # an empty input (no rows, or rows of no columns) must still come out with
    # the scale of an all-zero tensor, a = 2^-116: its own first pass writes
    # every partial its second pass reads, so nothing stale is picked up
    x0 = bf16_to_torch(synth.activation(4096, 1024, seed=703))
    q0 = torch.empty((4096, 1024), dtype=torch.uint8, device="cuda")
    s0 = torch.empty((1,), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, x0, q0, s0, mode) == 0
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    assert _noalloc(lib, x, q, s, mode) == 0
    _, s_ws = B.fp8q_quant_tensor(x, scale_mode=mode)
    _, s_zero = oracle.quant_tensor(np.zeros((1, 128), np.uint16), mode == 1)
    torch.cuda.synchronize()
    assert f32(s0)[0] > 0 and f32(s0)[0] != np.float32(s_zero), "first call gave a zero scale"
    assert_scales_equal(f32(s), f32(s_ws), f"scale M={M} K={K} (workspace form)")
    assert_scales_equal(f32(s), np.array([s_zero], np.float32), f"scale M={M} K={K} (oracle)")
