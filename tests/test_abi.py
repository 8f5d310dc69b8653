"""The C-ABI library builds, loads without a GPU and exports every entry point
declared in include/fp8q.h; the binding covers exactly those names."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "fp8q.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8q_[a-zA-Z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from fp8_fine_grained_amax_gb300.build import build_library
    build_library()
    from fp8_fine_grained_amax_gb300 import binding
    return binding.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "fp8q_gemm" in names and "fp8q_quant_act_T" in names
    for n in names:
        assert hasattr(lib, n), n


def test_binding_signatures_cover_header(lib):
    from fp8_fine_grained_amax_gb300 import binding
    assert sorted(binding.SIGNATURES) == _declared()


def test_host_only_calls(lib):
    from fp8_fine_grained_amax_gb300 import binding
    assert binding.fp8q_version() == 100
    assert "timed out" in binding.status_string(binding.FP8Q_ERR_TIMEOUT)
    # argument checks happen before any device work, so they run without a GPU
    assert lib.fp8q_quant_act(None, 4, 100, 100, None, 100, None, 4, 0, None) == \
        binding.FP8Q_ERR_SHAPE
    assert lib.fp8q_quant_act(None, 4, 128, 128, None, 128, None, 4, 9, None) == \
        binding.FP8Q_ERR_INVALID
    assert lib.fp8q_gemm(None, 128, None, 4, None, 128, None, 1, 7, None, 4, 0, 4, 4, 128,
                         None) == binding.FP8Q_ERR_INVALID
    assert lib.fp8q_grouped_gemm(None, 128, None, 4, None, 128, None, None, 0, None, 4, 0,
                                 4, 4, 128, None) == binding.FP8Q_ERR_SHAPE
    # zero-sized work is a successful no-op
    assert lib.fp8q_quant_act(None, 0, 128, 128, None, 128, None, 0, 0, None) == binding.FP8Q_OK


def test_tile_coordinate_limits_checked_on_the_host(lib):
    # the persistent quantisers step 32-bit tile coordinates: shapes past that
    # range are rejected before any pointer or device is touched
    from fp8_fine_grained_amax_gb300 import binding
    big = 1 << 31  # a multiple of 128 just past INT32_MAX
    assert lib.fp8q_requant_act_T(None, 128, big, big, None, 128, None, 128, None, big, 0,
                                  None) == binding.FP8Q_ERR_SHAPE
    assert lib.fp8q_requant_act_T(None, 128 * 65536, 128, 128, None, 128 * 65536, None,
                                  128 * 65536, None, 128, 0, None) == binding.FP8Q_ERR_SHAPE
    assert lib.fp8q_quant_act_T(None, 128, big, big, None, 128, None, big, None, 0, None, 0, 0,
                                None) == binding.FP8Q_ERR_SHAPE
    # one size smaller gets past the shape checks (to the pointer checks)
    assert lib.fp8q_requant_act_T(None, 128, big - 128, big - 128, None, 128, None, 128, None,
                                  big - 128, 0, None) == binding.FP8Q_ERR_INVALID
    assert lib.fp8q_quant_act_T(None, 128, big - 128, big - 128, None, 128, None, big - 128, None,
                                0, None, 0, 0, None) == binding.FP8Q_ERR_INVALID


def test_package_has_no_cpu_path():
    # the product package must not import the oracle
    pkg = os.path.join(ROOT, "fp8_fine_grained_amax_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
