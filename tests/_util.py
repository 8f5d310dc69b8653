"""Helpers shared by the tests: moving seeded numpy inputs to the GPU and back."""
import numpy as np
import torch


def bf16_to_torch(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy uint16 BF16 bit patterns -> torch bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint8)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float32)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:5].tolist()}: " \
        f"got {got[tuple(bad[0])]!r} want {want[tuple(bad[0])]!r}"


def assert_scales_equal(got: np.ndarray, want: np.ndarray, what: str):
    # bit-exact comparison of FP32 scales
    assert_bytes_equal(np.ascontiguousarray(got).view(np.uint32),
                       np.ascontiguousarray(want).view(np.uint32), what)


def assert_within_tolerance(got: np.ndarray, ref: np.ndarray, tol: np.ndarray, what: str):
    err = np.abs(got.astype(np.float64) - ref)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, f"{what}: {len(bad)} of {err.size} outside tolerance; first " \
        f"{bad[:3].tolist()}: got {got[tuple(bad[0])]} ref {ref[tuple(bad[0])]} " \
        f"tol {tol[tuple(bad[0])]}; max err/tol {np.max(err / np.maximum(tol, 1e-300)):.3g}"
