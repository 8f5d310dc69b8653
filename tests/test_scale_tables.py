"""The identity behind the table-driven FP32 scales of the 128x1 quantiser.

For a BF16 max-abs a = (1 + m/128) * 2^E (E >= -116 after the 2^-116 floor),
fl(a / 448) = fl(M / 448) * 2^E and fl(448 / a) = fl(448 / M) * 2^-E with
M = 1 + m/128, for every one of the 128 mantissas and every exponent, in IEEE
single precision (numpy float32 division rounds to nearest, as __fdiv_rn
does).  The kernel adds E to the exponent field of the tabulated quotients;
this checks that the result is the same number, so that the scales equal
the oracle's single divisions (the GPU test of every BF16 max-abs checks the
kernel itself)."""
import numpy as np


def test_power_of_two_scaling_commutes_with_the_division():
    m = np.arange(128, dtype=np.float32)
    M = np.float32(1) + m * np.float32(2.0 ** -7)
    c = np.float32(448)
    t_s = (M / c).astype(np.float32)
    t_inv = (c / M).astype(np.float32)
    with np.errstate(over="raise", under="raise"):
        for E in range(-116, 128):
            a = (M * np.float32(2.0 ** E)).astype(np.float32)
            s = (a / c).astype(np.float32)
            inv = (c / a).astype(np.float32)
            # adding E to the exponent field = multiplying by 2^E exactly
            s_tab = (t_s.view(np.uint32) + np.uint32((E * (1 << 23)) % (1 << 32))).view(np.float32)
            inv_tab = (t_inv.view(np.uint32) - np.uint32((E * (1 << 23)) % (1 << 32))).view(np.float32)
            assert np.array_equal(s.view(np.uint32), s_tab.view(np.uint32)), E
            assert np.array_equal(inv.view(np.uint32), inv_tab.view(np.uint32)), E
            # every result is a normal number
            assert np.all(np.abs(s) >= np.float32(2.0 ** -126))
            assert np.all(np.abs(inv) >= np.float32(2.0 ** -126))
