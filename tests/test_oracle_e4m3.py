"""Pins for the oracle's E4M3 codec (CPU only).

The pages fix the format only by name (E4M3, used for every tensor in the
"FP8 mixed precision" post of Data Science by ODS.ai) and the target of the
scaling (the largest finite FP8 value, "Deepseek - Not For everyone",
paragraph 4).  The codec is therefore pinned against the OCP 8-bit floating
point definition of E4M3 (bias 7, no infinities, one NaN mantissa pattern,
largest finite 448) through facts a wrong implementation would break:
published spot values, the shape of the value set, and an independent
nearest-value search for the encoder.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.fixture(scope="module")
def table(oracle):
    return oracle.e4m3_decode(np.arange(256, dtype=np.uint8))


def test_decode_spot_values(table):
    # Values the OCP definition lists for E4M3.
    assert table[0x00] == 0.0 and not math.copysign(1, table[0x00]) < 0
    assert table[0x80] == 0.0 and math.copysign(1, table[0x80]) < 0
    assert table[0x01] == 2.0 ** -9          # smallest subnormal
    assert table[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert table[0x08] == 2.0 ** -6          # smallest normal
    assert table[0x38] == 1.0
    assert table[0x3F] == 1.875
    assert table[0x40] == 2.0
    assert table[0x70] == 128.0
    assert table[0x77] == 240.0
    assert table[0x7E] == 448.0              # largest finite
    assert table[0xFE] == -448.0
    assert np.isnan(table[0x7F]) and np.isnan(table[0xFF])
    assert np.isnan(table).sum() == 2        # no other NaN, no infinity
    assert np.all(np.isfinite(table[~np.isnan(table)]))


def test_decode_structure(table):
    pos = table[:0x7F]
    assert np.all(np.diff(pos) > 0), "codes 0x00..0x7E must increase strictly"
    # sign bit is a pure sign
    for c in range(0x7F):
        assert table[c | 0x80] == -table[c]
    # subnormals and the first binade share the spacing 2^-9
    assert np.allclose(np.diff(pos[:17]), 2.0 ** -9, rtol=0, atol=0)
    # each normal binade holds 8 evenly spaced values, and the next exponent
    # doubles every value
    for c in range(0x08, 0x77):
        assert table[c + 8] == 2 * table[c]
    for e in range(1, 16):
        b = pos[8 * e: 8 * e + 8] if e < 15 else pos[8 * 15: 8 * 15 + 7]
        d = np.diff(b)
        assert np.all(d == d[0])
        assert b[0] == 2.0 ** (e - 7)


def _brute_encode(oracle, x):
    """Nearest E4M3 value by search over the value set; ties -> even code.

    Independent of the oracle's encoder (which scales by the grid spacing and
    calls rint); it only uses the decode table pinned above.
    """
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    x = np.asarray(x, np.float32)
    a = np.abs(x.astype(np.float64))
    hi = np.clip(np.searchsorted(mags, a, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    dlo = a - mags[lo]
    dhi = mags[hi] - a
    code = np.where(dlo < dhi, lo, hi)
    tie = dlo == dhi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a >= 448.0, 0x7E, code)
    code = code.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def test_encode_round_trip(oracle, table):
    for c in range(256):
        if np.isnan(table[c]):
            continue
        assert oracle.e4m3_encode_scalar(float(table[c])) == c


def test_encode_midpoints_ties_to_even(oracle, table):
    pos = table[:0x7F]
    for c in range(0x7E):
        mid = np.float32((pos[c] + pos[c + 1]) / 2)  # exact: <= 5 significant bits
        assert float(mid) == (pos[c] + pos[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode_scalar(float(mid)) == even
        assert oracle.e4m3_encode_scalar(float(np.nextafter(mid, np.float32(1e9)))) == c + 1
        assert oracle.e4m3_encode_scalar(float(np.nextafter(mid, np.float32(0)))) == c
        assert oracle.e4m3_encode_scalar(float(-mid)) == even | 0x80


def test_encode_saturation_and_specials(oracle):
    f32 = np.float32
    for v, code in [(448.0, 0x7E), (450.0, 0x7E), (464.0, 0x7E), (479.0, 0x7E),
                    (480.0, 0x7E), (1e38, 0x7E), (float("inf"), 0x7E),
                    (-448.0, 0xFE), (-1e30, 0xFE), (float("-inf"), 0xFE),
                    (2.0 ** -10, 0x00), (2.0 ** -11, 0x00), (-(2.0 ** -12), 0x80),
                    (float(np.nextafter(f32(2.0 ** -10), f32(1))), 0x01),
                    (3 * 2.0 ** -10, 0x02), (0.0, 0x00), (-0.0, 0x80),
                    (432.0, 0x7E), (431.99, 0x7D)]:
        assert oracle.e4m3_encode_scalar(v) == code, v
    assert oracle.e4m3_encode_scalar(float("nan")) == 0x7F


def test_encode_matches_search_random(oracle):
    rng = np.random.default_rng(1234)
    # wide log-uniform magnitudes, both signs, plus raw bit patterns
    mag = np.exp2(rng.uniform(-16, 10, 1 << 20)).astype(np.float32)
    x = np.where(rng.random(mag.size) < 0.5, -mag, mag).astype(np.float32)
    bits = rng.integers(0, 2 ** 32, 1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    for arr in (x, bits):
        got = oracle.e4m3_encode(arr)
        want = _brute_encode(oracle, arr)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (arr[bad[:5]], got[bad[:5]], want[bad[:5]])


@pytest.mark.parametrize("lo_exp", [-10, -7, 0, 8])
def test_encode_exhaustive_binade(oracle, lo_exp):
    # every float32 in [2^lo_exp, 2^(lo_exp+1)): subnormal-range rounding,
    # the first normal binade, a mid binade and the binade holding 448
    lo = np.array([2.0 ** lo_exp], np.float32).view(np.uint32)[0]
    hi = np.array([2.0 ** (lo_exp + 1)], np.float32).view(np.uint32)[0]
    arr = np.arange(lo, hi, dtype=np.uint32).view(np.float32)
    got = oracle.e4m3_encode(arr)
    want = _brute_encode(oracle, arr)
    assert np.array_equal(got, want)
