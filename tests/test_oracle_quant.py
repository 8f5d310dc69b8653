"""Pins for the oracle's quantisers (CPU only).

What the pages fix, and how each is pinned here:
  * grouping -- 1x128 per token per 128 channels for activations, 128x128 per
    128 input x 128 output channels for weights (dssusan.co.kr post 91437,
    paragraph 4, Figure 7 (a)); 128x1 along tokens in the backward pass (same
    paragraph): pinned by locality (a change inside one group moves only that
    group) and by cross-checks between the three groupings;
  * the scale maps each group's max-abs onto the largest finite E4M3 value,
    448 ("Deepseek - Not For everyone", paragraph 4): pinned by hand-worked
    tiles and the invariant that every nonzero group's max-abs element
    encodes to +-448;
  * power-of-two scales (dssusan.co.kr post 91437, paragraph 1): pinned by
    s being an exact power of two with max-abs/s in (224, 448];
  * the dequantisation error of round-to-nearest at E4M3 precision.
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth


def f32_to_bf16_bits(x):
    x = np.asarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "test values must be exact BF16"
    return (u >> 16).astype(np.uint16)


def test_all_ones_tile(oracle):
    x = f32_to_bf16_bits(np.ones((1, 128), np.float32))
    q, sa = oracle.quant_act(x)
    assert np.all(q == 0x7E)                       # 1.0 * (448/1) = 448
    assert sa[0, 0] == np.float32(1.0) / np.float32(448.0)


@pytest.mark.parametrize("j", [-20, -3, 0, 5, 40])
def test_single_element_at_448_pow(oracle, j):
    v = 448.0 * 2.0 ** j
    x = np.zeros((1, 128), np.float32)
    x[0, 17] = -v
    q, sa = oracle.quant_act(f32_to_bf16_bits(x))
    assert sa[0, 0] == np.float32(2.0 ** j)        # 448*2^j / 448, exact
    assert q[0, 17] == 0xFE
    assert np.all(np.delete(q[0], 17) == 0x00)
    qp, sp = oracle.quant_act(f32_to_bf16_bits(x), pow2=True)
    assert sp[0, 0] == np.float32(2.0 ** j) and qp[0, 17] == 0xFE


def test_zero_tile_and_tiny_tile(oracle):
    x = np.zeros((2, 256), np.float32)
    x[0, :128] = -0.0
    x[1, 128] = 2.0 ** -120                        # max-abs below the floor
    q, sa = oracle.quant_act(f32_to_bf16_bits(x))
    floor_s = np.float32(2.0 ** -116) / np.float32(448.0)
    assert np.all(np.isfinite(sa)) and np.all(sa > 0)
    assert sa[0, 0] == floor_s and sa[1, 0] == floor_s and sa[0, 1] == floor_s
    assert sa[1, 1] == floor_s                     # floored: 2^-120 < 2^-116
    assert np.all(q[0, :128] == 0x80)              # -0 keeps its sign
    assert np.all(q[0, 128:] == 0x00)
    # 2^-120 * (448 / 2^-116) = 28 -> exactly representable in E4M3
    assert oracle.e4m3_decode(q[1, 128]) == 28.0
    qp, sp = oracle.quant_act(f32_to_bf16_bits(x), pow2=True)
    assert np.all(sp == np.float32(2.0 ** -124))   # 448 * 2^-124 >= 2^-116 > 224 * 2^-124
    assert np.all(qp[0, :128] == 0x80)


def _invariants(oracle, x_bits, q, s, groups_of, pow2):
    """Check the per-group invariants; groups_of yields (x values, codes, s)."""
    vals = oracle.e4m3_decode(q)
    assert np.all(np.abs(vals) <= 448.0)
    assert not np.any(np.isnan(vals))
    for xv, qv, sv in groups_of:
        amax = np.max(np.abs(xv))
        a = max(amax, 2.0 ** -116)
        assert np.isfinite(sv) and sv > 0
        if pow2:
            e = np.log2(np.float64(sv))
            assert e == np.round(e), "power-of-two scale"
            assert 224.0 < a / sv <= 448.0
        else:
            i = int(np.argmax(np.abs(xv)))
            if amax > 0:
                assert oracle.e4m3_decode(qv[i]) == np.copysign(448.0, xv[i])
        # round-to-nearest error at E4M3 precision, plus FP32 rounding slack
        dq = oracle.e4m3_decode(qv) * np.float64(sv)
        t = np.abs(xv) / np.float64(sv)
        spacing = np.where(t < 2.0 ** -6, 2.0 ** -9,
                           np.exp2(np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 3))
        bound = 0.5 * spacing * sv * (1 + 2.0 ** -18) + np.abs(xv) * 2.0 ** -20
        bound = np.where(t > 448, np.inf, bound)
        assert np.all(np.abs(dq - xv) <= bound)


@pytest.mark.parametrize("pow2", [False, True])
def test_act_invariants(oracle, pow2):
    x = synth.activation(64, 1024, seed=3)
    q, sa = oracle.quant_act(x, pow2)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    groups = ((xf[m, g * 128:(g + 1) * 128], q[m, g * 128:(g + 1) * 128], sa[g, m])
              for m in range(64) for g in range(8))
    _invariants(oracle, x, q, sa, groups, pow2)


@pytest.mark.parametrize("pow2", [False, True])
def test_weight_invariants(oracle, pow2):
    w = synth.weight(300, 384, seed=4)              # ragged last row block
    q, sb = oracle.quant_weight(w, pow2)
    assert sb.shape == (3, 3)
    wf = synth.bf16_to_f32(w).astype(np.float64)
    groups = ((wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].ravel(),
               q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128].ravel(), sb[nb, kb])
              for nb in range(3) for kb in range(3))
    _invariants(oracle, w, q, sb, groups, pow2)


def test_act_group_locality(oracle):
    # one scale per token per 128 channels: moving one element changes only
    # its own (row, 128-group) scale and codes
    x = synth.activation(8, 512, seed=5)
    q0, s0 = oracle.quant_act(x)
    x2 = x.copy()
    x2[3, 200] = f32_to_bf16_bits(np.float32(1000.0))
    q1, s1 = oracle.quant_act(x2)
    diff_s = np.argwhere(s0 != s1)
    assert diff_s.tolist() == [[1, 3]]
    rows, cols = np.nonzero(q0 != q1)
    assert set(rows.tolist()) == {3} and cols.min() >= 128 and cols.max() < 256


def test_act_T_is_act_of_transpose(oracle):
    # 128x1 tiles along tokens are exactly 1x128 tiles of the transposed matrix
    x = synth.activation(384, 200, seed=6)
    for pow2 in (False, True):
        qT, sT = oracle.quant_act_T(x, pow2)
        q, sa = oracle.quant_act(np.ascontiguousarray(x.T), pow2)
        assert np.array_equal(qT, q) and np.array_equal(sT, sa)


def test_weight_block_scale_is_max_of_row_scales(oracle):
    # s = amax/448 is monotone in amax, so each 128x128 block scale is the
    # largest of the 1x128 scales of its rows
    w = synth.weight(256, 512, seed=7)
    _, sb = oracle.quant_weight(w)
    _, sa = oracle.quant_act(w)           # sa [K/128][N]
    for nb in range(2):
        assert np.array_equal(sb[nb], sa[:, nb * 128:(nb + 1) * 128].max(axis=1))


def test_weight_equals_act_when_rows_share_amax(oracle):
    # if every row of a block has the same max-abs, block and tile scaling agree
    w = synth.bf16_to_f32(synth.weight(128, 256, seed=8)).copy()
    w[:, 5] = 0.25
    w[:, 133] = -0.25
    wb = f32_to_bf16_bits(w)
    qw, sb = oracle.quant_weight(wb)
    qa, sa = oracle.quant_act(wb)
    assert np.array_equal(qw, qa)
    assert np.all(sb == sa[:, :1].T)


def test_weight_partial_block_rows(oracle):
    # a last partial block covers only the rows that exist: zero rows appended
    # to fill the block change nothing
    w = synth.weight(200, 256, seed=9)
    pad = np.zeros((256, 256), np.uint16)
    pad[:200] = w
    q1, s1 = oracle.quant_weight(w)
    q2, s2 = oracle.quant_weight(pad)
    assert np.array_equal(q1, q2[:200]) and np.array_equal(s1, s2)
    assert np.all(q2[200:] == 0)


def test_pow2_is_smallest_power(oracle):
    rng = np.random.default_rng(11)
    for amax in np.exp2(rng.uniform(-100, 100, 2000)).astype(np.float32):
        s, inv = oracle.group_scale(float(amax), True)
        assert 448.0 * np.float64(s) >= amax and 224.0 * np.float64(s) < amax
        assert np.float64(s) * np.float64(inv) == 1.0
    # exact boundary: amax = 448 * 2^e gives s = 2^e, just above doubles it
    s, _ = oracle.group_scale(448.0, True)
    assert s == 1.0
    s, _ = oracle.group_scale(float(np.nextafter(np.float32(448.0), np.float32(1e9))), True)
    assert s == 2.0


def test_fp32_scale_is_single_division(oracle):
    for amax in [1.0, 3.0, 0.02, 123.456, 1e-20, 3e38]:
        s, inv = oracle.group_scale(amax, False)
        a = np.float32(amax)
        assert s == a / np.float32(448.0) and inv == np.float32(448.0) / a


def test_requant_T_pow2_equals_quant_T_of_dequantised(oracle):
    # with power-of-two 1x128 scales the dequantised values decode(q) * 2^e are
    # exact and have at most 4 significant bits, so they are exact BF16 values:
    # requantising the FP8 cache must then equal quantising those values 128x1
    x = synth.activation(256, 384, seed=12)
    q, s = oracle.quant_act(x, pow2=True)
    deq = oracle.e4m3_decode(q) * np.repeat(s.T.astype(np.float64), 128, axis=1)
    deq32 = deq.astype(np.float32)
    assert np.array_equal(deq32.astype(np.float64), deq)
    bits = f32_to_bf16_bits(deq32)
    for pow2 in (False, True):
        qT_ref, sT_ref = oracle.quant_act_T(bits, pow2)
        qT, sT = oracle.requant_act_T(q, s, pow2)
        assert np.array_equal(qT, qT_ref) and np.array_equal(sT, sT_ref)


def test_requant_T_fp32_scales_invariants(oracle):
    # FP32 1x128 scales: every channel group's max-abs dequantised value must
    # land on +-448 again, and the codes stay within one E4M3 step of the
    # values requantised in double precision
    x = synth.activation(128, 256, seed=13)
    q, s = oracle.quant_act(x)
    qT, sT = oracle.requant_act_T(q, s)
    deq = (oracle.e4m3_decode(q).astype(np.float32) * np.repeat(s.T, 128, axis=1)).astype(np.float32)
    for c in range(256):
        col = deq[:, c].astype(np.float64)
        i = int(np.argmax(np.abs(col)))
        if col[i] != 0:
            assert oracle.e4m3_decode(qT[c, i]) == np.copysign(448.0, col[i])
        assert sT[0, c] == np.float32(np.max(np.abs(deq[:, c]))) / np.float32(448.0)


def test_quant_tensor_is_one_group(oracle):
    # a single 1x128 group is a whole tensor: per-tensor and per-group agree
    x = synth.activation(1, 128, seed=14)
    for pow2 in (False, True):
        q, s = oracle.quant_tensor(x, pow2)
        qa, sa = oracle.quant_act(x, pow2)
        assert np.array_equal(q, qa) and s == sa[0, 0]


def test_quant_tensor_scale_is_max_of_group_scales(oracle):
    # the tensor's scale is the largest 1x128 scale (monotone in max-abs), and
    # groups holding the tensor's max-abs quantise identically
    x = synth.activation(32, 512, seed=15)
    q, s = oracle.quant_tensor(x)
    qa, sa = oracle.quant_act(x)
    assert s == sa.max()
    g, m = np.unravel_index(np.argmax(sa), sa.shape)
    assert np.array_equal(q[m, g * 128:(g + 1) * 128], qa[m, g * 128:(g + 1) * 128])


def test_fine_grained_beats_per_tensor_on_outliers(oracle):
    # the pages' motivation: with 0.1% x100 outliers, one scale for the whole
    # tensor wastes precision on every other group; 1x128 scaling does not
    x = synth.activation(256, 1024, seed=16)
    xf = synth.bf16_to_f32(x).astype(np.float64)
    q, s = oracle.quant_tensor(x)
    qa, sa = oracle.quant_act(x)
    err_t = oracle.e4m3_decode(q) * np.float64(s) - xf
    err_g = oracle.e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1) - xf
    mse_t, mse_g = np.mean(err_t ** 2), np.mean(err_g ** 2)
    assert mse_g < mse_t / 4


def test_pow2_scale_of_infinite_max_abs(oracle):
    # a dequantised FP8-cache value can overflow FP32 (E4M3 256 * 2^120 = 2^128);
    # the exponent is then clamped to 127: s = 2^127, inv = 2^-127 (subnormal)
    s, inv = oracle.group_scale(float("inf"), True)
    assert s == np.float32(2.0 ** 127) and inv == np.float32(2.0 ** -127)
    s, inv = oracle.group_scale(float("inf"), False)
    assert np.isinf(s) and inv == 0.0
