"""Pins for the oracle's per-group-scaled GEMM and grouped GEMM (CPU only).

The GEMM of the method (dssusan.co.kr post 91437, paragraph 3, Figure 6)
multiplies FP8 codes on the tensor cores and applies the per-128-K-group scales
of both operands as a dequantisation step, accumulating in FP32.  Up to
rounding order that is the product of the dequantised operands, so the oracle
evaluates that product in double.  It is pinned against a library matmul of
the dequantised matrices (numpy, BLAS), against exact integer products, and
against special cases whose result is known in closed form.
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth


def _dequant_a(oracle, qa, sa):
    return oracle.e4m3_decode(qa) * np.repeat(sa.T.astype(np.float64), 128, axis=1)


def _dequant_b(oracle, qb, sb, kind):
    N, K = qb.shape
    n = np.arange(N)[:, None]
    kb = np.arange(K)[None, :] // 128
    if kind == 0:
        s = sb[n // 128, kb]
    elif kind == 1:
        s = sb[kb, n // 128]
    else:
        s = sb[kb, n]
    return oracle.e4m3_decode(qb) * s.astype(np.float64)


@pytest.mark.parametrize("kind", [0, 1, 2])
def test_gemm_matches_library_matmul(oracle, kind):
    M, N, K = 70, 200, 384
    x = synth.activation(M, K, seed=21)
    w = synth.weight(N, K, seed=22)
    qa, sa = oracle.quant_act(x)
    if kind == 0:
        qb, sb = oracle.quant_weight(w)
    elif kind == 1:
        qb, sb0 = oracle.quant_weight(w)
        sb = np.ascontiguousarray(sb0.T)
    else:
        qb, sb = oracle.quant_act(w)          # per-row scales, [K/128][N]
    c, ad = oracle.gemm_rows(qa, sa, qb, sb, kind)
    A = _dequant_a(oracle, qa, sa)
    B = _dequant_b(oracle, qb, sb, kind)
    ref = A @ B.T
    assert np.allclose(c, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(ad, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    assert np.all(ad >= np.abs(c))


def test_gemm_exact_integers(oracle):
    # unit scales and small-integer codes: the result is an exact integer GEMM
    rng = np.random.default_rng(5)
    M, N, K = 33, 48, 256
    ints = np.arange(-16, 17)
    codes = oracle.e4m3_encode(ints.astype(np.float32))
    assert np.array_equal(oracle.e4m3_decode(codes), ints)
    ia = rng.integers(0, ints.size, (M, K))
    ib = rng.integers(0, ints.size, (N, K))
    qa, qb = codes[ia], codes[ib]
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((1, K // 128), np.float32)
    c, _ = oracle.gemm_rows(qa, sa, qb, sb, 0)
    want = ints[ia].astype(np.int64) @ ints[ib].astype(np.int64).T
    assert np.array_equal(c, want.astype(np.float64))


def test_gemm_single_group(oracle):
    # all scales zero except group g: C is the scaled dot product of that group
    M, N, K = 16, 130, 512
    x = synth.activation(M, K, seed=31)
    w = synth.weight(N, K, seed=32)
    qa, sa = oracle.quant_act(x)
    qb, sb = oracle.quant_weight(w)
    g = 2
    sa2 = np.zeros_like(sa)
    sa2[g] = sa[g]
    c, ad = oracle.gemm_rows(qa, sa2, qb, sb, 0)
    sl = slice(g * 128, (g + 1) * 128)
    da = oracle.e4m3_decode(qa[:, sl])
    db = oracle.e4m3_decode(qb[:, sl])
    want = (da @ db.T) * sa[g][:, None].astype(np.float64) * \
        np.repeat(sb[:, g], 128)[:N][None, :].astype(np.float64)
    # the exact group dot product is scaled once here and per term in the
    # oracle: the two differ by rounding only (a few ulp of sum |a_k b_k|)
    assert np.all(np.abs(c - want) <= 1e-14 * ad)


def test_gemm_row_subset(oracle):
    x = synth.activation(64, 256, seed=41)
    w = synth.weight(96, 256, seed=42)
    qa, sa = oracle.quant_act(x)
    qb, sb = oracle.quant_weight(w)
    full, _ = oracle.gemm_rows(qa, sa, qb, sb, 0)
    rows = np.array([63, 0, 17, 17])
    part, _ = oracle.gemm_rows(qa, sa, qb, sb, 0, rows)
    assert np.array_equal(part, full[rows])


def test_grouped_gemm_is_per_expert_gemm(oracle):
    G, N, K = 4, 160, 256
    offs = np.array([0, 50, 50, 181, 300], np.int32)   # one empty expert
    M = int(offs[-1])
    x = synth.activation(M, K, seed=51)
    qa, sa = oracle.quant_act(x)
    qbs, sbs = [], []
    for g in range(G):
        qb, sb = oracle.quant_weight(synth.weight(N, K, seed=52 + g))
        qbs.append(qb)
        sbs.append(sb)
    qb = np.stack(qbs)
    sb = np.stack(sbs)
    c, ad = oracle.grouped_gemm_rows(qa, sa, qb, sb, offs)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        cg, adg = oracle.gemm_rows(qa, sa, qb[g], sb[g], 0, np.arange(lo, hi))
        assert np.array_equal(c[lo:hi], cg) and np.array_equal(ad[lo:hi], adg)


def test_tolerance_helper(oracle):
    # half a BF16 ulp: 1.0 -> 2^-8; just below 2 -> 2^-8; 2.0 -> 2^-7
    t = oracle.gemm_tolerance(np.array([1.0, 1.99, 2.0]), np.zeros(3), True)
    assert np.array_equal(t, [2.0 ** -8, 2.0 ** -8, 2.0 ** -7])
    t = oracle.gemm_tolerance(np.array([1.0]), np.array([10.0]), False)
    assert t[0] == pytest.approx(2e-3)


def _per_tensor_gemm(oracle, x, w, pow2):
    M, K = x.shape
    N = w.shape[0]
    qx, sx = oracle.quant_tensor(x, pow2)
    qw, sw = oracle.quant_tensor(w, pow2)
    c, _ = oracle.gemm_rows(qx, np.full((K // 128, M), sx, np.float32), qw,
                            np.full(((N + 127) // 128, K // 128), sw, np.float32),
                            oracle.BSCALE_BLOCK)
    return c


def test_gemm_error_fine_grained_vs_per_tensor(oracle):
    # GEMM-level comparison on the tiny Fprop inputs (0.1 % x100 outliers),
    # both against an unquantised BF16 product in double.  With FP32 scales the
    # 1x128 / 128x128 grouping lowers the error; with power-of-two scales a
    # finer scale only shifts exponents, so while every value stays in E4M3's
    # normal range the two give the same codes' relative precision.
    x = synth.activation(256, 512, seed=0, name="tiny.X")
    w = synth.weight(256, 512, seed=0, name="tiny.W")
    ref = oracle.bf16_gemm_rows(x, w)

    def rel(c):
        return np.linalg.norm(c - ref) / np.linalg.norm(ref)

    err = {}
    for pow2 in (False, True):
        qa, sa = oracle.quant_act(x, pow2)
        qb, sb = oracle.quant_weight(w, pow2)
        fine, _ = oracle.gemm_rows(qa, sa, qb, sb, oracle.BSCALE_BLOCK)
        err[pow2] = (rel(fine), rel(_per_tensor_gemm(oracle, x, w, pow2)))
    assert err[False][0] < 0.8 * err[False][1]
    assert err[True][0] <= err[True][1] * (1 + 1e-9)
    assert all(e < 0.1 for pair in err.values() for e in pair)
