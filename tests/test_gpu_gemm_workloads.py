"""GPU parity of both GEMM paths at the workloads' full sizes and on strided layouts.

* Linear backward, T = 8192, d_in = 7168, d_out = 2048: Dgrad (BF16 out, the
  weight's transposed codes and block scales) and Wgrad (FP32 out, both
  operands quantised 128x1 along tokens), launched as the benchmark launches
  them, checked on sampled rows of every column.
* The square GEMM sweep M = N = K in {2048, 4096, 8192, 16384}, sampled rows.
* Row strides larger than the rows (A, B, C and both scale arrays): the
  kernels must read and write through the strides and leave the padding alone.

Each runs on the FP32-scale GEMM (fp8q_gemm) and on the power-of-two GEMM
(fp8q_gemm_pow2, block-scaled MMA).  The oracle quantises the same inputs on
the CPU; the codes are compared byte for byte before the products are, and the
products must satisfy |C - C_ref| <= 2e-4 * sum_k |a_k b_k| (+ half a BF16 ulp
for BF16 outputs).
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import assert_bytes_equal, assert_scales_equal, assert_within_tolerance, \
    bf16_to_torch, f32, f64, u8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
B = pytest.importorskip("fp8_fine_grained_amax_gb300.binding")

MODES = ["fp32", "pow2"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_fine_grained_amax_gb300.build import build_library
    build_library()
    B.load_library()
    yield
    assert B.fp8q_sync_status() == 0


def _gemm(mode):
    return B.fp8q_gemm_pow2 if mode == "pow2" else B.fp8q_gemm


def _scale_mode(mode):
    return B.FP8Q_SCALE_POW2 if mode == "pow2" else B.FP8Q_SCALE_FP32


def _check(c_rows, ref, absdot, out_bf16, what):
    import oracle as orc
    tol = orc.gemm_tolerance(ref, absdot, out_bf16)
    assert_within_tolerance(f64(c_rows), ref, tol, what)


def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows |= {0, M - 1, min(M - 1, 127), min(M - 1, 128), min(M - 1, 255), min(M - 1, 256)}
    return np.array(sorted(rows), np.int64)


def _rows_of(c, rows):
    return c[torch.from_numpy(rows).to(c.device)]


@pytest.mark.parametrize("mode", MODES)
def test_linear_backward_full_size_sampled(oracle, mode):
    T, d_in, d_out = 8192, 7168, 2048
    p2 = mode == "pow2"
    sm = _scale_mode(mode)
    dy = synth.normal_bf16((T, d_out), 1e-3, 0, "bwd.dY")
    x = synth.activation(T, d_in, seed=0, name="bwd.X")
    w = synth.weight(d_out, d_in, seed=0, name="bwd.W")
    qdyT, sdyT, qdy, sdy = B.fp8q_quant_act_T(bf16_to_torch(dy), with_rows=True, scale_mode=sm)
    qxT, sxT = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=sm)
    qw, sw, qwT = B.fp8q_quant_weight(bf16_to_torch(w), with_transpose=True, scale_mode=sm)
    dX = _gemm(mode)(qdy, sdy, qwT, sw, bscale_kind=B.FP8Q_BSCALE_BLOCK_T)
    dW = _gemm(mode)(qdyT, sdyT, qxT, sxT, bscale_kind=B.FP8Q_BSCALE_ROW,
                     out_dtype=B.FP8Q_OUT_FP32)
    torch.cuda.synchronize()

    qdy_r, sdy_r = oracle.quant_act(dy, p2)
    qdyT_r, sdyT_r = oracle.quant_act_T(dy, p2)
    qxT_r, sxT_r = oracle.quant_act_T(x, p2)
    qw_r, sw_r = oracle.quant_weight(w, p2)
    qwT_r = np.ascontiguousarray(qw_r.T)
    assert_bytes_equal(u8(qdy), qdy_r, "dY codes")
    assert_scales_equal(f32(sdy), sdy_r, "dY scales")
    assert_bytes_equal(u8(qdyT), qdyT_r, "dY^T codes")
    assert_bytes_equal(u8(qxT), qxT_r, "X^T codes")
    assert_scales_equal(f32(sxT), sxT_r, "X^T scales")
    assert_bytes_equal(u8(qwT), qwT_r, "W^T codes")
    assert_scales_equal(f32(sw), sw_r, "W scales")

    rows = _sample_rows(T, 24, 2)
    ref, ad = oracle.gemm_rows(qdy_r, sdy_r, qwT_r, sw_r, oracle.BSCALE_BLOCK_T, rows)
    _check(_rows_of(dX, rows), ref, ad, True, f"{mode} dgrad 8192x7168x2048")
    rows = _sample_rows(d_out, 24, 3)
    ref, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW, rows)
    _check(_rows_of(dW, rows), ref, ad, False, f"{mode} wgrad 2048x7168x8192")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [2048, 4096, 8192, 16384])
def test_square_sweep_sampled(oracle, n, mode):
    p2 = mode == "pow2"
    sm = _scale_mode(mode)
    x = synth.activation(n, n, seed=0, name=f"square_{n}.X")
    w = synth.weight(n, n, seed=0, name=f"square_{n}.W")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=sm)
    qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=sm)
    c = _gemm(mode)(qa, sa, qb, sb)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act(x, p2)
    qb_r, sb_r = oracle.quant_weight(w, p2)
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    assert_bytes_equal(u8(qb), qb_r, "B codes")
    rows = _sample_rows(n, 10, n)
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK, rows)
    _check(_rows_of(c, rows), ref, ad, True, f"{mode} square {n}")


def _padded(t, pad_cols, fill):
    """Copy of 2-D tensor t inside a wider buffer; returns (view, buffer)."""
    buf = torch.full((t.shape[0], t.shape[1] + pad_cols), fill, dtype=t.dtype, device=t.device)
    buf[:, : t.shape[1]] = t
    return buf[:, : t.shape[1]], buf


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("kind", ["block", "block_t", "row"])
def test_strided_operands_and_output(oracle, mode, kind):
    # every array is a view of a wider buffer: A and B rows padded by 48 and 16
    # bytes, scale rows by 3 floats (odd strides), C rows by 16 bytes; the
    # padding of C must keep its sentinel
    p2 = mode == "pow2"
    sm = _scale_mode(mode)
    # (Wgrad: A's rows are dY's channels, so its BF16 rows need a 16-byte pitch;
    # Dgrad: N is the weight's inner dimension, a whole number of 128-groups)
    M, N, K = (264 if kind == "row" else 300), (384 if kind == "block_t" else 392), 640
    if kind == "row":
        # Wgrad shape: both operands quantised 128x1 along the K (token) axis
        dy = synth.normal_bf16((K, M), 1e-3, 21, "strided.dY")
        x = synth.activation(K, N, seed=22, name="strided.X")
        qa, sa = B.fp8q_quant_act_T(bf16_to_torch(dy), scale_mode=sm)
        qb, sb = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=sm)
        qa_r, sa_r = oracle.quant_act_T(dy, p2)
        qb_r, sb_r = oracle.quant_act_T(x, p2)
        bk, okind, out = B.FP8Q_BSCALE_ROW, oracle.BSCALE_ROW, B.FP8Q_OUT_FP32
    else:
        x = synth.activation(M, K, seed=23, name="strided.X")
        qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=sm)
        qa_r, sa_r = oracle.quant_act(x, p2)
        if kind == "block":
            w = synth.weight(N, K, seed=24, name="strided.W")
            qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=sm)
            qb_r, sb_r = oracle.quant_weight(w, p2)
            bk, okind = B.FP8Q_BSCALE_BLOCK, oracle.BSCALE_BLOCK
        else:
            # Dgrad: W [K][N] as [out][in]; the GEMM's B is its transposed codes
            w = synth.weight(K, N, seed=25, name="strided.Wt")
            _, sb, qb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=sm, with_transpose=True)
            qw_r, sb_r = oracle.quant_weight(w, p2)
            qb_r = np.ascontiguousarray(qw_r.T)
            bk, okind = B.FP8Q_BSCALE_BLOCK_T, oracle.BSCALE_BLOCK_T
        out = B.FP8Q_OUT_BF16
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    assert_bytes_equal(u8(qb), qb_r, "B codes")

    a_v, _ = _padded(qa, 48, 0x7E)
    b_v, _ = _padded(qb, 16, 0x7E)
    sa_v, _ = _padded(sa, 3, float("nan"))
    sb_v, _ = _padded(sb, 3, float("nan"))
    dt = torch.float32 if out == B.FP8Q_OUT_FP32 else torch.bfloat16
    pad_c = 16 // (4 if out == B.FP8Q_OUT_FP32 else 2)
    c_buf = torch.full((M, N + pad_c), -5.0, dtype=dt, device="cuda")
    c_v = c_buf[:, :N]
    _gemm(mode)(a_v, sa_v, b_v, sb_v, bscale_kind=bk, out_dtype=out, c=c_v)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, okind)
    _check(c_v, ref, ad, out == B.FP8Q_OUT_BF16, f"{mode} strided {kind}")
    assert torch.all(c_buf[:, N:] == -5.0), "padding of C was written"


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("N", [300, 13])
def test_bf16_rows_ending_inside_a_16_byte_unit(oracle, mode, N):
    # BF16 rows of N % 8 != 0 columns end inside a 16-byte unit: the kernels
    # must not write the padding of C (pitch rounded up to 16 bytes)
    p2 = mode == "pow2"
    sm = _scale_mode(mode)
    M, K = 200, 384
    x = synth.activation(M, K, seed=31, name="ragged.X")
    w = synth.weight(N, K, seed=32, name="ragged.W")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=sm)
    qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=sm)
    qa_r, sa_r = oracle.quant_act(x, p2)
    qb_r, sb_r = oracle.quant_weight(w, p2)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qb), qb_r, "B codes")
    ldc = (N + 7) // 8 * 8
    c_buf = torch.full((M, ldc), -5.0, dtype=torch.bfloat16, device="cuda")
    _gemm(mode)(qa, sa, qb, sb, c=c_buf[:, :N])
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c_buf[:, :N], ref, ad, True, f"{mode} ragged N={N}")
    assert torch.all(c_buf[:, N:] == -5.0), "padding of C was written"


def _effective_offsets(offs, M):
    """Expert row ranges as the grouped GEMM's interface defines them for
    offsets that break the ordering: clamp into [0, M]; an expert starts no
    earlier than the previous one ended; a decreasing step is an empty expert."""
    c = np.clip(offs.astype(np.int64), 0, M)
    eff = np.zeros_like(c)
    prev_hi = 0
    for g in range(offs.size - 1):
        lo = max(c[g], prev_hi)
        hi = max(lo, c[g + 1])
        eff[g] = lo
        prev_hi = hi
    eff[-1] = prev_hi
    return eff.astype(np.int32)


def _grouped(mode):
    return B.fp8q_grouped_gemm_pow2 if mode == "pow2" else B.fp8q_grouped_gemm


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", ["max_experts", "unordered_offsets"])
def test_grouped_gemm_offset_edge_cases(oracle, mode, case):
    p2 = mode == "pow2"
    sm = _scale_mode(mode)
    N, K = 136, 256
    if case == "max_experts":
        # 1024 experts (the most one call takes) over 3000 tokens, a third empty
        G, M = 1024, 3000
        rng = np.random.default_rng(41)
        counts = rng.integers(0, 6, G) * (rng.random(G) > 0.33)
        counts[-1] += M - counts.sum() if counts.sum() < M else 0
        offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        offs = np.minimum(offs, M).astype(np.int32)
    else:
        # offsets past M, a decreasing step and a negative start: clamped
        G, M = 6, 700
        offs = np.array([-5, 120, 90, 300, 301, 900, 650], np.int32)
    eff = _effective_offsets(offs, M)
    x = synth.activation(M, K, seed=42, name="goff.X")
    wq = np.empty((G, N, K), np.uint8)
    ws = np.empty((G, (N + 127) // 128, K // 128), np.float32)
    for g in range(G):
        wq[g], ws[g] = oracle.quant_weight(synth.weight(N, K, seed=1000 + g, name="goff.W"), p2)
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=sm)
    qa_r, sa_r = oracle.quant_act(x, p2)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    c = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    _grouped(mode)(qa, sa, torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda(),
                   torch.from_numpy(offs).cuda(), c=c)
    torch.cuda.synchronize()
    inside = np.arange(int(eff[0]), int(eff[-1]))
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, wq, ws, eff, inside)
    _check(c[torch.from_numpy(inside).cuda()], ref, ad, True, f"{mode} grouped {case}")
    outside = np.setdiff1d(np.arange(M), inside)
    if outside.size:
        assert torch.all(c[torch.from_numpy(outside).cuda()] == 3.0), "rows outside the experts written"
