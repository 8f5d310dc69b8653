"""GPU parity of the scaled FP8 GEMM and grouped GEMM against the CPU oracle.

The oracle evaluates the dequantised product in double; the GPU result must
lie within |C - C_ref| <= 2e-4 * sum_k |a_k b_k| (+ half a BF16 ulp for BF16
outputs), element by element.  Operands come from the quantisers, so every
test here also runs the quantisers on the GPU; the oracle quantises the same
inputs independently and the codes are checked to agree first.
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import (assert_bytes_equal, assert_scales_equal, assert_within_tolerance,
                   bf16_to_torch, f32, f64, u8)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
B = pytest.importorskip("fp8_fine_grained_amax_gb300.binding")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_fine_grained_amax_gb300.build import build_library
    build_library()
    B.load_library()
    yield
    assert B.fp8q_sync_status() == 0


def _quant_pair(oracle, x, w, transpose_w=False):
    """Quantise on both sides; check they agree; return GPU tensors + oracle arrays."""
    qa_ref, sa_ref = oracle.quant_act(x)
    qb_ref, sb_ref = oracle.quant_weight(w)
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x))
    out = B.fp8q_quant_weight(bf16_to_torch(w), with_transpose=transpose_w)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_ref, "A codes")
    assert_scales_equal(f32(sa), sa_ref, "A scales")
    assert_bytes_equal(u8(out[0]), qb_ref, "B codes")
    assert_scales_equal(f32(out[1]), sb_ref, "B scales")
    return (qa, sa, *out), (qa_ref, sa_ref, qb_ref, sb_ref)


def _check(c_gpu, ref, absdot, out_bf16, what):
    import oracle as orc
    tol = orc.gemm_tolerance(ref, absdot, out_bf16)
    assert_within_tolerance(f64(c_gpu), ref, tol, what)


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (200, 264, 384), (1, 8, 128),
                                   (129, 520, 256), (300, 1000, 640), (128, 256, 128),
                                   (640, 768, 1024)])
def test_gemm_fprop(oracle, M, N, K, out):
    x = synth.activation(M, K, seed=M + 7 * N)
    w = synth.weight(N, K, seed=K + 3 * N)
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _quant_pair(oracle, x, w)
    od = B.FP8Q_OUT_BF16 if out == "bf16" else B.FP8Q_OUT_FP32
    c = B.fp8q_gemm(qa, sa, qb, sb, out_dtype=od)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c, ref, ad, out == "bf16", f"fprop {M}x{N}x{K} {out}")


def test_gemm_tiny_fprop_error_vs_bf16(oracle):
    # the tiny Fprop workload; also reports (does not pin) the error against an
    # unquantised BF16 product
    M, N, K = 256, 256, 512
    x = synth.activation(M, K, seed=0, name="tiny.X")
    w = synth.weight(N, K, seed=0, name="tiny.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _quant_pair(oracle, x, w)
    c = B.fp8q_gemm(qa, sa, qb, sb)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c, ref, ad, True, "tiny fprop")
    exact = oracle.bf16_gemm_rows(x, w)
    rel = np.linalg.norm(f64(c) - exact) / np.linalg.norm(exact)
    assert rel < 0.1   # context: FP8 quantisation error, not a parity bound


def test_gemm_dgrad_block_transposed(oracle):
    # dX = dY * W with W [out][in]: B operand = W's transposed codes [in][out],
    # B scales = W's block grid read transposed
    T, d_in, d_out = 384, 640, 256
    dy = synth.normal_bf16((T, d_out), 1e-3, 1, "dgrad.dY")
    w = synth.weight(d_out, d_in, seed=2, name="dgrad.W")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(dy))
    qw, sbw, qwT = B.fp8q_quant_weight(bf16_to_torch(w), with_transpose=True)
    c = B.fp8q_gemm(qa, sa, qwT, sbw, bscale_kind=B.FP8Q_BSCALE_BLOCK_T)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act(dy)
    qw_r, sbw_r = oracle.quant_weight(w)
    assert_bytes_equal(u8(qwT), np.ascontiguousarray(qw_r.T), "W^T codes")
    ref, ad = oracle.gemm_rows(qa_r, sa_r, np.ascontiguousarray(qw_r.T), sbw_r,
                               oracle.BSCALE_BLOCK_T)
    _check(c, ref, ad, True, "dgrad")


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_gemm_wgrad_row_scales(oracle, out):
    # dW = dY^T X, both operands quantised 128x1 along tokens (K of this GEMM)
    T, d_in, d_out = 512, 392, 264
    dy = synth.normal_bf16((T, d_out), 1e-3, 3, "wgrad.dY")
    x = synth.activation(T, d_in, seed=4, name="wgrad.X")
    qdyT, sdyT = B.fp8q_quant_act_T(bf16_to_torch(dy))
    qxT, sxT = B.fp8q_quant_act_T(bf16_to_torch(x))
    od = B.FP8Q_OUT_FP32 if out == "fp32" else B.FP8Q_OUT_BF16
    c = B.fp8q_gemm(qdyT, sdyT, qxT, sxT, bscale_kind=B.FP8Q_BSCALE_ROW, out_dtype=od)
    torch.cuda.synchronize()
    qdyT_r, sdyT_r = oracle.quant_act_T(dy)
    qxT_r, sxT_r = oracle.quant_act_T(x)
    assert_bytes_equal(u8(qdyT), qdyT_r, "dY^T codes")
    assert_bytes_equal(u8(qxT), qxT_r, "X^T codes")
    ref, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW)
    _check(c, ref, ad, out == "bf16", "wgrad")


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_gemm_wgrad_row_scales_odd_n(oracle, out):
    # per-column scales with an odd N: the FP32 fragments end in a lone
    # column (scalar store) and BF16 rows end inside a 16-byte unit (row
    # stores, no tensor store); C is a strided view whose padding columns
    # must stay untouched
    T, d_in, d_out = 256, 101, 264
    dy = synth.normal_bf16((T, d_out), 1e-3, 7, "wgrad.dY.odd")
    x = synth.activation(T, d_in, seed=8, name="wgrad.X.odd")
    xpad = torch.zeros((T, 104), dtype=torch.bfloat16, device="cuda")
    xpad[:, :d_in] = bf16_to_torch(x)
    qdyT, sdyT = B.fp8q_quant_act_T(bf16_to_torch(dy))
    # channels are quantised independently: the first 101 of the padded X's
    # 104 are X's own (the 128x1 quantiser takes C in multiples of 8)
    qxT_full, sxT_full = B.fp8q_quant_act_T(xpad)
    qxT, sxT = qxT_full[:d_in], sxT_full[:, :d_in]
    fp32 = out == "fp32"
    od = B.FP8Q_OUT_FP32 if fp32 else B.FP8Q_OUT_BF16
    cbuf = torch.full((d_out, 104), 7.0, dtype=torch.float32 if fp32 else torch.bfloat16,
                      device="cuda")
    B.fp8q_gemm(qdyT, sdyT, qxT, sxT, bscale_kind=B.FP8Q_BSCALE_ROW, out_dtype=od,
                c=cbuf[:, :d_in])
    torch.cuda.synchronize()
    qdyT_r, sdyT_r = oracle.quant_act_T(dy)
    qxT_r, sxT_r = oracle.quant_act_T(x)
    assert_bytes_equal(u8(qxT), qxT_r, "X^T codes")
    ref, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW)
    _check(cbuf[:, :d_in], ref, ad, not fp32, "wgrad, odd N")
    assert bool((cbuf[:, d_in:] == 7.0).all()), "padding columns written"


def test_gemm_k_zero_writes_zeros():
    M, N = 130, 264
    a = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    b = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    sa = torch.empty((0, M), dtype=torch.float32, device="cuda")
    sb = torch.empty((3, 0), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    B.fp8q_gemm(a, sa, b, sb, out_dtype=B.FP8Q_OUT_FP32, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)


def _sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(n, M), replace=False).tolist())
    rows |= {0, M - 1, min(M - 1, 127), min(M - 1, 128)}
    return np.array(sorted(rows), np.int64)


def test_gemm_fprop_full_size_sampled(oracle):
    # the single-linear Fprop workload, M=4096, N=7168, K=7168, BF16 out,
    # checked on sampled rows (every column)
    M, N, K = 4096, 7168, 7168
    x = synth.activation(M, K, seed=0, name="fprop.X")
    w = synth.weight(N, K, seed=0, name="fprop.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _quant_pair(oracle, x, w)
    c = B.fp8q_gemm(qa, sa, qb, sb)
    torch.cuda.synchronize()
    rows = _sample_rows(M, 48, 1)
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK, rows)
    _check(c[torch.from_numpy(rows).cuda()], ref, ad, True, "fprop full size")


def _moe_case(oracle, offs, N, K, seed):
    G = offs.size - 1
    M = int(offs[-1])
    x = synth.activation(M, K, seed=seed, name="moe.X")
    ws = [synth.weight(N, K, seed=seed + 1 + g, name=f"moe.W{g}") for g in range(G)]
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x))
    qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((G, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for g in range(G):
        B.fp8q_quant_weight(bf16_to_torch(ws[g]), q=qb[g], sb=sb[g])
    torch.cuda.synchronize()
    qb_r = np.stack([oracle.quant_weight(wg)[0] for wg in ws])
    sb_r = np.stack([oracle.quant_weight(wg)[1] for wg in ws])
    qa_r, sa_r = oracle.quant_act(x)
    assert_bytes_equal(u8(qb), qb_r, "expert codes")
    return (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r)


@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_grouped_gemm_small(oracle, out):
    offs = np.array([0, 77, 77, 300, 301, 555], np.int32)   # one empty, one single-row expert
    N, K = 264, 384
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _moe_case(oracle, offs, N, K, 11)
    od = B.FP8Q_OUT_BF16 if out == "bf16" else B.FP8Q_OUT_FP32
    M = int(offs[-1])
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    c = torch.full((M + 5, N), 3.0, dtype=dt, device="cuda")   # rows past offs[G] untouched
    B.fp8q_grouped_gemm(torch.cat([qa, torch.zeros((5, K), dtype=torch.uint8, device="cuda")]),
                        torch.cat([sa, torch.ones((K // 128, 5), device="cuda")], dim=1)
                        .contiguous(), qb, sb, torch.from_numpy(offs).cuda(), out_dtype=od, c=c)
    torch.cuda.synchronize()
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r, sb_r, offs)
    _check(c[:M], ref, ad, out == "bf16", "grouped small")
    assert torch.all(c[M:] == 3.0)


def test_grouped_gemm_moe_workload_sampled(oracle):
    # MoE up-projection: 16 experts, 16384 tokens, Dirichlet(0.5) top-1 routing,
    # K=7168 -> N=4096; sampled rows of every expert
    offs = synth.moe_offsets(16384, 16, 0.5, seed=0)
    N, K = 4096, 7168
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _moe_case(oracle, offs, N, K, 0)
    c = B.fp8q_grouped_gemm(qa, sa, qb, sb, torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    rows = set()
    for g in range(16):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            rows |= {lo, hi - 1, (lo + hi) // 2}
    rows = np.array(sorted(rows), np.int64)
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r, sb_r, offs, rows)
    _check(c[torch.from_numpy(rows).cuda()], ref, ad, True, "moe up-proj")


def test_wait_timeout_is_reported():
    # a bounded wait on a barrier nothing completes must give up and report
    assert B.fp8q_sync_status() == 0
    B.fp8q_selftest_wait_timeout(2_000_000)   # 2 ms
    assert B.fp8q_sync_status() == B.FP8Q_ERR_TIMEOUT
    assert B.fp8q_sync_status() == 0          # cleared by the read


def test_gemm_accumulate_wgrad_two_microbatches(oracle):
    # dW accumulated over two micro-batches of tokens: dW = dY1^T X1 + dY2^T X2,
    # FP32, each term a 128x1-quantised Wgrad GEMM (per-row scales)
    T, d_in, d_out = 256, 264, 136
    acc = torch.zeros((d_out, d_in), dtype=torch.float32, device="cuda")
    ref = np.zeros((d_out, d_in))
    absdot = np.zeros((d_out, d_in))
    for mb in range(2):
        dy = synth.normal_bf16((T, d_out), 1e-3, 40 + mb, "acc.dY")
        x = synth.activation(T, d_in, seed=50 + mb, name="acc.X")
        qdyT, sdyT = B.fp8q_quant_act_T(bf16_to_torch(dy))
        qxT, sxT = B.fp8q_quant_act_T(bf16_to_torch(x))
        B.fp8q_gemm_accumulate(qdyT, sdyT, qxT, sxT, acc, bscale_kind=B.FP8Q_BSCALE_ROW)
        qdyT_r, sdyT_r = oracle.quant_act_T(dy)
        qxT_r, sxT_r = oracle.quant_act_T(x)
        r, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW)
        ref += r
        absdot += ad
    torch.cuda.synchronize()
    # each accumulation adds one FP32 rounding of the running sum
    tol = 2e-4 * absdot + 2 * np.abs(ref) * 2.0 ** -24
    assert_within_tolerance(f64(acc), ref, tol, "accumulated wgrad")


def test_gemm_accumulate_keeps_existing_values_for_k_zero():
    M, N = 40, 136
    c = torch.full((M, N), 1.5, dtype=torch.float32, device="cuda")
    a = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    b = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    sa = torch.empty((0, M), dtype=torch.float32, device="cuda")
    sb = torch.empty((2, 0), dtype=torch.float32, device="cuda")
    B.fp8q_gemm_accumulate(a, sa, b, sb, c)
    torch.cuda.synchronize()
    assert torch.all(c == 1.5)


@pytest.mark.parametrize("kind", ["block", "block_t"])
def test_gemm_accumulate_block_scales(oracle, kind):
    # C (FP32, random start values) += the block-scaled product, Fprop and
    # Dgrad scale layouts; ragged M and N
    M, N, K = 300, 392 if kind == "block" else 384, 640
    x = synth.activation(M, K, seed=81, name="accb.X")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x))
    qa_r, sa_r = oracle.quant_act(x)
    if kind == "block":
        w = synth.weight(N, K, seed=82, name="accb.W")
        qb, sb = B.fp8q_quant_weight(bf16_to_torch(w))
        qb_r, sb_r = oracle.quant_weight(w)
        bk, okind = B.FP8Q_BSCALE_BLOCK, oracle.BSCALE_BLOCK
    else:
        w = synth.weight(K, N, seed=83, name="accb.Wt")
        _, sb, qb = B.fp8q_quant_weight(bf16_to_torch(w), with_transpose=True)
        qw_r, sb_r = oracle.quant_weight(w)
        qb_r = np.ascontiguousarray(qw_r.T)
        bk, okind = B.FP8Q_BSCALE_BLOCK_T, oracle.BSCALE_BLOCK_T
    c0 = np.random.default_rng(84).standard_normal((M, N)).astype(np.float32)
    c = torch.from_numpy(c0).cuda()
    B.fp8q_gemm_accumulate(qa, sa, qb, sb, c, bscale_kind=bk)
    torch.cuda.synchronize()
    prod, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, okind)
    ref = c0.astype(np.float64) + prod
    # the product's bound, plus the one FP32 rounding of the addition
    tol = 2e-4 * ad + np.abs(ref) * 2.0 ** -24 + 1e-30
    assert_within_tolerance(f64(c), ref, tol, f"accumulate {kind}")


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("kind", ["fprop", "wgrad"])
def test_gemm_deep_k(oracle, kind, pow2):
    # K = 16384: 128 K-groups through the FP32 fold (both TMEM buffers cycle
    # 64 times) or through the power-of-two kernel's scale ring; Wgrad reduces
    # over 16384 tokens (per-column scales, FP32 out)
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    gemm = B.fp8q_gemm_pow2 if pow2 else B.fp8q_gemm
    K = 16384
    if kind == "fprop":
        M, N = 200, 256
        x = synth.activation(M, K, seed=91, name="deepk.X")
        w = synth.weight(N, K, seed=92, name="deepk.W")
        qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=mode)
        qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=mode)
        c = gemm(qa, sa, qb, sb)
        qa_r, sa_r = oracle.quant_act(x, pow2)
        qb_r, sb_r = oracle.quant_weight(w, pow2)
        bk, bf16_out = oracle.BSCALE_BLOCK, True
    else:
        M, N = 256, 136
        dy = synth.normal_bf16((K, M), 1e-3, 93, "deepk.dY")
        xx = synth.activation(K, N, seed=94, name="deepk.Xw")
        qa, sa = B.fp8q_quant_act_T(bf16_to_torch(dy), scale_mode=mode)
        qb, sb = B.fp8q_quant_act_T(bf16_to_torch(xx), scale_mode=mode)
        c = gemm(qa, sa, qb, sb, bscale_kind=B.FP8Q_BSCALE_ROW, out_dtype=B.FP8Q_OUT_FP32)
        qa_r, sa_r = oracle.quant_act_T(dy, pow2)
        qb_r, sb_r = oracle.quant_act_T(xx, pow2)
        bk, bf16_out = oracle.BSCALE_ROW, False
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    assert_bytes_equal(u8(qb), qb_r, "B codes")
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, bk)
    assert_within_tolerance(f64(c), ref, oracle.gemm_tolerance(ref, ad, bf16_out),
                            f"{kind} K={K}")
