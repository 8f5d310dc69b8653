"""GPU parity of fp8q_gemm_pow2 (power-of-two scales on the block-scaled MMA)
against the CPU oracle.

Operands are quantised with FP8Q_SCALE_POW2 on both sides (codes and scales
checked bit-exact first); the oracle's product of the dequantised operands in
double is the reference, with the same bound as the FP32-scale GEMM:
|C - C_ref| <= 2e-4 * sum_k |a_k b_k| (+ half a BF16 ulp for BF16 outputs).
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import (assert_bytes_equal, assert_scales_equal, assert_within_tolerance,
                   bf16_to_torch, f32, f64, u8)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
B = pytest.importorskip("fp8_fine_grained_amax_gb300.binding")

P2 = 1  # FP8Q_SCALE_POW2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_fine_grained_amax_gb300.build import build_library
    build_library()
    B.load_library()
    yield
    assert B.fp8q_sync_status() == 0


def _check(c_gpu, ref, absdot, out_bf16, what):
    import oracle as orc
    tol = orc.gemm_tolerance(ref, absdot, out_bf16)
    assert_within_tolerance(f64(c_gpu), ref, tol, what)


def _fprop_operands(oracle, x, w, transpose_w=False):
    qa_r, sa_r = oracle.quant_act(x, True)
    qb_r, sb_r = oracle.quant_weight(w, True)
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=P2)
    out = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=P2, with_transpose=transpose_w)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    assert_scales_equal(f32(sa), sa_r, "A scales")
    assert_bytes_equal(u8(out[0]), qb_r, "B codes")
    assert_scales_equal(f32(out[1]), sb_r, "B scales")
    return (qa, sa, *out), (qa_r, sa_r, qb_r, sb_r)


@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (200, 264, 384), (1, 8, 128),
                                   (129, 520, 256), (300, 1000, 640), (640, 768, 1024),
                                   (513, 312, 1152)])
def test_pow2_fprop(oracle, M, N, K, out):
    x = synth.activation(M, K, seed=M + 7 * N, name="p2.X")
    w = synth.weight(N, K, seed=K + 3 * N, name="p2.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _fprop_operands(oracle, x, w)
    od = B.FP8Q_OUT_BF16 if out == "bf16" else B.FP8Q_OUT_FP32
    c = B.fp8q_gemm_pow2(qa, sa, qb, sb, out_dtype=od)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c, ref, ad, out == "bf16", f"pow2 fprop {M}x{N}x{K} {out}")


def test_pow2_long_k_wraps_the_scale_ring(oracle):
    # 70 K-groups = 18 scale stages per tile: more than the 16 stages the
    # kernel keeps in tensor memory, so the ring wraps inside one tile
    M, N, K = 300, 384, 128 * 70
    x = synth.activation(M, K, seed=5, name="p2long.X")
    w = synth.weight(N, K, seed=6, name="p2long.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _fprop_operands(oracle, x, w)
    c = B.fp8q_gemm_pow2(qa, sa, qb, sb, out_dtype=B.FP8Q_OUT_FP32)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c, ref, ad, False, "pow2 long K")


def test_pow2_several_tiles_per_pair(oracle):
    # 8 x 10 = 80 tiles of 256 x 256: more tiles than CTA pairs fit on the GPU,
    # so pairs run on into a second tile (scale stages written ahead of it)
    M, N, K = 2048, 2560, 512
    x = synth.activation(M, K, seed=8, name="p2tiles.X")
    w = synth.weight(N, K, seed=9, name="p2tiles.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _fprop_operands(oracle, x, w)
    c = B.fp8q_gemm_pow2(qa, sa, qb, sb)
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    _check(c, ref, ad, True, "pow2 80 tiles")


def test_pow2_dgrad_block_transposed(oracle):
    T, d_in, d_out = 384, 640, 256
    dy = synth.normal_bf16((T, d_out), 1e-3, 1, "p2dgrad.dY")
    w = synth.weight(d_out, d_in, seed=2, name="p2dgrad.W")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(dy), scale_mode=P2)
    qw, sbw, qwT = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=P2, with_transpose=True)
    c = B.fp8q_gemm_pow2(qa, sa, qwT, sbw, bscale_kind=B.FP8Q_BSCALE_BLOCK_T)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act(dy, True)
    qw_r, sbw_r = oracle.quant_weight(w, True)
    assert_bytes_equal(u8(qa), qa_r, "dY codes")
    assert_bytes_equal(u8(qwT), np.ascontiguousarray(qw_r.T), "W^T codes")
    ref, ad = oracle.gemm_rows(qa_r, sa_r, np.ascontiguousarray(qw_r.T), sbw_r,
                               oracle.BSCALE_BLOCK_T)
    _check(c, ref, ad, True, "pow2 dgrad")


@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_pow2_wgrad_row_scales(oracle, out):
    T, d_in, d_out = 512, 392, 264
    dy = synth.normal_bf16((T, d_out), 1e-3, 3, "p2wgrad.dY")
    x = synth.activation(T, d_in, seed=4, name="p2wgrad.X")
    qdyT, sdyT = B.fp8q_quant_act_T(bf16_to_torch(dy), scale_mode=P2)
    qxT, sxT = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=P2)
    od = B.FP8Q_OUT_FP32 if out == "fp32" else B.FP8Q_OUT_BF16
    c = B.fp8q_gemm_pow2(qdyT, sdyT, qxT, sxT, bscale_kind=B.FP8Q_BSCALE_ROW, out_dtype=od)
    torch.cuda.synchronize()
    qdyT_r, sdyT_r = oracle.quant_act_T(dy, True)
    qxT_r, sxT_r = oracle.quant_act_T(x, True)
    assert_bytes_equal(u8(qdyT), qdyT_r, "dY^T codes")
    assert_scales_equal(f32(sxT), sxT_r, "X^T scales")
    ref, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW)
    _check(c, ref, ad, out == "bf16", "pow2 wgrad")


def test_pow2_accumulate_two_microbatches(oracle):
    T, d_in, d_out = 256, 264, 136
    acc = torch.zeros((d_out, d_in), dtype=torch.float32, device="cuda")
    ref = np.zeros((d_out, d_in))
    absdot = np.zeros((d_out, d_in))
    for mb in range(2):
        dy = synth.normal_bf16((T, d_out), 1e-3, 60 + mb, "p2acc.dY")
        x = synth.activation(T, d_in, seed=70 + mb, name="p2acc.X")
        qdyT, sdyT = B.fp8q_quant_act_T(bf16_to_torch(dy), scale_mode=P2)
        qxT, sxT = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=P2)
        B.fp8q_gemm_pow2_accumulate(qdyT, sdyT, qxT, sxT, acc, bscale_kind=B.FP8Q_BSCALE_ROW)
        qdyT_r, sdyT_r = oracle.quant_act_T(dy, True)
        qxT_r, sxT_r = oracle.quant_act_T(x, True)
        r, ad = oracle.gemm_rows(qdyT_r, sdyT_r, qxT_r, sxT_r, oracle.BSCALE_ROW)
        ref += r
        absdot += ad
    torch.cuda.synchronize()
    tol = 2e-4 * absdot + 2 * np.abs(ref) * 2.0 ** -24
    assert_within_tolerance(f64(acc), ref, tol, "pow2 accumulated wgrad")


def test_pow2_full_size_sampled(oracle):
    # the single-linear Fprop workload with power-of-two scales, sampled rows
    M, N, K = 4096, 7168, 7168
    x = synth.activation(M, K, seed=0, name="fprop.X")
    w = synth.weight(N, K, seed=0, name="fprop.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _fprop_operands(oracle, x, w)
    c = B.fp8q_gemm_pow2(qa, sa, qb, sb)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    rows = np.array(sorted(set(rng.choice(M, 48, replace=False).tolist()) | {0, 255, 256, M - 1}))
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK, rows)
    _check(c[torch.from_numpy(rows).cuda()], ref, ad, True, "pow2 fprop full size")


def test_pow2_k_zero():
    M, N = 130, 264
    a = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    b = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    sa = torch.empty((0, M), dtype=torch.float32, device="cuda")
    sb = torch.empty((3, 0), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    B.fp8q_gemm_pow2(a, sa, b, sb, out_dtype=B.FP8Q_OUT_FP32, c=c)
    torch.cuda.synchronize()
    assert torch.all(c == 0)
    c.fill_(1.5)
    B.fp8q_gemm_pow2_accumulate(a, sa, b, sb, c)
    torch.cuda.synchronize()
    assert torch.all(c == 1.5)


def test_pow2_rejects_other_scales_through_the_status_word():
    # FP32-mode scales are not powers of two: the call runs, and the device
    # status word reports FP8Q_ERR_INVALID (then reads back clear)
    x = synth.activation(256, 256, seed=12, name="p2bad.X")
    w = synth.weight(256, 256, seed=13, name="p2bad.W")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x))
    qb, sb = B.fp8q_quant_weight(bf16_to_torch(w))
    assert B.fp8q_sync_status() == 0
    B.fp8q_gemm_pow2(qa, sa, qb, sb)
    assert B.fp8q_sync_status() == B.FP8Q_ERR_INVALID
    assert B.fp8q_sync_status() == 0


def _moe_pow2(oracle, offs, N, K, seed):
    G = offs.size - 1
    M = int(offs[-1])
    x = synth.activation(M, K, seed=seed, name="p2moe.X")
    ws = [synth.weight(N, K, seed=seed + 1 + g, name=f"p2moe.W{g}") for g in range(G)]
    qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=P2)
    qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((G, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for g in range(G):
        B.fp8q_quant_weight(bf16_to_torch(ws[g]), q=qb[g], sb=sb[g], scale_mode=P2)
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act(x, True)
    qb_r = np.stack([oracle.quant_weight(wg, True)[0] for wg in ws])
    sb_r = np.stack([oracle.quant_weight(wg, True)[1] for wg in ws])
    assert_bytes_equal(u8(qb), qb_r, "expert codes")
    assert_scales_equal(f32(sa), sa_r, "A scales")
    return (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r)


@pytest.mark.parametrize("out", ["bf16", "fp32"])
def test_pow2_grouped_small(oracle, out):
    offs = np.array([0, 77, 77, 300, 301, 555], np.int32)   # one empty, one single-row expert
    N, K = 264, 384
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _moe_pow2(oracle, offs, N, K, 21)
    M = int(offs[-1])
    od = B.FP8Q_OUT_BF16 if out == "bf16" else B.FP8Q_OUT_FP32
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    c = torch.full((M + 5, N), 3.0, dtype=dt, device="cuda")   # rows past offs[G] untouched
    a_pad = torch.cat([qa, torch.zeros((5, K), dtype=torch.uint8, device="cuda")])
    sa_pad = torch.cat([sa, torch.ones((K // 128, 5), device="cuda")], dim=1).contiguous()
    B.fp8q_grouped_gemm_pow2(a_pad, sa_pad, qb, sb, torch.from_numpy(offs).cuda(), out_dtype=od,
                             c=c)
    torch.cuda.synchronize()
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r, sb_r, offs)
    _check(c[:M], ref, ad, out == "bf16", "pow2 grouped small")
    assert torch.all(c[M:] == 3.0)


def test_pow2_grouped_moe_workload_sampled(oracle):
    # MoE up-projection with power-of-two scales: 16 experts, 16384 tokens,
    # Dirichlet(0.5) top-1 routing, K=7168 -> N=4096; sampled rows of every expert
    offs = synth.moe_offsets(16384, 16, 0.5, seed=0)
    N, K = 4096, 7168
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _moe_pow2(oracle, offs, N, K, 0)
    c = B.fp8q_grouped_gemm_pow2(qa, sa, qb, sb, torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    rows = set()
    for g in range(16):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            rows |= {lo, hi - 1, (lo + hi) // 2}
    rows = np.array(sorted(rows), np.int64)
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r, sb_r, offs, rows)
    _check(c[torch.from_numpy(rows).cuda()], ref, ad, True, "pow2 moe up-proj")


def test_pow2_accumulate_block_scales(oracle):
    # C (FP32, random start values) += the power-of-two block-scaled product
    M, N, K = 300, 392, 640
    x = synth.activation(M, K, seed=91, name="p2accb.X")
    w = synth.weight(N, K, seed=92, name="p2accb.W")
    (qa, sa, qb, sb), (qa_r, sa_r, qb_r, sb_r) = _fprop_operands(oracle, x, w)
    c0 = np.random.default_rng(93).standard_normal((M, N)).astype(np.float32)
    c = torch.from_numpy(c0).cuda()
    B.fp8q_gemm_pow2_accumulate(qa, sa, qb, sb, c)
    torch.cuda.synchronize()
    prod, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, oracle.BSCALE_BLOCK)
    ref = c0.astype(np.float64) + prod
    tol = 2e-4 * ad + np.abs(ref) * 2.0 ** -24 + 1e-30
    assert_within_tolerance(f64(c), ref, tol, "pow2 accumulate block")
