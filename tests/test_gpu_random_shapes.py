"""GPU parity on seeded random shapes: every GEMM form (128x128 block scales,
transposed block scales, per-column scales), both output types and both
scale modes, with the operands produced by the library's own quantisers.

Codes and scales must equal the oracle's byte for byte; every product must
lie within |C - C_ref| <= 2e-4 * sum_k |a_k b_k| (+ half a BF16 ulp for BF16
outputs).  C is written into a strided view of a larger buffer whose padding
columns must keep their sentinel.  Shapes (fixed seed): M and N from 1 to
599 (multiples of 8 where a 128x1 quantiser produces the operand, N a
multiple of 128 where the transposed weight codes are the B operand), K a
multiple of 128 up to 640.
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


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = ("block", "block_T", "row")[i % 3]
        fp32_out = (i // 3) % 2 == 1
        pow2 = (i // 6) % 2 == 1
        M = int(rng.integers(1, 600))
        N = int(rng.integers(1, 600))
        K = 128 * int(rng.integers(1, 6))
        if kind == "block_T":
            N = 128 * max(1, N // 128)
        if kind == "row":
            M, N = max(8, M // 8 * 8), max(8, N // 8 * 8)
        out.append(pytest.param(kind, M, N, K, fp32_out, pow2,
                                id=f"{i}-{kind}-{M}x{N}x{K}-{'f32' if fp32_out else 'bf16'}"
                                   f"-{'pow2' if pow2 else 'fp32s'}"))
    return out


@pytest.mark.parametrize("kind,M,N,K,fp32_out,pow2", _cases())
def test_gemm_random_shape(oracle, kind, M, N, K, fp32_out, pow2):
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    tag = f"rand.{kind}.{M}.{N}.{K}"
    if kind == "block":            # Fprop: A 1x128, B 128x128 blocks
        x = synth.activation(M, K, seed=1, name=tag + ".X")
        w = synth.weight(N, K, seed=2, name=tag + ".W")
        qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=mode)
        qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=mode)
        qa_r, sa_r = oracle.quant_act(x, pow2)
        qb_r, sb_r = oracle.quant_weight(w, pow2)
        bk, okind = B.FP8Q_BSCALE_BLOCK, oracle.BSCALE_BLOCK
    elif kind == "block_T":        # Dgrad: A 1x128, B the transposed codes of W [K][N]
        x = synth.normal_bf16((M, K), 1.0, 3, tag + ".dY")
        w = synth.weight(K, N, seed=4, name=tag + ".W")
        qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=mode)
        _, sb, qb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=mode, with_transpose=True)
        qa_r, sa_r = oracle.quant_act(x, pow2)
        qw_r, sb_r = oracle.quant_weight(w, pow2)
        qb_r = np.ascontiguousarray(qw_r.T)
        bk, okind = B.FP8Q_BSCALE_BLOCK_T, oracle.BSCALE_BLOCK_T
    else:                          # Wgrad: both operands 128x1 along K (tokens)
        dy = synth.normal_bf16((K, M), 1e-3, 5, tag + ".dY")
        xx = synth.activation(K, N, seed=6, name=tag + ".X")
        qa, sa = B.fp8q_quant_act_T(bf16_to_torch(dy), scale_mode=mode)
        qb, sb = B.fp8q_quant_act_T(bf16_to_torch(xx), scale_mode=mode)
        qa_r, sa_r = oracle.quant_act_T(dy, pow2)
        qb_r, sb_r = oracle.quant_act_T(xx, pow2)
        bk, okind = B.FP8Q_BSCALE_ROW, oracle.BSCALE_ROW
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qa), qa_r, "A codes")
    assert_scales_equal(f32(sa), sa_r, "A scales")
    assert_bytes_equal(u8(qb), qb_r, "B codes")
    assert_scales_equal(f32(sb), sb_r, "B scales")

    esz = 4 if fp32_out else 2
    ldc = -(-N // (16 // esz)) * (16 // esz) + 16 // esz      # 16-byte rows, plus a guard unit
    dt = torch.float32 if fp32_out else torch.bfloat16
    cbuf = torch.full((M, ldc), 5.0, dtype=dt, device="cuda")
    gemm = B.fp8q_gemm_pow2 if pow2 else B.fp8q_gemm
    gemm(qa, sa, qb, sb, bscale_kind=bk,
         out_dtype=B.FP8Q_OUT_FP32 if fp32_out else B.FP8Q_OUT_BF16, c=cbuf[:, :N])
    torch.cuda.synchronize()
    ref, ad = oracle.gemm_rows(qa_r, sa_r, qb_r, sb_r, okind)
    tol = oracle.gemm_tolerance(ref, ad, not fp32_out)
    assert_within_tolerance(f64(cbuf[:, :N]), ref, tol, f"{kind} {M}x{N}x{K}")
    assert bool((cbuf[:, N:] == 5.0).all()), "padding columns written"


def _grouped_cases(n=12, seed=7):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        G = int(rng.integers(1, 21))
        sizes = rng.integers(0, 300, G)
        sizes[rng.random(G) < 0.2] = 0           # some experts get no tokens
        N = int(rng.integers(1, 400))
        K = 128 * int(rng.integers(1, 5))
        fp32_out = i % 2 == 1
        pow2 = (i // 2) % 2 == 1
        out.append(pytest.param(tuple(int(v) for v in sizes), N, K, fp32_out, pow2,
                                id=f"{i}-G{G}-{int(sizes.sum())}x{N}x{K}"
                                   f"-{'f32' if fp32_out else 'bf16'}-{'pow2' if pow2 else 'fp32s'}"))
    return out


@pytest.mark.parametrize("sizes,N,K,fp32_out,pow2", _grouped_cases())
def test_grouped_gemm_random_shape(oracle, sizes, N, K, fp32_out, pow2):
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    G = len(sizes)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M = int(offs[-1])
    tag = f"rand.moe.{G}.{M}.{N}.{K}"
    x = synth.activation(max(M, 1), K, seed=11, name=tag + ".X")[:M]
    ws = [synth.weight(N, K, seed=12 + g, name=f"{tag}.W{g}") for g in range(G)]
    qb = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    sb = torch.empty((G, (N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    for g in range(G):
        B.fp8q_quant_weight(bf16_to_torch(ws[g]), q=qb[g], sb=sb[g], scale_mode=mode)
    qa_r, sa_r = oracle.quant_act(x, pow2)
    qb_r = np.stack([oracle.quant_weight(wg, pow2)[0] for wg in ws])
    sb_r = np.stack([oracle.quant_weight(wg, pow2)[1] for wg in ws])
    esz = 4 if fp32_out else 2
    ldc = -(-N // (16 // esz)) * (16 // esz) + 16 // esz
    dt = torch.float32 if fp32_out else torch.bfloat16
    cbuf = torch.full((max(M, 1), ldc), 5.0, dtype=dt, device="cuda")
    gemm = B.fp8q_grouped_gemm_pow2 if pow2 else B.fp8q_grouped_gemm
    if M > 0:
        qa, sa = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=mode)
        torch.cuda.synchronize()
        assert_bytes_equal(u8(qa), qa_r, "A codes")
        assert_scales_equal(f32(sa), sa_r, "A scales")
    else:
        qa = torch.empty((0, K), dtype=torch.uint8, device="cuda")
        sa = torch.empty((K // 128, 0), dtype=torch.float32, device="cuda")
    assert_bytes_equal(u8(qb), qb_r, "expert codes")
    assert_scales_equal(f32(sb), sb_r, "expert scales")
    gemm(qa, sa, qb, sb, torch.from_numpy(offs).cuda(),
         out_dtype=B.FP8Q_OUT_FP32 if fp32_out else B.FP8Q_OUT_BF16, c=cbuf[:M, :N])
    torch.cuda.synchronize()
    if M > 0:
        ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r, sb_r, offs)
        tol = oracle.gemm_tolerance(ref, ad, not fp32_out)
        assert_within_tolerance(f64(cbuf[:M, :N]), ref, tol, f"grouped G={G} {M}x{N}x{K}")
    assert bool((cbuf[:, N:] == 5.0).all()), "padding columns written"


@pytest.mark.parametrize("T,C,pow2", [(128, 128, False), (384, 256, True), (256, 640, False),
                                      (640, 384, True)])
def test_requant_random_shape(oracle, T, C, pow2):
    # 128x1 requantisation of the FP8 cache: 64-channel tiles, several per
    # 128-channel row-scale group and a ragged number of tiles per CTA
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    x = synth.activation(T, C, seed=21, name=f"rand.rq.{T}.{C}")
    q, s = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=mode)
    qT, sT = B.fp8q_requant_act_T(q, s, scale_mode=mode)
    torch.cuda.synchronize()
    q_r, s_r = oracle.quant_act(x, pow2)
    qT_r, sT_r = oracle.requant_act_T(q_r, s_r, pow2)
    assert_bytes_equal(u8(qT), qT_r, "requantised codes")
    assert_scales_equal(f32(sT), sT_r, "requantised scales")
