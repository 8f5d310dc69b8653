"""GPU parity at the largest sizes of the MoE and sweep workloads, on the same
inputs and with the same launches as the benchmark.

* MoE down-projection: 16 experts, 16384 tokens routed top-1 by Dirichlet(0.5)
  probabilities, H [16384][2048] ~ N(0,1) quantised 1x128, the stacked expert
  weights [16 x 7168][2048] ~ N(0,0.02) quantised 128x128 in one call, grouped
  GEMM K=2048 -> N=7168, BF16 out; FP32 scales (fp8q_grouped_gemm) and
  power-of-two scales (fp8q_grouped_gemm_pow2, block-scaled MMA).  Power-of-two
  scaling is what the method prescribes for the activation gradient before the
  MoE down-projection (dssusan.co.kr post 91437, paragraph 1).  The codes and
  scales are compared byte for byte; the products on sampled rows of every
  expert, every column, against |C - C_ref| <= 2e-4 * sum_k |a_k b_k| + half a
  BF16 ulp.
* Sweep quantisers at 65536 x 7168 tokens: 128x1 (transposed codes) in both
  scale modes and 1x128 with power-of-two scales; the 128x128 quantiser on
  16 stacked 4096 x 7168 weights in both modes.  Bit-exact.
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


def _mode(mode):
    return B.FP8Q_SCALE_POW2 if mode == "pow2" else B.FP8Q_SCALE_FP32


@pytest.mark.parametrize("mode", MODES)
def test_moe_down_projection_full_size(oracle, mode):
    G, T, d_model, d_in = 16, 16384, 7168, 2048
    p2 = mode == "pow2"
    offs = synth.moe_offsets(T, G, 0.5, seed=0)
    h = synth.normal_bf16((T, d_in), 1.0, 0, "moe.H")
    w = synth.weight(G * d_model, d_in, seed=0, name="moe.Wdown")
    qa, sa = B.fp8q_quant_act(bf16_to_torch(h), scale_mode=_mode(mode))
    qb, sb = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=_mode(mode))
    ggemm = B.fp8q_grouped_gemm_pow2 if p2 else B.fp8q_grouped_gemm
    c = ggemm(qa, sa, qb.view(G, d_model, d_in), sb.view(G, d_model // 128, d_in // 128),
              torch.from_numpy(offs).cuda())
    torch.cuda.synchronize()
    qa_r, sa_r = oracle.quant_act(h, p2)
    qb_r, sb_r = oracle.quant_weight(w, p2)
    assert_bytes_equal(u8(qa), qa_r, "H codes")
    assert_scales_equal(f32(sa), sa_r, "H scales")
    assert_bytes_equal(u8(qb), qb_r, "expert weight codes")
    assert_scales_equal(f32(sb), sb_r, "expert weight scales")
    # every expert's first, middle and last token, plus a seeded sample
    rows = set(np.random.default_rng(3).choice(T, size=256, replace=False).tolist())
    for g in range(G):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            rows |= {lo, hi - 1, (lo + hi) // 2}
    rows = np.array(sorted(rows), np.int64)
    ref, ad = oracle.grouped_gemm_rows(qa_r, sa_r, qb_r.reshape(G, d_model, d_in),
                                       sb_r.reshape(G, d_model // 128, d_in // 128), offs, rows)
    tol = oracle.gemm_tolerance(ref, ad, True)
    assert_within_tolerance(f64(c[torch.from_numpy(rows).cuda()]), ref, tol,
                            f"MoE down-projection ({mode})")


@pytest.mark.parametrize("mode", MODES)
def test_quant_act_T_sweep_65536(oracle, mode):
    x = synth.activation(65536, 7168, seed=0, name="sweep.X65536")
    qT, sT = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=_mode(mode))
    torch.cuda.synchronize()
    qT_ref, sT_ref = oracle.quant_act_T(x, mode == "pow2")
    assert_bytes_equal(u8(qT), qT_ref, "transposed codes")
    assert_scales_equal(f32(sT), sT_ref, "128x1 scales")


def test_quant_act_pow2_sweep_65536(oracle):
    x = synth.activation(65536, 7168, seed=0, name="sweep.X65536")
    q, s = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=B.FP8Q_SCALE_POW2)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act(x, True)
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(s), s_ref, "power-of-two scales")


@pytest.mark.parametrize("mode", MODES)
def test_quant_weight_16_stacked_4096x7168(oracle, mode):
    w = synth.weight(16 * 4096, 7168, seed=0, name="sweep.W65536")
    q, s = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=_mode(mode))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_weight(w, mode == "pow2")
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(s), s_ref, "block scales")
