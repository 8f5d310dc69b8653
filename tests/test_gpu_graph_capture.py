"""Every entry point inside a CUDA graph, and independent calls on two streams
at once: one replay of the captured call writes the same bytes as the same
call run eagerly, and concurrent chains write what they write alone.  The library keeps no host state
that a graph would freeze: tensor maps and arguments travel by value in the
kernel parameters, and the stream is the caller's (here the capture stream).
Outputs are preallocated, so nothing is allocated while capturing.
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import bf16_to_torch

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


def _bytes(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def _eager_vs_graph(fn, make_out):
    """fn(out) writes into the tensors of `out`; eager and replayed results must match."""
    out_e, out_g = make_out(), make_out()
    fn(out_e)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(out_g)
    g.replay()
    torch.cuda.synchronize()
    assert B.fp8q_sync_status() == 0
    for i, (a, b) in enumerate(zip(out_e, out_g)):
        assert np.array_equal(_bytes(a), _bytes(b)), f"output {i} differs after the graph replay"


M, N, K = 256, 384, 512
U8, F32, BF = torch.uint8, torch.float32, torch.bfloat16


def _dev():
    return torch.device("cuda")


def _empty(shape, dt):
    return torch.empty(shape, dtype=dt, device=_dev())


@pytest.mark.parametrize("pow2", [False, True])
def test_quantisers_in_a_graph(pow2):
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    x = bf16_to_torch(synth.activation(M, K, seed=71, name="graph.X"))
    w = bf16_to_torch(synth.weight(N, K, seed=72, name="graph.W"))
    _eager_vs_graph(lambda o: B.fp8q_quant_act(x, scale_mode=mode, q=o[0], sa=o[1]),
                    lambda: (_empty((M, K), U8), _empty((K // 128, M), F32)))
    _eager_vs_graph(lambda o: B.fp8q_quant_act_T(x, scale_mode=mode, qT=o[0], sT=o[1]),
                    lambda: (_empty((K, M), U8), _empty((M // 128, K), F32)))
    _eager_vs_graph(lambda o: B.fp8q_quant_act_T(x, scale_mode=mode, with_rows=True, qT=o[0],
                                                 sT=o[1], q_rows=o[2], s_rows=o[3]),
                    lambda: (_empty((K, M), U8), _empty((M // 128, K), F32),
                             _empty((M, K), U8), _empty((K // 128, M), F32)))
    _eager_vs_graph(lambda o: B.fp8q_quant_weight(w, scale_mode=mode, q=o[0], sb=o[1]),
                    lambda: (_empty((N, K), U8), _empty((N // 128, K // 128), F32)))
    _eager_vs_graph(lambda o: B.fp8q_quant_weight(w, scale_mode=mode, with_transpose=True,
                                                  q=o[0], sb=o[1], qT=o[2]),
                    lambda: (_empty((N, K), U8), _empty((N // 128, K // 128), F32),
                             _empty((K, N), U8)))
    q, s = B.fp8q_quant_act(x, scale_mode=mode)
    _eager_vs_graph(lambda o: B.fp8q_requant_act_T(q, s, scale_mode=mode, qT=o[0], sT=o[1]),
                    lambda: (_empty((K, M), U8), _empty((M // 128, K), F32)))


@pytest.mark.parametrize("pow2", [False, True])
def test_gemms_in_a_graph(pow2):
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    gemm = B.fp8q_gemm_pow2 if pow2 else B.fp8q_gemm
    acc = B.fp8q_gemm_pow2_accumulate if pow2 else B.fp8q_gemm_accumulate
    x = bf16_to_torch(synth.activation(M, K, seed=73, name="graph.X"))
    w = bf16_to_torch(synth.weight(N, K, seed=74, name="graph.W"))
    dy = bf16_to_torch(synth.normal_bf16((M, N), 1e-3, 75, "graph.dY"))
    qa, sa = B.fp8q_quant_act(x, scale_mode=mode)
    qb, sb, qbT = B.fp8q_quant_weight(w, scale_mode=mode, with_transpose=True)
    qdy, sdy = B.fp8q_quant_act(dy, scale_mode=mode)
    qdyT, sdyT = B.fp8q_quant_act_T(dy, scale_mode=mode)
    qxT, sxT = B.fp8q_quant_act_T(x, scale_mode=mode)
    for out_dtype, dt in [(B.FP8Q_OUT_BF16, BF), (B.FP8Q_OUT_FP32, F32)]:
        # Fprop [M][N], Dgrad [M][K], Wgrad [N][K]
        _eager_vs_graph(lambda o: gemm(qa, sa, qb, sb, out_dtype=out_dtype, c=o[0]),
                        lambda: (_empty((M, N), dt),))
        _eager_vs_graph(lambda o: gemm(qdy, sdy, qbT, sb, bscale_kind=B.FP8Q_BSCALE_BLOCK_T,
                                       out_dtype=out_dtype, c=o[0]),
                        lambda: (_empty((M, K), dt),))
        _eager_vs_graph(lambda o: gemm(qdyT, sdyT, qxT, sxT, bscale_kind=B.FP8Q_BSCALE_ROW,
                                       out_dtype=out_dtype, c=o[0]),
                        lambda: (_empty((N, K), dt),))
    # dW += into zeros: one eager call and one replay give the same sums
    _eager_vs_graph(lambda o: acc(qdyT, sdyT, qxT, sxT, o[0], bscale_kind=B.FP8Q_BSCALE_ROW),
                    lambda: (torch.zeros((N, K), dtype=F32, device=_dev()),))


@pytest.mark.parametrize("pow2", [False, True])
def test_grouped_gemm_in_a_graph(pow2):
    mode = B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32
    grouped = B.fp8q_grouped_gemm_pow2 if pow2 else B.fp8q_grouped_gemm
    G, Ne, Ke = 3, 256, 256
    offs = torch.tensor([0, 100, 100, M], dtype=torch.int32, device=_dev())  # one empty expert
    x = bf16_to_torch(synth.activation(M, Ke, seed=76, name="graph.moe.X"))
    qa, sa = B.fp8q_quant_act(x, scale_mode=mode)
    qb = _empty((G, Ne, Ke), U8)
    sb = _empty((G, Ne // 128, Ke // 128), F32)
    for g in range(G):
        wg = bf16_to_torch(synth.weight(Ne, Ke, seed=77 + g, name=f"graph.moe.W{g}"))
        B.fp8q_quant_weight(wg, scale_mode=mode, q=qb[g], sb=sb[g])
    _eager_vs_graph(lambda o: grouped(qa, sa, qb, sb, offs, c=o[0]),
                    lambda: (_empty((M, Ne), BF),))


def test_independent_calls_on_two_streams():
    # two chains of calls on two streams with no dependency between them run
    # concurrently on the GPU; each must write exactly what it writes alone
    # (the library keeps no shared device state besides the error words and
    # the documented scratch of fp8q_quant_tensor_noalloc, not used here)
    x = bf16_to_torch(synth.activation(2048, 1024, seed=81, name="streams.X"))
    w = bf16_to_torch(synth.weight(1024, 1024, seed=82, name="streams.W"))
    dy = bf16_to_torch(synth.normal_bf16((2048, 1024), 1e-3, 83, "streams.dY"))
    q, s = B.fp8q_quant_act(x)
    torch.cuda.synchronize()

    def chain_a(st):
        qT, sT = B.fp8q_requant_act_T(q, s, stream=st)
        out = B.fp8q_quant_act_T(dy, with_rows=True, stream=st)
        _, sbw, qwT = B.fp8q_quant_weight(w, with_transpose=True, stream=st)
        dx = B.fp8q_gemm(out[2], out[3], qwT, sbw, bscale_kind=B.FP8Q_BSCALE_BLOCK_T, stream=st)
        return [qT, sT, *out, dx]

    def chain_b(st):
        qb, sb = B.fp8q_quant_weight(w, stream=st)
        y = B.fp8q_gemm(q, s, qb, sb, stream=st)
        return [qb, sb, y]

    ref = chain_a(torch.cuda.current_stream()) + chain_b(torch.cuda.current_stream())
    torch.cuda.synchronize()
    sa_, sb_ = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        sa_.wait_stream(torch.cuda.current_stream())
        sb_.wait_stream(torch.cuda.current_stream())
        got = chain_a(sa_) + chain_b(sb_)
        torch.cuda.synchronize()
        assert B.fp8q_sync_status() == 0
        for i, (a, b) in enumerate(zip(ref, got)):
            assert np.array_equal(_bytes(a), _bytes(b)), f"output {i} differs when run concurrently"
