"""GPU parity of the quantisers against the CPU oracle: bytes and scales bit-exact.

Every case runs the CUDA path through the C ABI (the Python binding of
libfp8q) on seeded synthetic inputs and compares every code and every scale
with the oracle on the same inputs.
"""
import numpy as np
import pytest

from fp8_fine_grained_amax_gb300 import synth
from _util import assert_bytes_equal, assert_scales_equal, bf16_to_torch, f32, u8

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


def _mode(pow2):
    return B.FP8Q_SCALE_POW2 if pow2 else B.FP8Q_SCALE_FP32


def _special_rows(x):
    """Overwrite a few groups with edge cases: zeros, -0, a tiny max-abs, a
    group whose max-abs is exactly 448 * 2^j, huge values."""
    x = x.copy()
    if x.shape[0] >= 4 and x.shape[1] >= 256:
        x[0, :128] = 0
        x[1, 128:256] = 0x8000                         # -0.0
        x[2, :128] = 0x0001                            # smallest BF16 subnormal
        x[3, :128] = 0x43E0                            # 448.0
        x[3, 5] = 0xC3E0                               # -448.0
    if x.shape[0] >= 6 and x.shape[1] >= 128:
        x[5, :128] = 0x7F7F                            # largest finite BF16
    return x


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M,K", [(256, 512), (1, 128), (63, 384), (200, 1024), (4096, 7168)])
def test_quant_act(oracle, M, K, pow2):
    x = _special_rows(synth.activation(M, K, seed=100 + M))
    q_ref, s_ref = oracle.quant_act(x, pow2)
    q, s = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=_mode(pow2))
    torch.cuda.synchronize()
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(s), s_ref, "scales")


def test_quant_act_strided(oracle):
    # row strides larger than K, and a scale array with ld_sa > M
    M, K, ldx = 100, 256, 384
    full = synth.activation(M, ldx, seed=7)
    x_dev = bf16_to_torch(full)[:, :K]
    q = torch.full((M, 272), 0xAB, dtype=torch.uint8, device="cuda")[:, :K]
    sa = torch.full((K // 128, 104), -1.0, dtype=torch.float32, device="cuda")
    B.fp8q_quant_act(x_dev, q=q, sa=sa[:, :M])
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act(np.ascontiguousarray(full[:, :K]))
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(sa[:, :M]), s_ref, "scales")
    assert np.all(f32(sa[:, M:]) == -1.0), "wrote past M in the scale rows"
    qfull = torch.as_strided(q, (M, 272), (272, 1))
    assert np.all(u8(qfull)[:, K:] == 0xAB), "wrote past K in the code rows"


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("T,C,rows", [(128, 8, False), (256, 200, False), (384, 256, True),
                                      (8192, 2048, True), (8192, 7168, False)])
def test_quant_act_T(oracle, T, C, rows, pow2):
    x = _special_rows(synth.activation(T, C, seed=200 + C))
    qT_ref, sT_ref = oracle.quant_act_T(x, pow2)
    out = B.fp8q_quant_act_T(bf16_to_torch(x), scale_mode=_mode(pow2), with_rows=rows)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(out[0]), qT_ref, "transposed codes")
    assert_scales_equal(f32(out[1]), sT_ref, "128x1 scales")
    if rows:
        q_ref, s_ref = oracle.quant_act(x, pow2)
        assert_bytes_equal(u8(out[2]), q_ref, "1x128 codes (fused)")
        assert_scales_equal(f32(out[3]), s_ref, "1x128 scales (fused)")


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("N,K,trans", [(256, 512, True), (300, 384, True), (1, 128, True),
                                       (130, 256, False), (7168, 7168, True),
                                       (2048, 7168, True), (2000, 4096, True)])
def test_quant_weight(oracle, N, K, trans, pow2):
    w = _special_rows(synth.weight(N, K, seed=300 + N))
    q_ref, s_ref = oracle.quant_weight(w, pow2)
    qT = None
    if trans:
        # the transposed rows need a leading dimension that is a multiple of 16;
        # pad it, and check that the padding is left alone
        ldqT = (N + 15) // 16 * 16
        qT_buf = torch.full((K, ldqT + 16), 0x5A, dtype=torch.uint8, device="cuda")
        qT = qT_buf[:, :N]
    out = B.fp8q_quant_weight(bf16_to_torch(w), scale_mode=_mode(pow2), with_transpose=trans,
                              qT=qT)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(out[0]), q_ref, "codes")
    assert_scales_equal(f32(out[1]), s_ref, "block scales")
    if trans:
        assert_bytes_equal(u8(out[2]), np.ascontiguousarray(q_ref.T), "transposed codes")
        assert np.all(u8(qT_buf)[:, N:] == 0x5A), "wrote past N in the transposed rows"


def test_quant_weight_transpose_needs_aligned_ld():
    w = torch.zeros((300, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.FP8QError) as e:
        B.fp8q_quant_weight(w, with_transpose=True)        # ldqT = 300
    assert e.value.status == B.FP8Q_ERR_ALIGN


def test_quant_act_full_sweep_size(oracle):
    # the largest activation of the sweep workload, tokens 65536 x 7168
    x = synth.activation(65536, 7168, seed=0, name="sweep.X65536")
    q_ref, s_ref = oracle.quant_act(x)
    q, s = B.fp8q_quant_act(bf16_to_torch(x))
    torch.cuda.synchronize()
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(s), s_ref, "scales")


def test_empty_inputs():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = B.fp8q_quant_act(x)
    assert q.shape == (0, 256) and s.shape == (2, 0)
    w = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    q, s = B.fp8q_quant_weight(w)
    assert q.shape == (0, 128)


def test_argument_errors():
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")   # K % 128 != 0
    with pytest.raises(B.FP8QError) as e:
        B.fp8q_quant_act(x)
    assert e.value.status == B.FP8Q_ERR_SHAPE
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.FP8QError) as e:
        B.fp8q_quant_act(x, scale_mode=7)
    assert e.value.status == B.FP8Q_ERR_INVALID
    xb = torch.zeros((4 * 128 + 1,), dtype=torch.bfloat16, device="cuda")[1:].view(4, 128)
    with pytest.raises(B.FP8QError) as e:
        B.fp8q_quant_act(xb)
    assert e.value.status == B.FP8Q_ERR_ALIGN


def test_cast_exhaustive(oracle):
    # every FP32 bit pattern, in chunks of 2^28: the kernel's conversion against
    # the oracle's.  NaN inputs must give a NaN code (either sign); every other
    # input must match exactly.
    n = 1 << 28
    q = torch.empty(n, dtype=torch.uint8, device="cuda")
    for chunk in range(16):
        bits = np.arange(n, dtype=np.uint32) + np.uint32(chunk * n)
        xs = bits.view(np.float32)
        x = torch.from_numpy(bits.view(np.int32)).to("cuda").view(torch.float32)
        B.fp8q_cast_e4m3(x, q=q)
        got = u8(q)
        want = oracle.e4m3_encode(xs)
        nan = np.isnan(xs)
        assert np.all((got[nan] & 0x7F) == 0x7F), f"chunk {chunk}: NaN not kept"
        assert_bytes_equal(got[~nan], want[~nan], f"chunk {chunk}")


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("T,C", [(128, 128), (384, 256), (8192, 7168)])
def test_requant_act_T_from_fp8_cache(oracle, T, C, pow2):
    # the forward pass's cached 1x128 codes (FP32 or power-of-two scales) are
    # requantised 128x1 for the backward pass
    x = _special_rows(synth.activation(T, C, seed=500 + C))
    q_r, s_r = oracle.quant_act(x, pow2)
    qT_ref, sT_ref = oracle.requant_act_T(q_r, s_r, pow2)
    q, s = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=_mode(pow2))
    qT, sT = B.fp8q_requant_act_T(q, s, scale_mode=_mode(pow2))
    torch.cuda.synchronize()
    assert_bytes_equal(u8(q), q_r, "cached codes")
    assert_bytes_equal(u8(qT), qT_ref, "requantised codes")
    assert_scales_equal(f32(sT), sT_ref, "requantised scales")


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("T,C,rows", [(256, 200, False), (384, 256, True)])
def test_quant_act_T_strided(oracle, T, C, rows, pow2):
    # every operand a view of a wider buffer: x (ldx > C), qT (ldqT > T),
    # sT (ld_sT > C) and, with the fused rows, q_rows (ldq > C) and s_rows
    # (ld_s_rows > T); the padding must keep its sentinel
    full = _special_rows(synth.activation(T, C + 64, seed=250 + C))
    x = bf16_to_torch(full)[:, :C]
    qT = torch.full((C, T + 32), 0xA5, dtype=torch.uint8, device="cuda")
    sT = torch.full((T // 128, C + 24), -3.0, dtype=torch.float32, device="cuda")
    kw = {}
    if rows:
        kw = dict(q_rows=torch.full((T, C + 48), 0x5A, dtype=torch.uint8, device="cuda")[:, :C],
                  s_rows=torch.full((C // 128, T + 12), -5.0, dtype=torch.float32,
                                    device="cuda")[:, :T])
    out = B.fp8q_quant_act_T(x, scale_mode=_mode(pow2), with_rows=rows, qT=qT[:, :T],
                             sT=sT[:, :C], **kw)
    torch.cuda.synchronize()
    xs = np.ascontiguousarray(full[:, :C])
    qT_ref, sT_ref = oracle.quant_act_T(xs, pow2)
    assert_bytes_equal(u8(out[0]), qT_ref, "transposed codes")
    assert_scales_equal(f32(out[1]), sT_ref, "128x1 scales")
    assert np.all(u8(qT)[:, T:] == 0xA5), "wrote past T in the transposed rows"
    assert np.all(f32(sT)[:, C:] == -3.0), "wrote past C in the scale rows"
    if rows:
        q_ref, s_ref = oracle.quant_act(xs, pow2)
        assert_bytes_equal(u8(out[2]), q_ref, "1x128 codes (fused)")
        assert_scales_equal(f32(out[3]), s_ref, "1x128 scales (fused)")
        qr = torch.as_strided(out[2], (T, C + 48), (C + 48, 1))
        sr = torch.as_strided(out[3], (C // 128, T + 12), (T + 12, 1))
        assert np.all(u8(qr)[:, C:] == 0x5A), "wrote past C in the fused code rows"
        assert np.all(f32(sr)[:, T:] == -5.0), "wrote past T in the fused scale rows"


@pytest.mark.parametrize("pow2", [False, True])
def test_requant_act_T_strided(oracle, pow2):
    # cached codes and row scales as views of wider buffers (ldq > C,
    # ld_s_rows > T, not a multiple of 4), outputs likewise (ldqT > T,
    # ld_sT > C); three 128-channel groups, three token blocks
    T, C = 384, 384
    x = _special_rows(synth.activation(T, C, seed=510))
    q = torch.full((T, C + 32), 0x11, dtype=torch.uint8, device="cuda")[:, :C]
    s = torch.full((C // 128, T + 13), -7.0, dtype=torch.float32, device="cuda")[:, :T]
    B.fp8q_quant_act(bf16_to_torch(x), scale_mode=_mode(pow2), q=q, sa=s)
    qT = torch.full((C, T + 48), 0x22, dtype=torch.uint8, device="cuda")
    sT = torch.full((T // 128, C + 8), -9.0, dtype=torch.float32, device="cuda")
    B.fp8q_requant_act_T(q, s, scale_mode=_mode(pow2), qT=qT[:, :T], sT=sT[:, :C])
    torch.cuda.synchronize()
    q_r, s_r = oracle.quant_act(x, pow2)
    qT_ref, sT_ref = oracle.requant_act_T(q_r, s_r, pow2)
    assert_bytes_equal(u8(q), q_r, "cached codes")
    assert_bytes_equal(u8(qT[:, :T]), qT_ref, "requantised codes")
    assert_scales_equal(f32(sT[:, :C]), sT_ref, "requantised scales")
    assert np.all(u8(qT)[:, T:] == 0x22), "wrote past T in the requantised rows"
    assert np.all(f32(sT)[:, C:] == -9.0), "wrote past C in the requantised scales"


@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("M,K", [(1, 8), (63, 200), (256, 1024), (4096, 7168)])
def test_quant_tensor(oracle, M, K, pow2):
    x = _special_rows(synth.activation(M, K, seed=600 + M)) if K >= 256 else \
        synth.activation(M, K, seed=600 + M)
    q_ref, s_ref = oracle.quant_tensor(x, pow2)
    ws = torch.full((B.fp8q_quant_tensor_workspace_bytes(M, K),), 0xEE, dtype=torch.uint8,
                    device="cuda")   # stale contents must not matter
    q, s = B.fp8q_quant_tensor(bf16_to_torch(x), scale_mode=_mode(pow2), workspace=ws)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(q), q_ref, "codes")
    assert_scales_equal(f32(s), np.array([s_ref], np.float32), "tensor scale")


def test_quant_tensor_workspace_too_small():
    x = torch.zeros((200, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty((4,), dtype=torch.uint8, device="cuda")     # needs 4 partials
    with pytest.raises(B.FP8QError) as e:
        B.fp8q_quant_tensor(x, workspace=ws)
    assert e.value.status == B.FP8Q_ERR_SHAPE


@pytest.mark.parametrize("pow2", [False, True])
def test_scale_of_every_bf16_max_abs(oracle, pow2):
    # Every positive finite BF16 value (0x0001 .. 0x7F7F) is the max-abs of one
    # 1x128 group and of one 128x1 channel group: the scales (and the codes of
    # the group's other values) must equal the oracle's for every possible
    # max-abs, the subnormal ones going through the 2^-116 floor.
    vals = np.arange(1, 0x7F80, dtype=np.uint16)
    M = vals.size
    x = np.zeros((M, 128), np.uint16)
    x[:, 0] = vals
    x[:, 77] = vals | 0x8000            # the same magnitude, negative
    x[:, 5] = vals >> 1                 # smaller values of the same group
    q_ref, s_ref = oracle.quant_act(x, pow2)
    q, s = B.fp8q_quant_act(bf16_to_torch(x), scale_mode=_mode(pow2))
    torch.cuda.synchronize()
    assert_bytes_equal(u8(q), q_ref, "1x128 codes")
    assert_scales_equal(f32(s), s_ref, "1x128 scales")
    C = (M + 7) // 8 * 8                # 128x1: one channel per value
    xt = np.zeros((128, C), np.uint16)
    xt[3, :M] = vals
    xt[100, :M] = vals | 0x8000
    xt[64, :M] = vals >> 2
    qT_ref, sT_ref = oracle.quant_act_T(xt, pow2)
    qT, sT = B.fp8q_quant_act_T(bf16_to_torch(xt), scale_mode=_mode(pow2))
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qT), qT_ref, "128x1 codes")
    assert_scales_equal(f32(sT), sT_ref, "128x1 scales")
    # the fused 1x128 rows of the 128x1 quantiser: the same rows, padded with
    # zero rows to a multiple of 128 tokens
    T = (M + 127) // 128 * 128
    xr = np.zeros((T, 128), np.uint16)
    xr[:M] = x
    qr_ref, sr_ref = oracle.quant_act(xr, pow2)
    _, _, qr, sr = B.fp8q_quant_act_T(bf16_to_torch(xr), scale_mode=_mode(pow2), with_rows=True)
    torch.cuda.synchronize()
    assert_bytes_equal(u8(qr), qr_ref, "fused 1x128 codes")
    assert_scales_equal(f32(sr), sr_ref, "fused 1x128 scales")
