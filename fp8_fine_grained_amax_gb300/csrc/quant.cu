// quant.cu -- online fine-grained E4M3 quantisers for sm_103a.
//
//   fp8q_quant_act     1x128 tiles (one scale per token per 128 channels)
//   fp8q_quant_act_T   128x1 tiles along tokens, codes written transposed,
//                      optionally also the 1x128 codes from the same read
//   fp8q_quant_weight  128x128 blocks, optionally also the transposed codes
//   fp8q_cast_e4m3     plain FP32 -> E4M3 conversion
//
// Grouping follows dssusan.co.kr post 91437, paragraph 4 (Figure 7 (a)); the
// scale maps each group's max-abs onto 448 ("Deepseek - Not For everyone",
// paragraph 4); power-of-two scales follow paragraph 1 of the dssusan post.
//
// All four kernels are HBM-bound streaming kernels: every BF16 input byte is
// read once with 16-byte non-caching loads, every code and scale written once.
// The max-abs of a group is a packed 16-bit integer max over |BF16| bit
// patterns, reduced with warp shuffles (a 1x128 group lives in 8 lanes) or
// through shared memory (128x1 columns, 128x128 blocks).
#include <cuda_runtime.h>

#include <cstdint>

#include "fp8q.h"
#include "fp8q_host.cuh"
#include "fp8q_ptx.cuh"

namespace fp8q {
namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 8 BF16 values times inv -> 8 E4M3 codes (little-endian order kept).
__device__ __forceinline__ uint2 quantise8(const uint4 &v, float inv) {
  uint2 r;
  r.x = pack_e4m3x4(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv),
                    __fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv));
  r.y = pack_e4m3x4(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv),
                    __fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv));
  return r;
}

// Max of |BF16| over the 16 values of two 16-byte vectors, as FP32 (exact).
// For finite BF16 values the order of the 15-bit magnitude patterns is the
// order of the magnitudes, so a packed unsigned 16-bit max on (bits & 0x7fff)
// finds the max-abs without converting any value.
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 &v) {
  const uint32_t m = 0x7FFF7FFFu;
  return umax16x2(umax16x2(v.x & m, v.y & m), umax16x2(v.z & m, v.w & m));
}
__device__ __forceinline__ float bits_to_f32_max(uint32_t packed) {
  const uint32_t hi = packed >> 16, lo = packed & 0xFFFFu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// ------------------------------------------------------------------ 1x128
// Grid (ceil(M / 64), K / 128).  A CTA handles 64 rows of one 128-wide column
// group.  Eight lanes own one row's group (16 BF16 = 32 bytes each), so a
// warp quantises four rows' groups per scale computation; every thread keeps
// two rows (64 bytes) in flight.
constexpr int kActRowsPerCta = 64;

template <bool kPow2>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t *__restrict__ x, int64_t M,
                                                        int64_t ldx, uint8_t *__restrict__ q,
                                                        int64_t ldq, float *__restrict__ sa,
                                                        int64_t ld_sa) {
  const int g = blockIdx.y;
  const int team = threadIdx.x >> 3, l8 = threadIdx.x & 7;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kActRowsPerCta + team;
  uint4 v[2][2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t m = m0 + u * 32;
    v[u][0] = v[u][1] = make_uint4(0, 0, 0, 0);
    if (m < M) {
      const uint16_t *src = x + m * ldx + g * 128 + l8 * 16;
      v[u][0] = ld_stream_v4(src);
      v[u][1] = ld_stream_v4(src + 8);
    }
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t m = m0 + u * 32;
    uint32_t mb = umax16x2(absmax_bits8(v[u][0]), absmax_bits8(v[u][1]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    float s, inv;
    group_scale(bits_to_f32_max(mb), kPow2, s, inv);
    if (m < M) {
      const uint2 lo = quantise8(v[u][0], inv), hi = quantise8(v[u][1], inv);
      *reinterpret_cast<uint4 *>(q + m * ldq + g * 128 + l8 * 16) = make_uint4(lo.x, lo.y, hi.x, hi.y);
      if (l8 == 0) sa[g * ld_sa + m] = s;
    }
  }
}

// ------------------------------------------------------------------ tiles
// Both tile quantisers below load one 128 x 128 BF16 tile per CTA: 512
// threads, a half-warp per 256-byte row, four rows per thread, 16-byte
// non-caching loads.  The tile goes to shared memory as BF16 pairs, read back
// by columns: thread (cp, tq) owns columns 2cp, 2cp+1 and rows 16tq..16tq+15.
constexpr int kTileThreads = 512;

// ------------------------------------------------------------------ 128x1
// Grid (ceil(C / 128), T / 128).  Optionally quantises each row's 128
// channels (1x128) from registers; then reduces each channel's max-abs over
// the 128 tokens and writes each channel's 128 codes contiguously
// (transposed output).
template <bool kPow2, bool kRows>
__global__ void __launch_bounds__(kTileThreads) quant_act_T_kernel(
    const uint16_t *__restrict__ x, int64_t C, int64_t ldx, uint8_t *__restrict__ qT, int64_t ldqT,
    float *__restrict__ sT, int64_t ld_sT, uint8_t *__restrict__ q_rows, int64_t ldq_rows,
    float *__restrict__ s_rows, int64_t ld_s_rows) {
  __shared__ uint32_t tile[128][64];  // [token][channel pair], BF16x2 words
  __shared__ float red[8][128];
  __shared__ float col_inv[128];

  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * 128;
  const bool chunk_ok = (c0 + l16 * 8) < C;  // C % 8 == 0: chunks are all-in or all-out

  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = make_uint4(0, 0, 0, 0);
    if (chunk_ok) v[i] = ld_stream_v4(x + (t0 + hw + 32 * i) * ldx + c0 + l16 * 8);
  }
  if (kRows) {  // C % 128 == 0 here: every chunk is in range
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t t = t0 + hw + 32 * i;
      uint32_t mb = absmax_bits8(v[i]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      float s, inv;
      group_scale(bits_to_f32_max(mb), kPow2, s, inv);
      *reinterpret_cast<uint2 *>(q_rows + t * ldq_rows + c0 + l16 * 8) = quantise8(v[i], inv);
      if (l16 == 0) s_rows[blockIdx.x * ld_s_rows + t] = s;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4 *>(&tile[hw + 32 * i][l16 * 4]) = v[i];
  __syncthreads();

  const int cp = tid & 63, tq = tid >> 6;
  uint32_t mw = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) mw = umax16x2(mw, tile[tq * 16 + j][cp] & 0x7FFF7FFFu);
  red[tq][2 * cp] = __uint_as_float(mw << 16);
  red[tq][2 * cp + 1] = __uint_as_float(mw & 0xFFFF0000u);
  __syncthreads();
  if (tid < 128) {
    float amax = red[0][tid];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i][tid]);
    float s, inv;
    group_scale(amax, kPow2, s, inv);
    col_inv[tid] = inv;
    if (c0 + tid < C) sT[blockIdx.y * ld_sT + c0 + tid] = s;
  }
  __syncthreads();

  const int64_t c = c0 + 2 * cp;
  if (c < C) {  // c even, C % 8 == 0: c + 1 < C as well
    const float inv_lo = col_inv[2 * cp], inv_hi = col_inv[2 * cp + 1];
    uint32_t out_lo[4], out_hi[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w0 = tile[tq * 16 + 4 * j + 0][cp], w1 = tile[tq * 16 + 4 * j + 1][cp];
      const uint32_t w2 = tile[tq * 16 + 4 * j + 2][cp], w3 = tile[tq * 16 + 4 * j + 3][cp];
      out_lo[j] = pack_e4m3x4(__fmul_rn(bf16_lo(w0), inv_lo), __fmul_rn(bf16_lo(w1), inv_lo),
                              __fmul_rn(bf16_lo(w2), inv_lo), __fmul_rn(bf16_lo(w3), inv_lo));
      out_hi[j] = pack_e4m3x4(__fmul_rn(bf16_hi(w0), inv_hi), __fmul_rn(bf16_hi(w1), inv_hi),
                              __fmul_rn(bf16_hi(w2), inv_hi), __fmul_rn(bf16_hi(w3), inv_hi));
    }
    *reinterpret_cast<uint4 *>(qT + c * ldqT + t0 + tq * 16) =
        make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
    *reinterpret_cast<uint4 *>(qT + (c + 1) * ldqT + t0 + tq * 16) =
        make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
  }
}

// ------------------------------------------------------------------ 128x128
// Grid (K / 128, ceil(N / 128)).  A CTA owns one block: reduces the block
// max-abs (packed max, warp shuffles, then across the 16 warps), writes the
// codes row-wise from registers and, if asked, transposed through shared
// memory.
template <bool kPow2, bool kTrans>
__global__ void __launch_bounds__(kTileThreads) quant_weight_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t ldw, uint8_t *__restrict__ q, int64_t ldq,
    uint8_t *__restrict__ qT, int64_t ldqT, float *__restrict__ sb, int64_t ld_sb) {
  __shared__ uint32_t tile[kTrans ? 128 : 1][64];
  __shared__ uint32_t warp_amax[16];
  __shared__ float blk_inv;

  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 128;

  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t n = n0 + hw + 32 * i;
    v[i] = make_uint4(0, 0, 0, 0);
    if (n < N) v[i] = ld_stream_v4(w + n * ldw + k0 + l16 * 8);
  }
  uint32_t mb = umax16x2(umax16x2(absmax_bits8(v[0]), absmax_bits8(v[1])),
                         umax16x2(absmax_bits8(v[2]), absmax_bits8(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  if ((tid & 31) == 0) warp_amax[tid >> 5] = mb;
  if (kTrans) {
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4 *>(&tile[hw + 32 * i][l16 * 4]) = v[i];
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = warp_amax[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) a = umax16x2(a, warp_amax[i]);
    float s, inv;
    group_scale(bits_to_f32_max(a), kPow2, s, inv);
    sb[blockIdx.y * ld_sb + blockIdx.x] = s;
    blk_inv = inv;
  }
  __syncthreads();
  const float inv = blk_inv;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t n = n0 + hw + 32 * i;
    if (n < N) *reinterpret_cast<uint2 *>(q + n * ldq + k0 + l16 * 8) = quantise8(v[i], inv);
  }
  if (kTrans) {
    // thread (kp, nq): columns k0 + 2kp, k0 + 2kp + 1; rows n0 + 16nq .. + 15
    const int kp = tid & 63, nq = tid >> 6;
    uint32_t out_lo[4], out_hi[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w0 = tile[nq * 16 + 4 * j + 0][kp], w1 = tile[nq * 16 + 4 * j + 1][kp];
      const uint32_t w2 = tile[nq * 16 + 4 * j + 2][kp], w3 = tile[nq * 16 + 4 * j + 3][kp];
      out_lo[j] = pack_e4m3x4(__fmul_rn(bf16_lo(w0), inv), __fmul_rn(bf16_lo(w1), inv),
                              __fmul_rn(bf16_lo(w2), inv), __fmul_rn(bf16_lo(w3), inv));
      out_hi[j] = pack_e4m3x4(__fmul_rn(bf16_hi(w0), inv), __fmul_rn(bf16_hi(w1), inv),
                              __fmul_rn(bf16_hi(w2), inv), __fmul_rn(bf16_hi(w3), inv));
    }
    const int64_t nb0 = n0 + nq * 16;
    uint8_t *row_lo = qT + (k0 + 2 * kp) * ldqT + nb0;
    uint8_t *row_hi = qT + (k0 + 2 * kp + 1) * ldqT + nb0;
    if (nb0 + 16 <= N) {
      *reinterpret_cast<uint4 *>(row_lo) = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
      *reinterpret_cast<uint4 *>(row_hi) = make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
    } else {
      for (int j = 0; j < 16 && nb0 + j < N; ++j) {
        row_lo[j] = static_cast<uint8_t>(out_lo[j >> 2] >> (8 * (j & 3)));
        row_hi[j] = static_cast<uint8_t>(out_hi[j >> 2] >> (8 * (j & 3)));
      }
    }
  }
}

// ------------------------------------------------------------------ cast
__global__ void __launch_bounds__(256) cast_e4m3_kernel(const float *__restrict__ x, int64_t n,
                                                        uint8_t *__restrict__ q) {
  const int64_t n4 = n >> 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += stride) {
    const float4 f = reinterpret_cast<const float4 *>(x)[i];
    reinterpret_cast<uint32_t *>(q)[i] = pack_e4m3x4(f.x, f.y, f.z, f.w);
  }
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
    const int64_t i = n4 * 4 + threadIdx.x;
    q[i] = static_cast<uint8_t>(pack_e4m3x2(x[i], 0.0f) & 0xFF);
  }
}

bool valid_mode(int m) { return m == FP8Q_SCALE_FP32 || m == FP8Q_SCALE_POW2; }

}  // namespace
}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status fp8q_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx, void *q,
                                      int64_t ldq, float *sa, int64_t ld_sa, int scale_mode,
                                      void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  if (M < 0 || K < 0 || K % 128 != 0 || ldx < K || ldq < K || ld_sa < M) return FP8Q_ERR_SHAPE;
  if (K / 128 > 65535) return FP8Q_ERR_SHAPE;
  if (M == 0 || K == 0) return FP8Q_OK;
  if (!x || !q || !sa) return FP8Q_ERR_INVALID;
  if (!aligned16(x) || !aligned16(q) || !aligned4(sa) || ldx % 8 || ldq % 16)
    return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  const dim3 grid(static_cast<unsigned>((M + kActRowsPerCta - 1) / kActRowsPerCta),
                  static_cast<unsigned>(K / 128));
  auto s = static_cast<cudaStream_t>(stream);
  auto xp = static_cast<const uint16_t *>(x);
  auto qp = static_cast<uint8_t *>(q);
  if (scale_mode == FP8Q_SCALE_POW2)
    quant_act_kernel<true><<<grid, 256, 0, s>>>(xp, M, ldx, qp, ldq, sa, ld_sa);
  else
    quant_act_kernel<false><<<grid, 256, 0, s>>>(xp, M, ldx, qp, ldq, sa, ld_sa);
  return launch_status();
}

extern "C" fp8q_status fp8q_quant_act_T(const void *x, int64_t T, int64_t C, int64_t ldx, void *qT,
                                        int64_t ldqT, float *sT, int64_t ld_sT, void *q_rows,
                                        int64_t ldq_rows, float *s_rows, int64_t ld_s_rows,
                                        int scale_mode, void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  const bool rows = q_rows != nullptr;
  if (T < 0 || C < 0 || T % 128 != 0 || C % 8 != 0 || ldx < C || ldqT < T || ld_sT < C)
    return FP8Q_ERR_SHAPE;
  if (rows && (C % 128 != 0 || ldq_rows < C || ld_s_rows < T)) return FP8Q_ERR_SHAPE;
  if (T / 128 > 65535) return FP8Q_ERR_SHAPE;
  if (T == 0 || C == 0) return FP8Q_OK;
  if (!x || !qT || !sT || (rows && !s_rows)) return FP8Q_ERR_INVALID;
  if (!aligned16(x) || !aligned16(qT) || !aligned4(sT) || ldx % 8 || ldqT % 16)
    return FP8Q_ERR_ALIGN;
  if (rows && (!aligned16(q_rows) || !aligned4(s_rows) || ldq_rows % 16)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  const dim3 grid(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>(T / 128));
  auto s = static_cast<cudaStream_t>(stream);
  auto xp = static_cast<const uint16_t *>(x);
  auto qp = static_cast<uint8_t *>(qT);
  auto rp = static_cast<uint8_t *>(q_rows);
  const bool p2 = scale_mode == FP8Q_SCALE_POW2;
  if (p2 && rows)
    quant_act_T_kernel<true, true>
        <<<grid, kTileThreads, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else if (p2)
    quant_act_T_kernel<true, false>
        <<<grid, kTileThreads, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else if (rows)
    quant_act_T_kernel<false, true>
        <<<grid, kTileThreads, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else
    quant_act_T_kernel<false, false>
        <<<grid, kTileThreads, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  return launch_status();
}

extern "C" fp8q_status fp8q_quant_weight(const void *w, int64_t N, int64_t K, int64_t ldw,
                                         void *q, int64_t ldq, void *qT, int64_t ldqT, float *sb,
                                         int64_t ld_sb, int scale_mode, void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  const bool trans = qT != nullptr;
  if (N < 0 || K < 0 || K % 128 != 0 || ldw < K || ldq < K || ld_sb < K / 128)
    return FP8Q_ERR_SHAPE;
  if (trans && ldqT < N) return FP8Q_ERR_SHAPE;
  if ((N + 127) / 128 > 65535) return FP8Q_ERR_SHAPE;
  if (N == 0 || K == 0) return FP8Q_OK;
  if (!w || !q || !sb) return FP8Q_ERR_INVALID;
  if (!aligned16(w) || !aligned16(q) || !aligned4(sb) || ldw % 8 || ldq % 16)
    return FP8Q_ERR_ALIGN;
  if (trans && (!aligned16(qT) || ldqT % 16)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  const dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>((N + 127) / 128));
  auto s = static_cast<cudaStream_t>(stream);
  auto wp = static_cast<const uint16_t *>(w);
  auto qp = static_cast<uint8_t *>(q);
  auto tp = static_cast<uint8_t *>(qT);
  const bool p2 = scale_mode == FP8Q_SCALE_POW2;
  if (p2 && trans)
    quant_weight_kernel<true, true><<<grid, kTileThreads, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else if (p2)
    quant_weight_kernel<true, false><<<grid, kTileThreads, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else if (trans)
    quant_weight_kernel<false, true><<<grid, kTileThreads, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else
    quant_weight_kernel<false, false>
        <<<grid, kTileThreads, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  return launch_status();
}

extern "C" fp8q_status fp8q_cast_e4m3(const float *x, int64_t n, void *q, void *stream) {
  if (n < 0) return FP8Q_ERR_SHAPE;
  if (n == 0) return FP8Q_OK;
  if (!x || !q) return FP8Q_ERR_INVALID;
  if (!aligned16(x) || !aligned16(q)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  const int64_t n4 = (n >> 2) > 0 ? (n >> 2) : 1;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
  if (blocks > cap) blocks = cap;
  cast_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, n, static_cast<uint8_t *>(q));
  return launch_status();
}
