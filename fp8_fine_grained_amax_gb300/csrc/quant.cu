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
// The max-abs of a group is reduced with warp shuffles (1x128 groups live in
// one half-warp) or through shared memory (128x1 columns, 128x128 blocks).
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

__device__ __forceinline__ float absmax8(const uint4 &v) {
  return fmaxf(fmaxf(absmax_bf16x2(v.x), absmax_bf16x2(v.y)),
               fmaxf(absmax_bf16x2(v.z), absmax_bf16x2(v.w)));
}

// Max over the 16 lanes of a half-warp (xor offsets < 16 stay in the half).
__device__ __forceinline__ float halfwarp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
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

// ------------------------------------------------------------------ 1x128
// Grid (ceil(M / 64), K / 128).  A CTA handles 64 rows of one 128-wide column
// group; each half-warp owns one row's group at a time (16 lanes x 8 BF16),
// four rows per thread in flight.
constexpr int kActRowsPerCta = 64;
constexpr int kActUnroll = 4;

template <bool kPow2>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t *__restrict__ x, int64_t M,
                                                        int64_t ldx, uint8_t *__restrict__ q,
                                                        int64_t ldq, float *__restrict__ sa,
                                                        int64_t ld_sa) {
  const int g = blockIdx.y;
  const int hw = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * kActRowsPerCta + hw;
  uint4 v[kActUnroll];
#pragma unroll
  for (int u = 0; u < kActUnroll; ++u) {
    const int64_t m = m0 + u * 16;
    v[u] = make_uint4(0, 0, 0, 0);
    if (m < M) v[u] = ld_stream_v4(x + m * ldx + g * 128 + l16 * 8);
  }
#pragma unroll
  for (int u = 0; u < kActUnroll; ++u) {
    const int64_t m = m0 + u * 16;
    const float amax = halfwarp_max(absmax8(v[u]));
    float s, inv;
    group_scale(amax, kPow2, s, inv);
    if (m < M) {
      *reinterpret_cast<uint2 *>(q + m * ldq + g * 128 + l16 * 8) = quantise8(v[u], inv);
      if (l16 == 0) sa[g * ld_sa + m] = s;
    }
  }
}

// ------------------------------------------------------------------ 128x1
// Grid (ceil(C / 128), T / 128).  A CTA loads a 128-token x 128-channel tile
// once into registers (row-wise, 16-byte loads) and shared memory, then
//  - optionally quantises each row's 128 channels (1x128) from registers,
//  - reduces each channel's max-abs over the 128 tokens,
//  - writes each channel's 128 codes contiguously (transposed output).
template <bool kPow2, bool kRows>
__global__ void __launch_bounds__(256) quant_act_T_kernel(
    const uint16_t *__restrict__ x, int64_t C, int64_t ldx, uint8_t *__restrict__ qT, int64_t ldqT,
    float *__restrict__ sT, int64_t ld_sT, uint8_t *__restrict__ q_rows, int64_t ldq_rows,
    float *__restrict__ s_rows, int64_t ld_s_rows) {
  __shared__ uint32_t tile[128][64];  // [token][channel pair], BF16x2 words
  __shared__ float red[4][128];
  __shared__ float col_inv[128];

  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t t0 = static_cast<int64_t>(blockIdx.y) * 128;
  const bool chunk_ok = (c0 + l16 * 8) < C;  // C % 8 == 0: chunks are all-in or all-out

  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = hw + 16 * i;
    v[i] = make_uint4(0, 0, 0, 0);
    if (chunk_ok) v[i] = ld_stream_v4(x + (t0 + r) * ldx + c0 + l16 * 8);
  }

  if (kRows) {  // C % 128 == 0 here: every chunk is in range
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t t = t0 + hw + 16 * i;
      const float amax = halfwarp_max(absmax8(v[i]));
      float s, inv;
      group_scale(amax, kPow2, s, inv);
      *reinterpret_cast<uint2 *>(q_rows + t * ldq_rows + c0 + l16 * 8) = quantise8(v[i], inv);
      if (l16 == 0) s_rows[blockIdx.x * ld_s_rows + t] = s;
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(&tile[hw + 16 * i][l16 * 4]) = v[i];
  __syncthreads();

  const int cp = tid & 63, tq = tid >> 6;  // channel pair, quarter of the tokens
  float m_lo = 0.0f, m_hi = 0.0f;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const uint32_t w = tile[tq * 32 + j][cp];
    m_lo = fmaxf(m_lo, fabsf(bf16_lo(w)));
    m_hi = fmaxf(m_hi, fabsf(bf16_hi(w)));
  }
  red[tq][2 * cp] = m_lo;
  red[tq][2 * cp + 1] = m_hi;
  __syncthreads();
  if (tid < 128) {
    const float amax = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
    float s, inv;
    group_scale(amax, kPow2, s, inv);
    col_inv[tid] = inv;
    if (c0 + tid < C) sT[blockIdx.y * ld_sT + c0 + tid] = s;
  }
  __syncthreads();

  const int64_t c = c0 + 2 * cp;
  if (c < C) {  // c even, C % 8 == 0: c + 1 < C as well
    const float inv_lo = col_inv[2 * cp], inv_hi = col_inv[2 * cp + 1];
    uint32_t out_lo[8], out_hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w0 = tile[tq * 32 + 4 * j + 0][cp], w1 = tile[tq * 32 + 4 * j + 1][cp];
      const uint32_t w2 = tile[tq * 32 + 4 * j + 2][cp], w3 = tile[tq * 32 + 4 * j + 3][cp];
      out_lo[j] = pack_e4m3x4(__fmul_rn(bf16_lo(w0), inv_lo), __fmul_rn(bf16_lo(w1), inv_lo),
                              __fmul_rn(bf16_lo(w2), inv_lo), __fmul_rn(bf16_lo(w3), inv_lo));
      out_hi[j] = pack_e4m3x4(__fmul_rn(bf16_hi(w0), inv_hi), __fmul_rn(bf16_hi(w1), inv_hi),
                              __fmul_rn(bf16_hi(w2), inv_hi), __fmul_rn(bf16_hi(w3), inv_hi));
    }
    uint4 *dst_lo = reinterpret_cast<uint4 *>(qT + c * ldqT + t0 + tq * 32);
    uint4 *dst_hi = reinterpret_cast<uint4 *>(qT + (c + 1) * ldqT + t0 + tq * 32);
    dst_lo[0] = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
    dst_lo[1] = make_uint4(out_lo[4], out_lo[5], out_lo[6], out_lo[7]);
    dst_hi[0] = make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
    dst_hi[1] = make_uint4(out_hi[4], out_hi[5], out_hi[6], out_hi[7]);
  }
}

// ------------------------------------------------------------------ 128x128
// Grid (K / 128, ceil(N / 128)).  A CTA owns one block: loads it once into
// registers, reduces the block max-abs (warp shuffles, then across warps),
// writes the codes row-wise and, if asked, transposed through shared memory.
template <bool kPow2, bool kTrans>
__global__ void __launch_bounds__(256) quant_weight_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t ldw, uint8_t *__restrict__ q, int64_t ldq,
    uint8_t *__restrict__ qT, int64_t ldqT, float *__restrict__ sb, int64_t ld_sb) {
  __shared__ uint32_t tile[kTrans ? 128 : 1][64];
  __shared__ float warp_amax[8];
  __shared__ float blk_inv;

  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 128;

  uint4 v[8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = n0 + hw + 16 * i;
    v[i] = make_uint4(0, 0, 0, 0);
    if (n < N) v[i] = ld_stream_v4(w + n * ldw + k0 + l16 * 8);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, absmax8(v[i]));
  amax = warp_max(amax);
  if ((tid & 31) == 0) warp_amax[tid >> 5] = amax;
  if (kTrans) {
#pragma unroll
    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(&tile[hw + 16 * i][l16 * 4]) = v[i];
  }
  __syncthreads();
  if (tid == 0) {
    float a = warp_amax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, warp_amax[i]);
    float s, inv;
    group_scale(a, kPow2, s, inv);
    sb[blockIdx.y * ld_sb + blockIdx.x] = s;
    blk_inv = inv;
  }
  __syncthreads();
  const float inv = blk_inv;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t n = n0 + hw + 16 * i;
    if (n < N) *reinterpret_cast<uint2 *>(q + n * ldq + k0 + l16 * 8) = quantise8(v[i], inv);
  }
  if (kTrans) {
    // thread (kp, nq): columns k0 + 2kp, k0 + 2kp + 1; rows n0 + 32nq .. + 31
    const int kp = tid & 63, nq = tid >> 6;
    uint32_t out_lo[8], out_hi[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w0 = tile[nq * 32 + 4 * j + 0][kp], w1 = tile[nq * 32 + 4 * j + 1][kp];
      const uint32_t w2 = tile[nq * 32 + 4 * j + 2][kp], w3 = tile[nq * 32 + 4 * j + 3][kp];
      out_lo[j] = pack_e4m3x4(__fmul_rn(bf16_lo(w0), inv), __fmul_rn(bf16_lo(w1), inv),
                              __fmul_rn(bf16_lo(w2), inv), __fmul_rn(bf16_lo(w3), inv));
      out_hi[j] = pack_e4m3x4(__fmul_rn(bf16_hi(w0), inv), __fmul_rn(bf16_hi(w1), inv),
                              __fmul_rn(bf16_hi(w2), inv), __fmul_rn(bf16_hi(w3), inv));
    }
    const int64_t nb0 = n0 + nq * 32;
    uint8_t *row_lo = qT + (k0 + 2 * kp) * ldqT + nb0;
    uint8_t *row_hi = qT + (k0 + 2 * kp + 1) * ldqT + nb0;
    if (nb0 + 32 <= N) {
      reinterpret_cast<uint4 *>(row_lo)[0] = make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
      reinterpret_cast<uint4 *>(row_lo)[1] = make_uint4(out_lo[4], out_lo[5], out_lo[6], out_lo[7]);
      reinterpret_cast<uint4 *>(row_hi)[0] = make_uint4(out_hi[0], out_hi[1], out_hi[2], out_hi[3]);
      reinterpret_cast<uint4 *>(row_hi)[1] = make_uint4(out_hi[4], out_hi[5], out_hi[6], out_hi[7]);
    } else {
      for (int j = 0; j < 32 && nb0 + j < N; ++j) {
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
        <<<grid, 256, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else if (p2)
    quant_act_T_kernel<true, false>
        <<<grid, 256, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else if (rows)
    quant_act_T_kernel<false, true>
        <<<grid, 256, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
  else
    quant_act_T_kernel<false, false>
        <<<grid, 256, 0, s>>>(xp, C, ldx, qp, ldqT, sT, ld_sT, rp, ldq_rows, s_rows, ld_s_rows);
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
    quant_weight_kernel<true, true><<<grid, 256, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else if (p2)
    quant_weight_kernel<true, false><<<grid, 256, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else if (trans)
    quant_weight_kernel<false, true><<<grid, 256, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
  else
    quant_weight_kernel<false, false>
        <<<grid, 256, 0, s>>>(wp, N, ldw, qp, ldq, tp, ldqT, sb, ld_sb);
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
