// quant.cu -- online fine-grained E4M3 quantisers for sm_103a.
//
//   fp8q_quant_act      1x128 tiles (one scale per token per 128 channels)
//   fp8q_quant_act_T    128x1 tiles along tokens, codes written transposed,
//                       optionally also the 1x128 codes from the same read
//   fp8q_requant_act_T  128x1 tiles from FP8-cached 1x128 activations
//   fp8q_quant_weight   128x128 blocks, optionally also the transposed codes
//   fp8q_quant_tensor   one scale per tensor (comparison), with a caller
//                       workspace or (_noalloc) a fixed static scratch
//   fp8q_cast_e4m3      plain FP32 -> E4M3 conversion
//
// Grouping follows dssusan.co.kr post 91437, paragraph 4 (Figure 7 (a)); the
// scale maps each group's max-abs onto 448 ("Deepseek - Not For everyone",
// paragraph 4); power-of-two scales follow paragraph 1 of the dssusan post.
//
// They are HBM-bound streaming kernels: every input byte is read once (16-byte
// non-caching loads or TMA tiles), every code and scale written once.  The
// max-abs of a group is a packed 16-bit integer max over |BF16| bit patterns,
// reduced with warp shuffles (a 1x128 group lives in 8 lanes, a 128x1 channel
// in 4 lanes after ldmatrix.trans) or across warps (128x128 blocks).  The
// transposed outputs leave through TMA tensor stores of swizzled shared-memory
// tiles.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8q.h"
#include "fp8q_host.cuh"
#include "fp8q_ptx.cuh"

namespace fp8q {

// Device status word of the quantisers: 0, or FP8Q_ERR_TIMEOUT after one of
// their bounded waits gave up (read and cleared by fp8q_sync_status()).
__device__ int g_quant_status;

fp8q_status quant_status_take(cudaStream_t s) {
  int v = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_quant_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_quant_status, &zero, sizeof(int)) != cudaSuccess) return FP8Q_ERR_CUDA;
  }
  return static_cast<fp8q_status>(v);
}

namespace {

// Wait for a phase for at most 1 s regardless of any abort (own copies only).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > 1000000000ull) return;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two BF16 values (one 32-bit word) times inv -> two E4M3 codes: one packed
// FP32 multiply (mul.rn.f32x2 rounds each lane as __fmul_rn does and keeps
// subnormals) and one convert.
__device__ __forceinline__ uint32_t quantise2(uint32_t w, uint64_t inv2) {
  const float2 p = unpack_f32x2(fmul2(pack_f32x2(bf16_lo(w), bf16_hi(w)), inv2));
  return pack_e4m3x2(p.x, p.y);
}

// 8 BF16 values times inv -> 8 E4M3 codes (little-endian order kept).
__device__ __forceinline__ uint2 quantise8(const uint4 &v, float inv) {
  const uint64_t inv2 = pack_f32x2(inv, inv);
  uint2 r;
  r.x = quantise2(v.x, inv2) | (quantise2(v.y, inv2) << 16);
  r.y = quantise2(v.z, inv2) | (quantise2(v.w, inv2) << 16);
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

// FP32-mode scales of BF16 max-abs values from two 128-entry tables.  After
// the 2^-116 floor a BF16 max-abs is a = (1 + m/128) * 2^E with E >= -116,
// and a / 448 = fl(M / 448) * 2^E, 448 / a = fl(448 / M) * 2^-E exactly, M =
// 1 + m/128: scaling by a power of two commutes with rounding while the
// result stays normal, and s and inv stay within [2^-125, 2^125].  The
// tables hold the IEEE quotients (__fdiv_rn) of the 128 mantissas; an
// infinite or NaN max-abs goes through group_scale() itself.
struct ScaleTables {
  uint32_t s[128];    // bits of fl(M / 448)
  uint32_t inv[128];  // bits of fl(448 / M)
};

// Threads 0..127 fill entry tid; the caller synchronises before use.
__device__ __forceinline__ void scale_tables_init(ScaleTables &t, int tid) {
  if (tid < 128) {
    const float M = 1.0f + static_cast<float>(tid) * 0x1p-7f;
    t.s[tid] = __float_as_uint(__fdiv_rn(M, 448.0f));
    t.inv[tid] = __float_as_uint(__fdiv_rn(448.0f, M));
  }
}

// Scale of a group from the packed 16-bit max-abs patterns of two BF16 lanes
// (as umax16x2 leaves them): equal to group_scale(bits_to_f32_max(packed)).
__device__ __forceinline__ void group_scale_bf16(const ScaleTables &t, uint32_t packed, bool pow2,
                                                 float &s, float &inv) {
  if (pow2) {
    group_scale(bits_to_f32_max(packed), true, s, inv);
    return;
  }
  const uint32_t hi = packed >> 16, lo = packed & 0xFFFFu;
  uint32_t b = (hi > lo ? hi : lo) << 16;  // FP32 bits of the max-abs
  if (b < 0x05800000u) b = 0x05800000u;    // 2^-116
  if (b >= 0x7F800000u) {
    group_scale(__uint_as_float(b), false, s, inv);
    return;
  }
  const uint32_t m = (b >> 16) & 0x7Fu;
  const uint32_t e = (b >> 23) - 127u;  // E mod 2^32: added to the exponent field
  s = __uint_as_float(t.s[m] + (e << 23));
  inv = __uint_as_float(t.inv[m] - (e << 23));
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
// The BF16 tile quantisers below (128x1 and 128x128) work on 128 x 128 tiles
// with 512 threads (16 warps); the requantiser from FP8 uses 128 x 64 tiles
// with 256 threads (its own constants).
constexpr int kTileThreads = 512;

// ------------------------------------------------------------------ 128x1
// Persistent: each CTA walks 128-token x 128-channel tiles (channel blocks
// fastest) with a two-deep ring of input tiles filled by TMA, so the next
// tile streams in while this one is reduced and converted.  There is no CTA
// barrier in the loop: the last warp to finish reading an input buffer
// refills it.
//  - Input: two 64-channel halves per tile, 128-byte swizzled (the 16-byte
//    chunk k of token row r sits at chunk k ^ (r % 8)), so that ldmatrix.trans
//    reads 8 consecutive token rows of one chunk without bank conflicts.
//  - Warp w owns channels 8w .. 8w+7: four ldmatrix.x4.trans give each thread
//    32 values of one channel (c = 8w + lane/4; tokens 8m + 2(lane%4) + {0,1},
//    m = 0..15).  The channel's max-abs is a packed max over them and two
//    shuffles; no other warp is involved.
//  - Codes go to a swizzled shared-memory copy of the transposed tile
//    (channel rows of 128 bytes); each warp writes its 8 rows (1 KB) with its
//    own TMA store, so the transposed output costs no per-thread global
//    stores and no CTA barrier.
//  - Optionally the 1x128 codes of each token row (eight lanes per row, 32
//    bytes each).
// Channels past C are zero-filled by TMA; a warp whose 8 channel rows lie
// past C (C % 8 == 0: all of them or none) issues no store.
constexpr uint32_t kTileBytesBF16 = 128 * 128 * 2;
constexpr uint32_t kHalfBytesBF16 = kTileBytesBF16 / 2;   // 128 tokens x 64 channels
constexpr uint32_t kTileBytesQ = 128 * 128;                // one 128 x 128 tile of E4M3 codes

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

template <bool kPow2, bool kRows>
__global__ void __launch_bounds__(kTileThreads) quant_act_T_kernel(
    const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmQ, int64_t T,
    int64_t C, float *__restrict__ sT, int64_t ld_sT, uint8_t *__restrict__ q_rows,
    int64_t ldq_rows, float *__restrict__ s_rows, int64_t ld_s_rows, uint64_t timeout_ns) {
  extern __shared__ uint8_t dsm_raw[];
  const uint32_t in0 = (smem_u32(dsm_raw) + 1023u) & ~1023u;  // 2 x 32 KB input tiles
  const uint32_t st0 = in0 + 2 * kTileBytesBF16;               // 2 x 16 KB staged codes
  __shared__ uint64_t full[2];
  __shared__ uint32_t consumed[2];  // warps done with the buffer's current tile
  __shared__ int pending[2];        // parity of the last copy issued per buffer, or -1
  __shared__ int abort_flag;
  __shared__ ScaleTables tabs;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kWarps = kTileThreads / 32;
  scale_tables_init(tabs, tid);  // visible after the __syncthreads below
  // tile t = (token block t / ncb, channel block t % ncb); this CTA takes
  // t = blockIdx.x + i * gridDim.x, walked incrementally
  const uint32_t ncb = static_cast<uint32_t>((C + 127) / 128), ntb = static_cast<uint32_t>(T / 128);
  const uint32_t dcb = gridDim.x % ncb, dtb = gridDim.x / ncb;
  auto step = [&](uint32_t &cb, uint32_t &tb) {
    cb += dcb;
    tb += dtb;
    if (cb >= ncb) {
      cb -= ncb;
      ++tb;
    }
  };
  auto issue_load = [&](int b, uint32_t cb, uint32_t tb) {
    const uint32_t bar = smem_u32(&full[b]);
    mbar_arrive_expect_tx(bar, kTileBytesBF16);
    const int32_t c0 = static_cast<int32_t>(cb * 128), t0 = static_cast<int32_t>(tb * 128);
    tma_load_2d(in0 + b * kTileBytesBF16, &tmX, bar, c0, t0);
    tma_load_2d(in0 + b * kTileBytesBF16 + kHalfBytesBF16, &tmX, bar, c0 + 64, t0);
  };
  uint32_t cb = blockIdx.x % ncb, tb = blockIdx.x / ncb;  // this tile
  uint32_t cbn = cb, tbn = tb;                            // the tile two ahead
  if (tid == 0) {
    abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&full[b]), 1);
      consumed[b] = 0;
      pending[b] = -1;
    }
    fence_barrier_init();
  }
  for (int b = 0; b < 2; ++b) {
    if (tid == 0 && tbn < ntb) {
      issue_load(b, cbn, tbn);
      pending[b] = 0;
    }
    step(cbn, tbn);
  }
  __syncthreads();

  // this warp's channels: half h, 16-byte chunk j of each token row
  const uint32_t h = static_cast<uint32_t>(warp >> 3), j = static_cast<uint32_t>(warp & 7);
  const int cw = 8 * warp + (lane >> 2);  // this thread's channel within the tile
  int buf = 0;
  uint32_t phase = 0;
  while (tb < ntb) {
    const bool got = mbar_wait_bounded(smem_u32(&full[buf]), phase, &abort_flag,
                                       &g_quant_status, timeout_ns, FP8Q_ERR_TIMEOUT);
    if (__any_sync(0xffffffffu, !got)) break;
    const uint32_t tin = in0 + buf * kTileBytesBF16;
    const int64_t c0 = static_cast<int64_t>(cb) * 128, t0 = static_cast<int64_t>(tb) * 128;

    if (kRows) {  // C % 128 == 0 here: every chunk is in range
      // eight lanes per token row, 16 channels (two 16-byte chunks) each
      const int tr = tid >> 3, l8 = tid & 7;
      const uint32_t half = static_cast<uint32_t>(l8 >> 2) * kHalfBytesBF16;
      const uint32_t ch0 = static_cast<uint32_t>(2 * l8) & 7u;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t r = static_cast<uint32_t>(tr + 64 * i);
        uint4 v0, v1;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w)
                     : "r"(tin + half + swz128(r, ch0)));
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w)
                     : "r"(tin + half + swz128(r, ch0 + 1)));
        uint32_t mb = umax16x2(absmax_bits8(v0), absmax_bits8(v1));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
        float sc, inv;
        group_scale_bf16(tabs, mb, kPow2, sc, inv);
        const uint2 lo = quantise8(v0, inv), hi = quantise8(v1, inv);
        *reinterpret_cast<uint4 *>(q_rows + (t0 + r) * ldq_rows + c0 + l8 * 16) =
            make_uint4(lo.x, lo.y, hi.x, hi.y);
        if (l8 == 0) s_rows[(c0 / 128) * ld_s_rows + t0 + r] = sc;
      }
    }

    // ---- 128x1: this thread's channel, 32 of its 128 tokens
    uint32_t v[16];
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t r4[4];
      ldmatrix_x4_trans(tin + h * kHalfBytesBF16 + swz128(32u * qd + lane, j), r4);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[4 * qd + e] = r4[e];
    }
    __syncwarp();  // the warp's reads of buffer `buf` are done
    if (lane == 0) {
      uint32_t prev;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "r"(smem_u32(&consumed[buf]))
                   : "memory");
      if (prev == kWarps - 1) {  // the last reader refills the buffer
        consumed[buf] = 0;
        if (tbn < ntb) {
          fence_proxy_async_shared();  // generic-proxy reads above, async-proxy write below
          pending[buf] = static_cast<int>(phase ^ 1u);
          issue_load(buf, cbn, tbn);
        }
      }
    }
    step(cb, tb);
    step(cbn, tbn);

    uint32_t mw = 0;
#pragma unroll
    for (int m = 0; m < 16; ++m) mw = umax16x2(mw, v[m] & 0x7FFF7FFFu);
    mw = umax16x2(mw, __shfl_xor_sync(0xffffffffu, mw, 1));
    mw = umax16x2(mw, __shfl_xor_sync(0xffffffffu, mw, 2));
    float sc, inv;
    group_scale_bf16(tabs, mw, kPow2, sc, inv);
    if ((lane & 3) == 0 && c0 + cw < C) sT[(t0 / 128) * ld_sT + c0 + cw] = sc;
    uint32_t code[16];  // tokens 8m + 2(lane%4), +1 of channel cw
    const uint64_t inv2 = pack_f32x2(inv, inv);
#pragma unroll
    for (int m = 0; m < 16; ++m) code[m] = quantise2(v[m], inv2);

    // this warp's 8 channel rows (1 KB) of the staged transposed tile; its
    // store two tiles ago must have read them
    const uint32_t stg = st0 + buf * kTileBytesQ + static_cast<uint32_t>(warp) * 1024u;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int m = 0; m < 16; ++m)
      st_shared_u16(stg + swz128(static_cast<uint32_t>(lane >> 2), static_cast<uint32_t>(m >> 1)) +
                        8u * (m & 1) + 2u * (lane & 3),
                    code[m]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0 && c0 + 8 * warp < C) {  // C % 8 == 0: the 8 rows are all in range or all out
      tma_store_2d(&tmQ, stg, static_cast<int32_t>(t0), static_cast<int32_t>(c0 + 8 * warp));
      bulk_commit_group();
    }
    buf ^= 1;
    if (buf == 0) phase ^= 1u;
  }
  // every warp has left the loop (all tiles done, or a wait gave up): copies
  // still in flight after an abort land before the CTA's shared memory goes
  __syncthreads();
  if (tid == 0 && abort_flag)
    for (int b = 0; b < 2; ++b)
      if (pending[b] >= 0) mbar_wait_drain(smem_u32(&full[b]), static_cast<uint32_t>(pending[b]));
  if (lane == 0) bulk_wait_group_all();
}

// ------------------------------------------------------------------ 128x1 from FP8
// Persistent, like the BF16 128x1 quantiser.  Requantises FP8-cached
// activations: input E4M3 [T][C] with one 1x128 scale per (token, 128
// channels), output the 128x1 codes transposed.  Each value is first
// dequantised with one FP32 multiply, x = fl32(decode(q) * s_row), exactly as a
// BF16 input would be read.
//  - Tiles of 128 tokens x 128 channels (one row-scale group), channel blocks
//    fastest; the raw codes arrive by TMA in a two-deep ring, 128-byte
//    swizzled (16-byte chunk k of token row r at chunk k ^ (r % 8)); three
//    CTAs of 256 threads per SM.
//  - Warp w owns channels 16w..16w+15.  Four byte-wise ldmatrix.trans give
//    lane 4g + t the codes of tokens 32p + 16h + 4t + {0..3} (p = 0..3,
//    h = 0..1) of channels g and g + 8, four tokens of one channel per
//    register: the codes are transposed as bytes, and decoding, scaling, the
//    channel max-abs (two shuffles) and the new codes all happen in registers
//    in the transposed orientation, channel g first, then g + 8 (so that 32
//    FP32 values are live, not 64, and three CTAs fit an SM).
//  - Each warp stages its 16 channel rows of new codes (128-byte swizzle,
//    conflict-free 32-bit stores) and writes them with its own TMA store.
//  - No CTA barrier in the loop: each warp keeps its own copy of the row
//    scales (loaded one tile ahead), and the last warp to finish reading an
//    input stage refills it (a shared counter with acquire-release order).
constexpr int kRqThreads = 256;
constexpr int kRqWarps = kRqThreads / 32;
constexpr int kRqStages = 2;
constexpr int kRqCtasPerSm = 3;
constexpr uint32_t kRqTileBytes = 128 * 128;   // raw codes, 128-byte token rows
constexpr uint32_t kRqStripBytes = 16 * 128;   // one warp's 16 rows of new codes
template <bool kPow2>
__global__ void __launch_bounds__(kRqThreads, kRqCtasPerSm) requant_act_T_kernel(
    const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQT, int64_t T,
    int64_t C, const float *__restrict__ s_rows, int64_t ld_s_rows, float *__restrict__ sT,
    int64_t ld_sT, uint64_t timeout_ns) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ __align__(16) float srow[kRqWarps][2][128];
  __shared__ uint64_t full[kRqStages];
  __shared__ uint32_t consumed[kRqStages];  // warps done with the stage's current tile
  __shared__ int pending[kRqStages];        // parity of the last copy issued per stage, or -1
  __shared__ int abort_flag;
  const uint32_t raw0 = (smem_u32(dsm_raw) + 1023u) & ~1023u;  // kRqStages x 16 KB
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  // two 2 KB strips of staged codes per warp
  const uint32_t strip0 = raw0 + kRqStages * kRqTileBytes + warp * 2 * kRqStripBytes;

  // tile t = (token block t / ncb, channel block t % ncb); this CTA takes
  // t = blockIdx.x + i * gridDim.x, walked incrementally
  const uint32_t ncb = static_cast<uint32_t>(C / 128), ntb = static_cast<uint32_t>(T / 128);
  const uint32_t dcb = gridDim.x % ncb, dtb = gridDim.x / ncb;
  auto step = [&](uint32_t &cb, uint32_t &tb) {
    cb += dcb;
    tb += dtb;
    if (cb >= ncb) {
      cb -= ncb;
      ++tb;
    }
  };
  auto issue_load = [&](int st, uint32_t cb, uint32_t tb) {
    const uint32_t bar = smem_u32(&full[st]);
    mbar_arrive_expect_tx(bar, kRqTileBytes);
    tma_load_2d(raw0 + st * kRqTileBytes, &tmQ, bar, static_cast<int32_t>(cb * 128),
                static_cast<int32_t>(tb * 128));
  };
  // lane l: the row scales of tokens l + 32i of tile (cb, tb)
  auto load_scales = [&](uint32_t cb, uint32_t tb, float (&v)[4]) {
    const float *p = s_rows + static_cast<int64_t>(cb) * ld_s_rows + tb * 128u + lane;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = p[32 * i];
  };

  uint32_t cb = blockIdx.x % ncb, tb = blockIdx.x / ncb;  // this tile
  uint32_t cbn = cb, tbn = tb;                            // the tile kRqStages ahead
  if (tid == 0) {
    abort_flag = 0;
    for (int st = 0; st < kRqStages; ++st) {
      mbar_init(smem_u32(&full[st]), 1);
      consumed[st] = 0;
      pending[st] = -1;
    }
    fence_barrier_init();
  }
  for (int st = 0; st < kRqStages; ++st) {
    if (tid == 0 && tbn < ntb) {
      issue_load(st, cbn, tbn);
      pending[st] = 0;
    }
    step(cbn, tbn);
  }
  float sn[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (tb < ntb) load_scales(cb, tb, sn);
  __syncthreads();

  // ldmatrix: lane l gives token row 32p + l, chunk `warp` of it (swizzled)
  const uint32_t ld_off = static_cast<uint32_t>(lane) * 128u +
                          ((static_cast<uint32_t>(warp) ^ (static_cast<uint32_t>(lane) & 7u)) << 4);
  int st = 0;
  uint32_t phase = 0, sb = 0;
  while (tb < ntb) {
    const bool got = mbar_wait_bounded(smem_u32(&full[st]), phase, &abort_flag,
                                       &g_quant_status, timeout_ns, FP8Q_ERR_TIMEOUT);
    if (__any_sync(0xffffffffu, !got)) break;
    // r[4p + 2h + j]: channel g + 8j, tokens 32p + 16h + 4tq + {0..3}
    uint32_t r[16];
    const uint32_t in = raw0 + st * kRqTileBytes;
#pragma unroll
    for (int p = 0; p < 4; ++p) ldmatrix_b8_x2_trans(in + 4096u * p + ld_off, &r[4 * p]);
    float *srw = srow[warp][sb];
#pragma unroll
    for (int i = 0; i < 4; ++i) srw[lane + 32 * i] = sn[i];
    __syncwarp();  // the warp's reads of stage `st` are done; its row scales are visible
    if (lane == 0) {
      uint32_t prev;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                   : "=r"(prev)
                   : "r"(smem_u32(&consumed[st]))
                   : "memory");
      if (prev == kRqWarps - 1) {  // the last reader refills the stage
        consumed[st] = 0;
        if (tbn < ntb) {
          fence_proxy_async_shared();  // generic-proxy reads above, async-proxy write below
          pending[st] = static_cast<int>(phase ^ 1u);
          issue_load(st, cbn, tbn);
        }
      }
    }
    const uint32_t cbc = cb, tbc = tb;
    step(cb, tb);
    step(cbn, tbn);
    if (tb < ntb) load_scales(cb, tb, sn);  // next tile's row scales, used one tile later
    if (++st == kRqStages) {
      st = 0;
      phase ^= 1u;
    }

    const uint32_t stg = strip0 + sb * kRqStripBytes;
    const float *srwc = srw;
    sb ^= 1u;
    if (lane == 0) bulk_wait_group_read<1>();  // this strip's store two tiles ago has read it
    __syncwarp();
    // one channel at a time (g, then g + 8): decode and scale, x[2ph], x[2ph+1]
    // are tokens {0,1} and {2,3} of r[2ph + j] as packed FP32 (one
    // mul.rn.f32x2 by the pair of row scales), then max-abs, scale and codes
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint64_t x[16];
      float am = 0.0f;
#pragma unroll
      for (int ph = 0; ph < 8; ++ph) {
        const ulonglong2 sp = *reinterpret_cast<const ulonglong2 *>(&srwc[16 * ph + 4 * tq]);
        const int k = 2 * ph + j;
        const uint32_t h01 = decode_e4m3x2(static_cast<uint16_t>(r[k] & 0xFFFFu));
        const uint32_t h23 = decode_e4m3x2(static_cast<uint16_t>(r[k] >> 16));
        x[2 * ph] = fmul2(pack_f32x2(f16_lo(h01), f16_hi(h01)), sp.x);
        x[2 * ph + 1] = fmul2(pack_f32x2(f16_lo(h23), f16_hi(h23)), sp.y);
        const float2 a = unpack_f32x2(x[2 * ph]), b = unpack_f32x2(x[2 * ph + 1]);
        am = fmaxf(am, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))));
      }
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      float sc, inv;
      group_scale(am, kPow2, sc, inv);
      if (tq == 0) sT[static_cast<int64_t>(tbc) * ld_sT + cbc * 128u + 16 * warp + g + 8 * j] = sc;
      const uint64_t iv = pack_f32x2(inv, inv);
#pragma unroll
      for (int ph = 0; ph < 8; ++ph) {
        const float2 a = unpack_f32x2(fmul2(x[2 * ph], iv));
        const float2 b = unpack_f32x2(fmul2(x[2 * ph + 1], iv));
        // channel row g + 8j, token chunk ph (bytes 16ph + 4tq), swizzled by row % 8 = g
        st_shared_u32(stg + static_cast<uint32_t>(g + 8 * j) * 128u +
                          ((static_cast<uint32_t>(ph) ^ static_cast<uint32_t>(g)) << 4) + 4u * tq,
                      pack_e4m3x4(a.x, a.y, b.x, b.y));
      }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&tmQT, stg, static_cast<int32_t>(tbc * 128), static_cast<int32_t>(cbc * 128 + 16 * warp));
      bulk_commit_group();
    }
  }
  // every warp has left the loop (all tiles done, or a wait gave up): copies
  // still in flight after an abort land before the CTA's shared memory goes
  __syncthreads();
  if (tid == 0 && abort_flag)
    for (int b = 0; b < kRqStages; ++b)
      if (pending[b] >= 0) mbar_wait_drain(smem_u32(&full[b]), static_cast<uint32_t>(pending[b]));
  if (lane == 0) bulk_wait_group_all();
}

// ------------------------------------------------------------------ 128x128
// Grid (K / 128, ceil(N / 128)).  A CTA owns one block: reduces the block
// max-abs (packed max, warp shuffles, then across the 16 warps) and writes the
// codes row-wise from registers.  With the transposed copy, the block also
// goes to shared memory in two 128-byte-swizzled halves (as the 128x1
// quantiser's TMA tiles); warp w reads columns 8w .. 8w+7 of all 128 rows
// with ldmatrix.trans, and the transposed codes are staged and written by one
// TMA store (rows past N clipped by it).
template <bool kPow2, bool kTrans>
__global__ void __launch_bounds__(kTileThreads) quant_weight_kernel(
    const uint16_t *__restrict__ w, int64_t N, int64_t ldw, uint8_t *__restrict__ q, int64_t ldq,
    const __grid_constant__ CUtensorMap tmQT, uint8_t *__restrict__ qT_ptr, int64_t ldqT,
    float *__restrict__ sb, int64_t ld_sb) {
  extern __shared__ uint8_t dsm_raw[];
  __shared__ uint32_t warp_amax[16];
  __shared__ float blk_inv;

  const int tid = threadIdx.x, hw = tid >> 4, l16 = tid & 15;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 128;
  const uint32_t tin = kTrans ? ((smem_u32(dsm_raw) + 1023u) & ~1023u) : 0u;  // 2 x 16 KB
  const uint32_t stg = tin + kTileBytesBF16;                                  // 16 KB

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
    for (int i = 0; i < 4; ++i)
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                       tin + (l16 >> 3) * kHalfBytesBF16 +
                       swz128(static_cast<uint32_t>(hw + 32 * i), static_cast<uint32_t>(l16 & 7))),
                   "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                   : "memory");
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
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t h = static_cast<uint32_t>(warp >> 3), j = static_cast<uint32_t>(warp & 7);
    const uint32_t kw = static_cast<uint32_t>(8 * warp + (lane >> 2));  // this thread's column
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t r4[4];
      ldmatrix_x4_trans(tin + h * kHalfBytesBF16 + swz128(32u * qd + lane, j), r4);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = 4 * qd + e;  // rows 8m + 2(lane%4), +1
        st_shared_u16(stg + swz128(kw, static_cast<uint32_t>(m >> 1)) + 8u * (m & 1) +
                          2u * (lane & 3),
                      pack_e4m3x2(__fmul_rn(bf16_lo(r4[e]), inv), __fmul_rn(bf16_hi(r4[e]), inv)));
      }
    }
    if (n0 + 128 <= N) {  // a whole block: one TMA store
      fence_proxy_async_shared();
      __syncthreads();
      if (tid == 0) {
        tma_store_2d(&tmQT, stg, static_cast<int32_t>(n0), static_cast<int32_t>(k0));
        bulk_commit_group();
        bulk_wait_group_all();
      }
    } else {
      // the last, partial block: the TMA store would clip the row at 16-byte
      // granularity and could write past N, so copy the staged rows out with
      // bounds (thread: row kk, 32 bytes)
      __syncthreads();
      const uint32_t kk = static_cast<uint32_t>(tid >> 2);
      uint8_t *row = qT_ptr + (k0 + kk) * ldqT + n0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const uint32_t chunk = 2u * (tid & 3) + c;
        uint4 b;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                     : "r"(stg + swz128(kk, chunk)));
        const int64_t nb = n0 + 16 * chunk;
        if (nb + 16 <= N) {
          *reinterpret_cast<uint4 *>(row + 16 * chunk) = b;
        } else {
          const uint32_t wds[4] = {b.x, b.y, b.z, b.w};
          for (int e = 0; e < 16 && nb + e < N; ++e)
            row[16 * chunk + e] = static_cast<uint8_t>(wds[e >> 2] >> (8 * (e & 3)));
        }
      }
    }
  }
}

// ------------------------------------------------------------------ per tensor
// Comparison path: one scale for a whole [M][K] tensor.  Two passes over a
// workspace of one 32-bit partial per 64-row slab:
//   pass 1: each CTA writes the packed max of |BF16| bits over its 64 rows;
//   pass 2: each CTA reduces all partials to the tensor's max-abs, derives
//           the scale (CTA 0 stores it) and quantises its 64 rows.
constexpr int kTensorRows = 64;

__global__ void __launch_bounds__(256) tensor_amax_kernel(const uint16_t *__restrict__ x,
                                                          int64_t M, int64_t K, int64_t ldx,
                                                          uint32_t *__restrict__ partials) {
  __shared__ uint32_t warp_max[8];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTensorRows;
  const int64_t r1 = r0 + kTensorRows < M ? r0 + kTensorRows : M;
  const int64_t chunks = K / 8;  // 16-byte chunks per row
  uint32_t mb = 0;
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x)
      mb = umax16x2(mb, absmax_bits8(ld_stream_v4(x + r * ldx + c * 8)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mb;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = warp_max[0];
    for (int i = 1; i < 8; ++i) a = umax16x2(a, warp_max[i]);
    partials[blockIdx.x] = a;
  }
}

template <bool kPow2>
__global__ void __launch_bounds__(256) tensor_quant_kernel(const uint16_t *__restrict__ x,
                                                           int64_t M, int64_t K, int64_t ldx,
                                                           uint8_t *__restrict__ q, int64_t ldq,
                                                           float *__restrict__ s_out,
                                                           const uint32_t *__restrict__ partials,
                                                           int n_partials) {
  __shared__ uint32_t warp_max[8];
  __shared__ float sh_inv;
  uint32_t mb = 0;
  for (int i = threadIdx.x; i < n_partials; i += blockDim.x) mb = umax16x2(mb, partials[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mb = umax16x2(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mb;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = warp_max[0];
    for (int i = 1; i < 8; ++i) a = umax16x2(a, warp_max[i]);
    float sc, inv;
    group_scale(bits_to_f32_max(a), kPow2, sc, inv);
    sh_inv = inv;
    if (blockIdx.x == 0) *s_out = sc;
  }
  __syncthreads();
  const float inv = sh_inv;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTensorRows;
  const int64_t r1 = r0 + kTensorRows < M ? r0 + kTensorRows : M;
  const int64_t chunks = K / 8;
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t c = threadIdx.x; c < chunks; c += blockDim.x)
      *reinterpret_cast<uint2 *>(q + r * ldq + c * 8) = quantise8(ld_stream_v4(x + r * ldx + c * 8), inv);
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

constexpr int kActTCtasPerSm = 2;  // 2 x 32 KB input ring + 2 x 16 KB staged codes each
constexpr size_t kActTSmem = 2 * kTileBytesBF16 + 2 * kTileBytesQ + 1024;

template <bool kPow2, bool kRows>
fp8q_status launch_act_T(unsigned grid, cudaStream_t s, const CUtensorMap &tmX,
                         const CUtensorMap &tmQ, int64_t T, int64_t C, float *sT, int64_t ld_sT,
                         uint8_t *q_rows, int64_t ldq_rows, float *s_rows, int64_t ld_s_rows,
                         uint64_t timeout_ns) {
  auto kern = quant_act_T_kernel<kPow2, kRows>;
  static bool attr_set[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kActTSmem)) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  return launch_on(kern, dim3(grid), dim3(kTileThreads), kActTSmem, s, tmX, tmQ, T, C, sT, ld_sT,
                   q_rows, ldq_rows, s_rows, ld_s_rows, timeout_ns);
}

constexpr size_t kRequantSmem =
    kRqStages * kRqTileBytes + (kRqThreads / 32) * 2 * kRqStripBytes + 1024;

template <bool kPow2>
fp8q_status launch_requant(unsigned grid, cudaStream_t s, const CUtensorMap &tmQ,
                           const CUtensorMap &tmQT, int64_t T, int64_t C, const float *s_rows,
                           int64_t ld_s_rows, float *sT, int64_t ld_sT, uint64_t timeout_ns) {
  auto kern = requant_act_T_kernel<kPow2>;
  static bool attr_set[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kRequantSmem)) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  return launch_on(kern, dim3(grid), dim3(kRqThreads), kRequantSmem, s, tmQ, tmQT, T, C, s_rows,
                   ld_s_rows, sT, ld_sT, timeout_ns);
}

constexpr size_t kWeightTSmem = kTileBytesBF16 + kTileBytesQ + 1024;  // transposed path only

template <bool kPow2, bool kTrans>
fp8q_status launch_weight(dim3 grid, cudaStream_t s, const uint16_t *w, int64_t N, int64_t ldw,
                          uint8_t *q, int64_t ldq, const CUtensorMap &tmQT, uint8_t *qT,
                          int64_t ldqT, float *sb, int64_t ld_sb) {
  auto kern = quant_weight_kernel<kPow2, kTrans>;
  const size_t smem = kTrans ? kWeightTSmem : 0;
  if (kTrans) {
    static bool attr_set[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  return launch_on(kern, grid, dim3(kTileThreads), smem, s, w, N, ldw, q, ldq, tmQT, qT, ldqT, sb,
                   ld_sb);
}

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
  return launch_on(scale_mode == FP8Q_SCALE_POW2 ? quant_act_kernel<true> : quant_act_kernel<false>,
                   grid, dim3(256), 0, s, xp, M, ldx, qp, ldq, sa, ld_sa);
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
  if (T / 128 > 65535 || C > INT32_MAX - 127) return FP8Q_ERR_SHAPE;  // 32-bit tile coordinates
  if (T == 0 || C == 0) return FP8Q_OK;
  if (!x || !qT || !sT || (rows && !s_rows)) return FP8Q_ERR_INVALID;
  if (!aligned16(x) || !aligned16(qT) || !aligned4(sT) || ldx % 8 || ldqT % 16)
    return FP8Q_ERR_ALIGN;
  if (rows && (!aligned16(q_rows) || !aligned4(s_rows) || ldq_rows % 16)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  // input: 64-channel x 128-token boxes, 128-byte swizzle; output: the
  // transposed codes qT [C][T], 128-token x 8-channel boxes (one warp's
  // rows), same swizzle
  CUtensorMap tmX, tmQ;
  if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(T),
                    static_cast<uint64_t>(C), static_cast<uint64_t>(ldx) * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, qT, static_cast<uint64_t>(C),
                    static_cast<uint64_t>(T), static_cast<uint64_t>(ldqT), 128, 8,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8Q_ERR_CUDA;
  const int64_t ntiles = ((C + 127) / 128) * (T / 128);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * kActTCtasPerSm;
  const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
  auto s = static_cast<cudaStream_t>(stream);
  auto rp = static_cast<uint8_t *>(q_rows);
  const uint64_t tmo = wait_timeout_ns().load();
  const bool p2 = scale_mode == FP8Q_SCALE_POW2;
  fp8q_status st = FP8Q_OK;
  if (p2 && rows)
    st = launch_act_T<true, true>(grid, s, tmX, tmQ, T, C, sT, ld_sT, rp, ldq_rows, s_rows,
                                  ld_s_rows, tmo);
  else if (p2)
    st = launch_act_T<true, false>(grid, s, tmX, tmQ, T, C, sT, ld_sT, rp, ldq_rows, s_rows,
                                   ld_s_rows, tmo);
  else if (rows)
    st = launch_act_T<false, true>(grid, s, tmX, tmQ, T, C, sT, ld_sT, rp, ldq_rows, s_rows,
                                   ld_s_rows, tmo);
  else
    st = launch_act_T<false, false>(grid, s, tmX, tmQ, T, C, sT, ld_sT, rp, ldq_rows, s_rows,
                                    ld_s_rows, tmo);
  return st;
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
  // the transposed codes qT [K][N]: 128-row x 128-column boxes, 128-byte swizzle
  CUtensorMap tmQT{};
  if (trans && !make_tmap_2d(&tmQT, CU_TENSOR_MAP_DATA_TYPE_UINT8, qT, static_cast<uint64_t>(K),
                             static_cast<uint64_t>(N), static_cast<uint64_t>(ldqT), 128, 128,
                             CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8Q_ERR_CUDA;
  const bool p2 = scale_mode == FP8Q_SCALE_POW2;
  if (p2 && trans) return launch_weight<true, true>(grid, s, wp, N, ldw, qp, ldq, tmQT, static_cast<uint8_t *>(qT), ldqT, sb, ld_sb);
  if (p2) return launch_weight<true, false>(grid, s, wp, N, ldw, qp, ldq, tmQT, static_cast<uint8_t *>(qT), ldqT, sb, ld_sb);
  if (trans) return launch_weight<false, true>(grid, s, wp, N, ldw, qp, ldq, tmQT, static_cast<uint8_t *>(qT), ldqT, sb, ld_sb);
  return launch_weight<false, false>(grid, s, wp, N, ldw, qp, ldq, tmQT, static_cast<uint8_t *>(qT), ldqT, sb, ld_sb);
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
  return launch_on(cast_e4m3_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                   static_cast<cudaStream_t>(stream), x, n, static_cast<uint8_t *>(q));
}

extern "C" fp8q_status fp8q_requant_act_T(const void *q, int64_t T, int64_t C, int64_t ldq,
                                          const float *s_rows, int64_t ld_s_rows, void *qT,
                                          int64_t ldqT, float *sT, int64_t ld_sT, int scale_mode,
                                          void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  if (T < 0 || C < 0 || T % 128 != 0 || C % 128 != 0 || ldq < C || ld_s_rows < T || ldqT < T ||
      ld_sT < C)
    return FP8Q_ERR_SHAPE;
  if (T / 128 > 65535 || C > INT32_MAX) return FP8Q_ERR_SHAPE;  // 32-bit tile coordinates
  if (T == 0 || C == 0) return FP8Q_OK;
  if (!q || !s_rows || !qT || !sT) return FP8Q_ERR_INVALID;
  if (!aligned16(q) || !aligned16(qT) || !aligned4(s_rows) || !aligned4(sT) || ldq % 16 ||
      ldqT % 16)
    return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  // codes [T][C] in boxes of 128 tokens x 128 bytes; qT [C][T] in boxes of 16
  // channel rows x 128 bytes (one warp's strip); both 128-byte swizzled
  CUtensorMap tmQ, tmQT;
  if (!make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, static_cast<uint64_t>(T),
                    static_cast<uint64_t>(C), static_cast<uint64_t>(ldq), 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmQT, CU_TENSOR_MAP_DATA_TYPE_UINT8, qT, static_cast<uint64_t>(C),
                    static_cast<uint64_t>(T), static_cast<uint64_t>(ldqT), 128, 16,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8Q_ERR_CUDA;
  const int64_t ntiles = (C / 128) * (T / 128);
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * kRqCtasPerSm;
  const unsigned grid = static_cast<unsigned>(ntiles < cap ? ntiles : cap);
  auto s = static_cast<cudaStream_t>(stream);
  const uint64_t tmo = wait_timeout_ns().load();
  return scale_mode == FP8Q_SCALE_POW2
             ? launch_requant<true>(grid, s, tmQ, tmQT, T, C, s_rows, ld_s_rows, sT, ld_sT, tmo)
             : launch_requant<false>(grid, s, tmQ, tmQT, T, C, s_rows, ld_s_rows, sT, ld_sT, tmo);
}

// The two passes of the per-tensor quantiser over the partials array `part`.
static fp8q_status tensor_passes(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                                 int64_t ldq, float *s, uint32_t *part, int64_t P, int scale_mode,
                                 cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>(P));
  if (fp8q_status e = launch_on(tensor_amax_kernel, grid, dim3(256), 0, st, x, M, K, ldx, part))
    return e;
  return launch_on(scale_mode == FP8Q_SCALE_POW2 ? tensor_quant_kernel<true>
                                                 : tensor_quant_kernel<false>,
                   grid, dim3(256), 0, st, x, M, K, ldx, q, ldq, s,
                   static_cast<const uint32_t *>(part), static_cast<int>(P));
}

static int64_t tensor_partials(int64_t M) { return M > 0 ? (M + kTensorRows - 1) / kTensorRows : 1; }

extern "C" int64_t fp8q_quant_tensor_workspace_bytes(int64_t M, int64_t K) {
  (void)K;
  return M < 0 ? 0 : tensor_partials(M) * static_cast<int64_t>(sizeof(uint32_t));
}

extern "C" fp8q_status fp8q_quant_tensor(const void *x, int64_t M, int64_t K, int64_t ldx, void *q,
                                         int64_t ldq, float *s, void *workspace,
                                         int64_t workspace_bytes, int scale_mode, void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  if (M < 0 || K < 0 || K % 8 != 0 || ldx < K || ldq < K) return FP8Q_ERR_SHAPE;
  const int64_t P = tensor_partials(M);
  if (P > (1ll << 31) - 1) return FP8Q_ERR_SHAPE;
  if (!s || !workspace) return FP8Q_ERR_INVALID;
  if (workspace_bytes < P * static_cast<int64_t>(sizeof(uint32_t))) return FP8Q_ERR_SHAPE;
  if (M > 0 && K > 0 && (!x || !q)) return FP8Q_ERR_INVALID;
  if ((M > 0 && K > 0) && (!aligned16(x) || !aligned16(q) || ldx % 8 || ldq % 8))
    return FP8Q_ERR_ALIGN;
  if (!aligned4(s) || !aligned4(workspace)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  auto st_ = static_cast<cudaStream_t>(stream);
  auto xp = static_cast<const uint16_t *>(x);
  auto part = static_cast<uint32_t *>(workspace);
  return tensor_passes(xp, M, K, ldx, static_cast<uint8_t *>(q), ldq, s, part, P, scale_mode, st_);
}

// ------------------------------------------------------------------ per tensor, no allocation
// fp8q_quant_tensor without a caller-supplied workspace, for callers that
// cannot allocate device memory at call time: code running inside an
// allocator's or memory pool's own callbacks (allocating there would re-enter
// the allocator), or a runtime that has handed all device memory to its own
// pools and has none left to lend.  Its scratch is one fixed array per device
// in the library's static device memory, sized for kNoAllocPartials partials
// of kTensorRows rows each (M <= 65536).  Nothing in the array has to start at
// zero: pass 1 writes every partial that pass 2 reads.  All calls on a device
// share the array, so two of them that overlap on the GPU (different streams,
// no ordering) race.
constexpr int64_t kNoAllocPartials = 1024;  // 4 KB per device, held until the process exits
static __device__ __align__(256) uint32_t g_noalloc_partials[kNoAllocPartials];

// Unique id of the calling thread's current CUDA context, or 0 when no
// context is current or the driver cannot say (driver entry points looked up
// through the runtime, as for the tensor-map encoder).
static uint64_t current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext *);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array in the current device's current context.  The
// address is cached per device together with the id of the context it was
// looked up in, and looked up again whenever that context is not the current
// one (after cudaDeviceReset, or after the primary context was released and
// created anew, the old address belongs to a context that no longer exists).
// Without a context id the lookup is simply repeated on every call.
static fp8q_status noalloc_partials(uint32_t **out) {
  struct Slot {
    uint64_t ctx_id = 0;
    uint32_t *ptr = nullptr;
  };
  static Slot slots[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  Slot &slot = slots[dev];
  const uint64_t now = current_context_id();
  if (slot.ptr == nullptr || now == 0 || now != slot.ctx_id) {
    uint32_t *ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_partials) != cudaSuccess ||
        ptr == nullptr)
      return FP8Q_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    slot.ctx_id = current_context_id();
    slot.ptr = slot.ctx_id != 0 ? ptr : nullptr;
    *out = ptr;
    return FP8Q_OK;
  }
  *out = slot.ptr;
  return FP8Q_OK;
}

extern "C" fp8q_status fp8q_quant_tensor_noalloc(const void *x, int64_t M, int64_t K, int64_t ldx,
                                                 void *q, int64_t ldq, float *s, int scale_mode,
                                                 void *stream) {
  if (!valid_mode(scale_mode)) return FP8Q_ERR_INVALID;
  if (M < 0 || K < 0 || K % 8 != 0 || ldx < K || ldq < K) return FP8Q_ERR_SHAPE;
  const int64_t P = tensor_partials(M);
  if (P > kNoAllocPartials) return FP8Q_ERR_SHAPE;
  if (!s) return FP8Q_ERR_INVALID;
  if (M > 0 && K > 0 && (!x || !q)) return FP8Q_ERR_INVALID;
  if ((M > 0 && K > 0) && (!aligned16(x) || !aligned16(q) || ldx % 8 || ldq % 8))
    return FP8Q_ERR_ALIGN;
  if (!aligned4(s)) return FP8Q_ERR_ALIGN;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  uint32_t *part = nullptr;
  if (fp8q_status st = noalloc_partials(&part)) return st;
  auto st_ = static_cast<cudaStream_t>(stream);
  auto xp = static_cast<const uint16_t *>(x);
  return tensor_passes(xp, M, K, ldx, static_cast<uint8_t *>(q), ldq, s, part, P, scale_mode, st_);
}
