// gemm.cu -- FP8 (E4M3) GEMM with per-128-K-group scaling for sm_103a.
//
//   C[m][n] = sum_kb sa(m,kb) * sb(n,kb) * P_kb[m][n],
//   P_kb[m][n] = sum_{k in kb} a[m][k] * b[n][k]   (tensor cores, FP32)
//
// The method (dssusan.co.kr post 91437, paragraph 3, Figure 6) scales each
// 128-wide group of the inner dimension K separately, so the group partial
// sums must be scaled before they are added; on the pages' Hopper parts the
// partials are copied from the tensor cores to FP32 registers at a fixed K
// interval.  Here the interval is one 128-K group and the hardware is
// tcgen05:
//
//   warp 0      TMA producer: A and B tiles (128 K-bytes per row, 128-byte
//               swizzle) into a kStages-deep shared-memory ring, completing
//               on "full" mbarriers.
//   warp 1      MMA issuer (one thread; in a CTA pair, of the leading CTA):
//               per K-group, 4 x tcgen05.mma (kind::f8f6f4, K=32, N=256; M=256
//               across the pair with cta_group::2, each CTA's 128 rows in its
//               own TMEM) into one of two TMEM partial buffers, then
//               tcgen05.commit to release the ring slot and to signal the
//               partial.
//   warps 2-3   idle (they complete the first warpgroup).
//   warps 4-11  epilogue: tcgen05.ld the partial (each thread one row, 128
//               columns, 16 at a time), acc += P * sa(m,kb) * sb(n,kb) in FP32
//               registers with packed two-lane FMAs (fma.rn.f32x2), release the
//               TMEM buffer; after the last group, round C to BF16 (nearest
//               even) or keep FP32 and write it out through 8 KB of shared
//               memory per warp: BF16 as two 128-byte-swizzled boxes and TMA
//               tensor stores, otherwise as coalesced 16-byte stores, both
//               with an L2 evict-first policy.  The scales of group kb+1 are
//               loaded while group kb is folded.
//
// Registers: the kernel is built for 384 threads at 168 registers each (the
// register file of each SM sub-partition holds three warps at 168).  The
// first warpgroup then gives registers back (setmaxnreg.dec to 40) and the two
// epilogue warpgroups take them (setmaxnreg.inc to 232): per sub-partition
// 40 + 232 + 232 = 504 = 3 x 168, so the increase is always satisfiable.
//
// The two TMEM buffers (2 x 256 columns = all 512) let the tensor cores fill
// group kb+1 while the epilogue folds group kb.  The kernel is persistent
// (one CTA per SM, static round-robin over output tiles).  Every mbarrier wait
// is bounded in time; a wait that gives up raises a CTA-wide abort flag and
// records FP8Q_ERR_TIMEOUT in the device status word, and every role then
// drains its own in-flight copies / MMAs before the CTA frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8q.h"
#include "fp8q_host.cuh"
#include "fp8q_ptx.cuh"

namespace fp8q {

// Device status word: 0, or the fp8q_status of the first device-side failure
// since it was last cleared by fp8q_sync_status().
__device__ int g_status;

namespace {

constexpr int BM = 128, BN = 256, BK = 128;   // per-CTA rows, tile columns, K-group
constexpr int kEpiWarps = 8;                     // 2 warpgroups: 4 TMEM lane quarters x 2
constexpr int kEpiCols = BN / (kEpiWarps / 4);   // columns folded by each epilogue thread
constexpr int kThreads = 128 + kEpiWarps * 32;   // control warpgroup + epilogue warpgroups
constexpr int kWarpsPerSubpartition = kThreads / 128;
constexpr int kLaunchRegs = 168;                 // must match ptxas' count (checked by the build)
constexpr int kCtlRegs = 40, kEpiRegs = 232;
// setmaxnreg can only hand out what the launch allocated on each sub-partition
// (one control warp and kWarpsPerSubpartition - 1 epilogue warps there)
static_assert(kCtlRegs + (kWarpsPerSubpartition - 1) * kEpiRegs <=
                  kWarpsPerSubpartition * kLaunchRegs,
              "register split must fit the launch allocation");
static_assert(kLaunchRegs * kThreads <= 65536, "launch register budget");
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupM = 16;   // L2 rasterisation band (m-tiles) for the dense GEMM
constexpr int kMaxGroups = 1024;
constexpr uint64_t kDrainNs = 1000000000ull;  // 1 s for draining after an abort
constexpr int kMaxStages = 6;
constexpr bool kGroupedPair = true;   // tile shape of the grouped (MoE) GEMM
constexpr bool kDensePair = true;    // tile shape of the dense GEMMs

// Two shapes of the same pipeline:
//  single CTA: tile 128 x 256 per CTA; ring stage = A 128 rows + B 256 rows.
//  CTA pair  : tile 256 x 256 per cluster of two CTAs; each CTA stages its own
//              128 rows of A and 128 rows (half the columns) of B, and one
//              tcgen05.mma.cta_group::2 (M = 256) in the leading CTA reads both
//              CTAs' shared memory and writes both CTAs' tensor memory.  Per SM
//              that is 32 KB of operands per K-group instead of 48 KB, refilled
//              with a third less traffic; four stages (measured as fast as
//              six) leave 64 KB for the output staging.
template <bool kPair>
struct Cfg {
  static constexpr int kStages = kPair ? 4 : 2;
  static constexpr uint32_t kABytes = BM * BK;                    // per CTA
  static constexpr uint32_t kBBytes = (kPair ? BN / 2 : BN) * BK;  // per CTA
  static constexpr int kTileM = kPair ? 2 * BM : BM;              // C rows per tile
  static constexpr uint32_t kIdesc = idesc_e4m3_f32(kPair ? 2 * BM : BM, BN);
  static constexpr uint32_t kTxBytes = (kPair ? 2 : 1) * (kABytes + kBBytes);
  static constexpr int kTemptyCount = (kPair ? 2 : 1) * kEpiWarps;
  static constexpr size_t kTileBytes = static_cast<size_t>(kStages) * (kABytes + kBBytes);
  static_assert(kStages <= kMaxStages, "ring too deep for SmemCtl");
};

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Wait for a phase regardless of the abort flag, for at most kDrainNs; used
// only to let a CTA's own copies and MMAs finish before it exits.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kDrainNs) return;
}

// Spin for `ns` nanoseconds (lets copies issued just before an abort land).
__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

struct GemmArgs {
  const float *sa;
  int64_t ld_sa;
  const float *sb;
  int64_t ld_sb;
  void *c;
  int64_t ldc;
  int M, N;
  int num_kb;
  int tiles_m, tiles_n;
  const int32_t *offs;  // grouped only
  int G;
  uint64_t timeout_ns;
};

// Shared-memory control block, after the operand ring and the output staging.
struct alignas(8) SmemCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  // per-column B scales (Wgrad): each epilogue warp stages the scales of its
  // own columns for the current K-group, double-buffered
  alignas(16) float sb_warp[kEpiWarps][2][kEpiCols];
};

// Output staging: 8 KB per epilogue warp: its 32 rows x 128 BF16 columns as
// two 32-row x 128-byte boxes for TMA tensor stores (grouped GEMM), or, in
// its first 2 KB, the 32 x 64-byte blocks of the coalesced stores.
constexpr uint32_t kStageWarpBytes = 8192;
constexpr uint32_t kStageCBytes = kEpiWarps * kStageWarpBytes;

__host__ __device__ constexpr size_t smem_bytes(bool grouped, bool pair) {
  return 1024 /* alignment slack */ + (pair ? Cfg<true>::kTileBytes : Cfg<false>::kTileBytes) +
         kStageCBytes + sizeof(SmemCtl) + (grouped ? 2 * (kMaxGroups + 1) * sizeof(int) : 0);
}
static_assert(smem_bytes(true, true) <= 227 * 1024 && smem_bytes(true, false) <= 227 * 1024,
              "shared memory per CTA");

struct Tile {
  int a_row;    // first row of A (and of C) covered by the tile (first CTA of a pair)
  int row_end;  // rows >= row_end are not stored
  int b_row;    // first row of B (expert-offset for grouped)
  int n0;       // first output column
  int g;        // expert (grouped) or 0
};

// Grouped tables in shared memory: s_lo[g] .. s_lo[g + 1] = clamped row range of
// expert g, s_pre[g] = number of m-tiles of experts before g (s_pre[G] = all).
template <bool kGrouped, int kTileM>
__device__ __forceinline__ Tile tile_of(int t, const GemmArgs &p, const int *s_lo,
                                        const int *s_pre) {
  Tile r;
  if (!kGrouped) {
    const int band_tiles = kGroupM * p.tiles_n;
    const int band = t / band_tiles, within = t - band * band_tiles;
    const int mt0 = band * kGroupM;
    const int rows = min(kGroupM, p.tiles_m - mt0);
    const int mt = mt0 + within % rows, nt = within / rows;
    r.a_row = mt * kTileM;
    r.row_end = p.M;
    r.n0 = nt * BN;
    r.b_row = r.n0;
    r.g = 0;
  } else {
    // expert-major order; inside an expert the m-tiles vary fastest so that
    // neighbouring CTAs share the expert's B tile
    int lo = 0, hi = p.G;  // largest g with s_pre[g] * tiles_n <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] * p.tiles_n <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int mtiles = s_pre[g + 1] - s_pre[g];
    const int local = t - s_pre[g] * p.tiles_n;
    const int mt = local % mtiles, nt = local / mtiles;
    r.a_row = s_lo[g] + mt * kTileM;
    r.row_end = s_lo[g + 1];
    r.n0 = nt * BN;
    r.b_row = g * p.N + r.n0;
    r.g = g;
  }
  return r;
}

// kTmaOut (dense BF16, N a multiple of 8): C leaves only as whole-block TMA
// tensor stores; without the coalesced-store path in the same kernel the fold
// keeps its registers.
template <int kBScale, bool kOutF32, bool kGrouped, bool kPair, bool kAccum = false,
          bool kTmaOut = false>
__global__ void __launch_bounds__(kThreads, 1)
    fp8q_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmArgs p) {
  using C = Cfg<kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::kStages * C::kABytes;
  uint8_t *sC = smem + C::kTileBytes;  // output staging (1024-byte aligned)
  SmemCtl *ctl = reinterpret_cast<SmemCtl *>(sC + kStageCBytes);
  int *s_lo = reinterpret_cast<int *>(ctl + 1);  // grouped only (see tile_of)
  int *s_prefix = s_lo + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &ctl->abort_flag;
  const uint32_t rank = kPair ? cluster_ctarank() : 0;  // 0 = the CTA that issues the MMAs
  const int tile_first = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tile_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), C::kTemptyCount);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
  }
  if (warp == 1) {
    if (kPair) tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
    else tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tc_fence_before();
  }
  // barriers initialised and TMEM allocated in every CTA before any CTA of the
  // pair signals a peer
  __syncwarp();
  if (kPair) cluster_sync_all();
  else __syncthreads();
  // grouped: clamp the expert offsets into [0, M] and build the m-tile prefix
  int total_tiles;
  if (kGrouped) {
    for (int g = threadIdx.x; g <= p.G; g += blockDim.x) s_lo[g] = min(max(p.offs[g], 0), p.M);
    __syncthreads();
    if (threadIdx.x == 0) {
      // ranges never overlap: an expert starts no earlier than the previous
      // one ended, and a decreasing offset makes it empty; expert g then
      // owns rows s_lo[g] .. s_lo[g + 1]
      int acc = 0, prev_hi = 0;
      for (int g = 0; g < p.G; ++g) {
        const int lo = max(s_lo[g], prev_hi);
        const int hi = max(lo, s_lo[g + 1]);
        s_lo[g] = lo;
        s_prefix[g] = acc;
        acc += (hi - lo + C::kTileM - 1) / C::kTileM;
        prev_hi = hi;
      }
      s_lo[p.G] = prev_hi;
      s_prefix[p.G] = acc;
    }
    __syncthreads();
    total_tiles = s_prefix[p.G] * p.tiles_n;
  } else {
    total_tiles = p.tiles_m * p.tiles_n;
  }
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    // ================================================== epilogue
    const int ew = warp - 4;
    const int quarter = warp & 3;        // TMEM lanes this warp may access
    const int col_base = (ew >> 2) * kEpiCols;  // this warp's columns of the 256
    const int row_in_tile = static_cast<int>(rank) * BM + quarter * 32 + lane;
    // Per-column scales: the partial is read in 16-lane x 8-column fragments,
    // so that a thread needs the scales of 32 columns per K-group instead of
    // 128 (shared-memory reads of the column scales bound the fold otherwise).
    // Thread (g, q) = (lane / 4, lane % 4) holds rows g, g+8, g+16, g+24 of the
    // warp's 32 and columns 8i + 2q, 8i + 2q + 1 (i = 0..15) of its 128, as
    // acc[4i + r].  FP32 results leave straight from the fragments (the four
    // lanes of a quad write 32 contiguous bytes of a row); BF16 results go back
    // to one row per thread through shared memory first.
    constexpr bool kFrag = kBScale == FP8Q_BSCALE_ROW;
    const int g8 = lane >> 2, q4 = lane & 3;
    const int fr[4] = {g8, g8 + 8, g8 + 16, g8 + 24};
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int NB = (p.N + 127) / 128;
    // the TMEM-empty barriers live in the MMA-issuing CTA
    const uint32_t tempty_addr0 = kPair ? mapa_shared(smem_u32(&ctl->tempty[0]), 0)
                                        : smem_u32(&ctl->tempty[0]);
    const uint32_t tempty_addr1 = kPair ? mapa_shared(smem_u32(&ctl->tempty[1]), 0)
                                        : smem_u32(&ctl->tempty[1]);
    int tb = 0;
    uint32_t tphase = 0;
    uint32_t sb_iter = 0;
    bool ok = true;
    for (int t = tile_first; ok && t < total_tiles; t += tile_step) {
      const Tile tl = tile_of<kGrouped, C::kTileM>(t, p, s_lo, s_prefix);
      const int m = tl.a_row + row_in_tile;
      const int ncol0 = tl.n0 + col_base;
      const int nb = ncol0 / 128;
      const float *sb_g = p.sb;
      if (kGrouped) sb_g += static_cast<int64_t>(tl.g) * NB * p.num_kb;
      // Scales of K-group kb: sa of this lane's row (per-column kind: each
      // thread takes its four rows' scales from their lanes by shuffles); sb
      // of this warp's columns (block kinds: one value; per-column kind: lane
      // l loads the scales of columns c, c+1, c+8, c+9, c = 16(l % 8) + 2(l / 8),
      // and stores them at 4l..4l+3 of the warp's shared-memory row, so that
      // thread (g, q) finds the 32 scales of its columns at 32q..32q+31).
      // Pointers to group 0's values advance by one group's stride per group;
      // rows past M, blocks past N and columns past N read as 0.
      const bool sa_in = m < p.M;
      const float *sa_ptr = p.sa + (sa_in ? m : 0);
      const bool sb_in = kBScale == FP8Q_BSCALE_ROW || nb < NB;
      const float *sb_ptr =
          kBScale == FP8Q_BSCALE_BLOCK
              ? sb_g + static_cast<int64_t>(sb_in ? nb : 0) * (kGrouped ? p.num_kb : p.ld_sb)
          : kBScale == FP8Q_BSCALE_BLOCK_T ? p.sb + (sb_in ? nb : 0)
                                           : p.sb + ncol0 + 16 * (lane & 7) + 2 * (lane >> 3);
      const int64_t sb_step = kBScale == FP8Q_BSCALE_BLOCK ? 1 : p.ld_sb;
      // per-column kind: this lane's first column
      const int ncol = ncol0 + 16 * (lane & 7) + 2 * (lane >> 3);
      auto load_sa = [&]() { return sa_in ? __ldg(sa_ptr) : 0.0f; };
      auto load_sb = [&]() {
        return kBScale != FP8Q_BSCALE_ROW && sb_in ? __ldg(sb_ptr) : 0.0f;
      };
      auto load_sb4 = [&]() {
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (kBScale == FP8Q_BSCALE_ROW) {
          if (ncol + 0 < p.N) v.x = __ldg(sb_ptr + 0);
          if (ncol + 1 < p.N) v.y = __ldg(sb_ptr + 1);
          if (ncol + 8 < p.N) v.z = __ldg(sb_ptr + 8);
          if (ncol + 9 < p.N) v.w = __ldg(sb_ptr + 9);
        }
        return v;
      };
      static_assert(kEpiCols == 4 * 32, "per-column scale staging assumes 4 columns per lane");
      uint64_t acc[kEpiCols / 2];  // packed FP32 pairs: columns (2i, 2i+1) of this thread's
#pragma unroll
      for (int j = 0; j < kEpiCols / 2; ++j) acc[j] = 0ull;
      float sa_nx = p.num_kb > 0 ? load_sa() : 0.0f;
      float sb_nx = p.num_kb > 0 ? load_sb() : 0.0f;
      float4 sb4_nx = p.num_kb > 0 ? load_sb4() : make_float4(0.0f, 0.0f, 0.0f, 0.0f);

      for (int kb = 0; kb < p.num_kb; ++kb) {
        // the scales of group kb were loaded one iteration ago; fetch kb+1 now
        const float sa_v = sa_nx, sb_v = sb_nx;
        const float4 sb4 = sb4_nx;
        if (kb + 1 < p.num_kb) {
          sa_ptr += p.ld_sa;
          sb_ptr += sb_step;
          sa_nx = load_sa();
          sb_nx = load_sb();
          sb4_nx = load_sb4();
        }
        if (kBScale == FP8Q_BSCALE_ROW) {
          // the buffer written here was last read two K-groups ago, before the
          // previous iteration's __syncwarp
          *reinterpret_cast<float4 *>(&ctl->sb_warp[ew][sb_iter & 1][4 * lane]) = sb4;
          __syncwarp();
        }
        const uint64_t scale2 = pack_f32x2(sa_v * sb_v, sa_v * sb_v);
        uint64_t sa2f[4];  // per-column kind: this thread's four row scales, packed twice
        if (kFrag) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float v = __shfl_sync(0xffffffffu, sa_v, fr[r]);
            sa2f[r] = pack_f32x2(v, v);
          }
        }
        const bool got = mbar_wait_bounded(smem_u32(&ctl->tfull[tb]), tphase, abort_flag,
                                           &g_status, p.timeout_ns, FP8Q_ERR_TIMEOUT);
        if (!__all_sync(0xffffffffu, got)) {  // tcgen05.ld below needs the whole warp
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(tb * BN + col_base);
        if (kFrag) {
          // this thread's 32 column scales, eight per 32-column chunk
          const uint32_t sbw = smem_u32(&ctl->sb_warp[ew][sb_iter & 1][q4 * 32]);
#pragma unroll
          for (int c = 0; c < kEpiCols / 32; ++c) {
            uint32_t ra[16], rb[16];  // rows g, g+8 and g+16, g+24; columns 32c + 8k + 2q, +1
            tmem_ld_16x256b_x4(taddr + c * 32, ra);
            tmem_ld_16x256b_x4(taddr + (16u << 16) + c * 32, rb);
            tmem_wait_ld_tied(ra);
            reg_tie(rb);
            const uint4 s0 = ld_shared_v4(sbw + c * 32), s1 = ld_shared_v4(sbw + c * 32 + 16);
            const uint64_t sp[4] = {pack_u32x2(s0.x, s0.y), pack_u32x2(s0.z, s0.w),
                                    pack_u32x2(s1.x, s1.y), pack_u32x2(s1.z, s1.w)};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = 4 * c + k;
              ffma2(acc[4 * i + 0], pack_u32x2(ra[4 * k], ra[4 * k + 1]), fmul2(sp[k], sa2f[0]));
              ffma2(acc[4 * i + 1], pack_u32x2(ra[4 * k + 2], ra[4 * k + 3]), fmul2(sp[k], sa2f[1]));
              ffma2(acc[4 * i + 2], pack_u32x2(rb[4 * k], rb[4 * k + 1]), fmul2(sp[k], sa2f[2]));
              ffma2(acc[4 * i + 3], pack_u32x2(rb[4 * k + 2], rb[4 * k + 3]), fmul2(sp[k], sa2f[3]));
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < kEpiCols / 16; ++ch) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(taddr + ch * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ffma2(acc[ch * 8 + j], pack_u32x2(r[2 * j], r[2 * j + 1]), scale2);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kPair) mbar_arrive_cluster(tb ? tempty_addr1 : tempty_addr0);
          else mbar_arrive(smem_u32(&ctl->tempty[tb]));
        }
        tb ^= 1;
        if (tb == 0) tphase ^= 1;
        ++sb_iter;
      }
      if (!ok) break;

      if (kFrag && kOutF32 && !kGrouped) {
        // FP32 straight from the fragments: for each (i, r) the four lanes of a
        // quad write 32 contiguous bytes of one row (8 rows per instruction)
        const uint64_t pol = l2_evict_first_policy();
        const int wrow = tl.a_row + static_cast<int>(rank) * BM + quarter * 32;
#pragma unroll
        for (int i = 0; i < kEpiCols / 8; ++i) {
          const int col = ncol0 + 8 * i + 2 * q4;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = wrow + fr[r];
            if (row >= tl.row_end || col >= p.N) continue;
            float *dst = static_cast<float *>(p.c) + static_cast<int64_t>(row) * p.ldc + col;
            float2 v = unpack_f32x2(acc[4 * i + r]);
            if (col + 1 < p.N) {
              if (kAccum) {
                const float2 o = *reinterpret_cast<const float2 *>(dst);
                v.x = __fadd_rn(o.x, v.x);
                v.y = __fadd_rn(o.y, v.y);
              }
              st_global_b64_hint(dst, pack_f32x2(v.x, v.y), pol);
            } else {
              dst[0] = kAccum ? __fadd_rn(dst[0], v.x) : v.x;
            }
          }
        }
        continue;
      }
      if (kFrag) {
        // BF16: fragments -> one row per thread, 64 columns at a time, through
        // the warp's staging buffer (16-byte units XOR-swizzled by row), then
        // the row-per-thread store below
        const uint32_t buf = smem_u32(sC) + static_cast<uint32_t>(ew) * kStageWarpBytes;
        if (lane == 0) bulk_wait_group_read<0>();  // the previous tile's stores have read it
        __syncwarp();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t unit = static_cast<uint32_t>(2 * i + (q4 >> 1));
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const uint32_t row = static_cast<uint32_t>(fr[r]);
              st_shared_b64(buf + row * 256 + 16 * (unit ^ (row & 7)) + 8 * (q4 & 1),
                            acc[4 * (8 * h + i) + r]);
            }
          }
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const uint4 v = ld_shared_v4(buf + lane * 256 + 16 * (u ^ (lane & 7)));
            acc[32 * h + 2 * u] = pack_u32x2(v.x, v.y);
            acc[32 * h + 2 * u + 1] = pack_u32x2(v.z, v.w);
          }
          __syncwarp();
        }
      }

      // ---- store this warp's 32 rows x kEpiCols columns
      // BF16 (dense with N a multiple of 8, and grouped): the whole block goes
      // into the warp's 8 KB of shared memory (two 32-row x 128-byte boxes,
      // 128-byte swizzle) and leaves as two TMA tensor stores, which drain
      // while the next tile is folded.  Otherwise (FP32, C +=, a grouped warp
      // whose rows cross the expert's end -- the tensor map only clips at M
      // -- or a row segment ending inside a 16-byte unit past N -- tensor
      // stores clip the inner dimension at 16-byte granularity): coalesced
      // 64-byte blocks through the first 2 KB (each 16-byte store instruction
      // writes eight whole 64-byte row segments).
      constexpr int kEsz = kOutF32 ? 4 : 2;
      const int wrow0 = tl.a_row + row_in_tile - lane;
      if (ncol0 < p.N && wrow0 < tl.row_end) {
        const uint32_t stage = smem_u32(sC) + static_cast<uint32_t>(ew) * kStageWarpBytes;
        const bool rows_all = !kGrouped || wrow0 + 32 <= tl.row_end;
        const bool cols_ok = (p.N * kEsz) % 16 == 0 || ncol0 + kEpiCols <= p.N;
        // the previous tile's tensor stores must have read the buffer
        if (lane == 0) bulk_wait_group_read<0>();
        __syncwarp();
        static_assert(!kTmaOut || (!kOutF32 && !kAccum && !kGrouped), "dense BF16 only");
        if (kTmaOut || (kGrouped && !kOutF32 && rows_all && cols_ok)) {
          static_assert(kEpiCols == 128, "two 64-column boxes per warp");
#pragma unroll
          for (int q = 0; q < 16; ++q) {  // 16-byte unit q: columns 8q .. 8q+7
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 v = unpack_f32x2(acc[4 * q + e]);
              __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
              w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            st_shared_v4(stage + (q >> 3) * 4096 + lane * 128 + 16 * ((q & 7) ^ (lane & 7)),
                         make_uint4(w[0], w[1], w[2], w[3]));
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            // C is not read back: evict-first keeps the operands in L2
            const uint64_t pol = l2_evict_first_policy();
            tma_store_2d_hint(&tmC, stage, ncol0, wrow0, pol);
            if (ncol0 + 64 < p.N) tma_store_2d_hint(&tmC, stage + 4096, ncol0 + 64, wrow0, pol);
            bulk_commit_group();
          }
        } else if (!kTmaOut) {
          constexpr int kRowCols = 64 / kEsz;
#pragma unroll
          for (int j = 0; j < kEpiCols; j += kRowCols) {
            if (ncol0 + j >= p.N) break;
            uint4 u[4];
            if (kOutF32) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                u[q] = make_uint4(static_cast<uint32_t>(acc[j / 2 + 2 * q]),
                                  static_cast<uint32_t>(acc[j / 2 + 2 * q] >> 32),
                                  static_cast<uint32_t>(acc[j / 2 + 2 * q + 1]),
                                  static_cast<uint32_t>(acc[j / 2 + 2 * q + 1] >> 32));
            } else {
              uint32_t w[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float2 v = unpack_f32x2(acc[j / 2 + e]);
                __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
                w[e] = *reinterpret_cast<uint32_t *>(&h);
              }
#pragma unroll
              for (int q = 0; q < 4; ++q)
                u[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
            warp_store_block64<kEsz, kAccum>(stage, u, p.c, p.ldc, wrow0, tl.row_end, ncol0 + j,
                                             p.N, lane);
          }
        }
      }
    }
    // every tensor store of this warp has written global memory
    if (lane == 0) bulk_wait_group_all();
    // teardown (epilogue side): TMEM reads are complete
    __syncwarp();
    tc_fence_before();
    if (kPair) cluster_sync_all();
    else named_barrier_sync(1, kThreads);
    return;
  }

  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
  if (warp == 0) {
    // ================================================== TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_phase = 0;  // per-stage bit masks
      bool ok = true;
      for (int t = tile_first; ok && t < total_tiles; t += tile_step) {
        const Tile tl = tile_of<kGrouped, C::kTileM>(t, p, s_lo, s_prefix);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1, abort_flag, &g_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[stage]);
          if (kPair) {
            // both CTAs' copies complete on the MMA-issuing CTA's barrier, which
            // expects the bytes of both
            if (rank == 0) mbar_arrive_expect_tx(fb, C::kTxBytes);
            const uint32_t fb0 = mapa_shared(fb, 0);
            tma_load_2d_pair(smem_u32(sA + stage * C::kABytes), &tmA, fb0, kb * BK,
                             tl.a_row + static_cast<int>(rank) * BM);
            tma_load_2d_pair(smem_u32(sB + stage * C::kBBytes), &tmB, fb0, kb * BK,
                             tl.b_row + static_cast<int>(rank) * (BN / 2));
          } else {
            mbar_arrive_expect_tx(fb, C::kTxBytes);
            tma_load_2d(smem_u32(sA + stage * C::kABytes), &tmA, fb, kb * BK, tl.a_row);
            tma_load_2d(smem_u32(sB + stage * C::kBBytes), &tmB, fb, kb * BK, tl.b_row);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // drain: every armed stage's copy must land before the CTA exits (the
        // MMA-issuing CTA's barriers see both CTAs' copies; a second CTA of a
        // pair cannot wait on them and instead waits long enough for any copy)
        if (!kPair || rank == 0) {
          for (int s = 0; s < C::kStages; ++s)
            if (armed & (1u << s))
              mbar_wait_drain(smem_u32(&ctl->full[s]), (armed_phase >> s) & 1);
        }
        if (kPair) spin_ns(1000000);
      }
    }
  } else if (warp == 1) {
    // ================================================== MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int tb = 0;
      uint32_t tphase = 0;
      bool ok = true, issued = false;
      for (int t = tile_first; ok && t < total_tiles; t += tile_step) {
        for (int kb = 0; kb < p.num_kb; ++kb) {
          // (in a pair the epilogues of both CTAs arrive here; their tcgen05.ld
          // are ordered by the fences around the barrier, not by its scope)
          if (!mbar_wait_bounded(smem_u32(&ctl->tempty[tb]), tphase ^ 1, abort_flag,
                                 &g_status, p.timeout_ns, FP8Q_ERR_TIMEOUT) ||
              !mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_flag, &g_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * C::kBBytes));
          const uint32_t d = tmem_base + static_cast<uint32_t>(tb * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            if (kPair) mma_f8f6f4_pair(d, adesc + 2 * k, bdesc + 2 * k, C::kIdesc, k > 0 ? 1u : 0u);
            else mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, C::kIdesc, k > 0 ? 1u : 0u);
          }
          if (kPair) {
            mma_commit_pair_multicast(smem_u32(&ctl->empty[stage]), 0x3);
            mma_commit_pair_multicast(smem_u32(&ctl->tfull[tb]), 0x3);
          } else {
            mma_commit(smem_u32(&ctl->empty[stage]));
            mma_commit(smem_u32(&ctl->tfull[tb]));
          }
          issued = true;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
          tb ^= 1;
          if (tb == 0) tphase ^= 1;
        }
      }
      if (!ok && issued) {
        // drain: all MMAs issued so far must finish before TMEM is freed
        if (kPair) mma_commit_pair_multicast(smem_u32(&ctl->drain), 0x1);
        else mma_commit(smem_u32(&ctl->drain));
        mbar_wait_drain(smem_u32(&ctl->drain), 0);
      }
    }
  }
  // teardown (control side): wait for every warp (of both CTAs), then free TMEM
  __syncwarp();
  tc_fence_before();
  if (kPair) cluster_sync_all();
  else named_barrier_sync(1, kThreads);
  if (warp == 1) {
    tc_fence_after();
    if (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// One CTA waits on an mbarrier that nothing completes, with the same bounded
// wait as the GEMM; it must give up and record FP8Q_ERR_TIMEOUT.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, &g_status, timeout_ns, FP8Q_ERR_TIMEOUT);
  __syncthreads();
}

// ------------------------------------------------------------------ host
// 2-D byte tensor [rows][cols] with row pitch ld (bytes), box 128 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rows, cols, ld, 128, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// C [rows][cols] (BF16 or FP32) with row pitch ld elements, box 32 rows x 128
// bytes in the 128-byte swizzle: the epilogue's staged output boxes.
bool make_tmap_c(CUtensorMap *m, void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                 bool f32) {
  return make_tmap_2d(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      base, rows, cols, ld * (f32 ? 4 : 2), f32 ? 32 : 64, 32,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

// Launch one instantiation.  `work_tiles` is the number of output tiles (an
// upper bound for the grouped GEMM); the grid is persistent: one CTA (or one
// CTA pair) per SM that can hold one, never more than there are tiles.
template <int kBScale, bool kOutF32, bool kGrouped, bool kPair, bool kAccum = false,
          bool kTmaOut = false>
fp8q_status launch(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                   const GemmArgs &args, int64_t work_tiles, cudaStream_t s) {
  auto kern = fp8q_gemm_kernel<kBScale, kOutF32, kGrouped, kPair, kAccum, kTmaOut>;
  const size_t smem = smem_bytes(kGrouped, kPair);
  static int max_units[kMaxDevices] = {};  // co-resident CTAs (or CTA pairs) per device
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (kPair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  {
    std::lock_guard<std::mutex> lock(mu);
    if (max_units[dev] == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      int n = 0;
      if (kPair) {
        cfg.gridDim = dim3(2, 1, 1);
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
          return FP8Q_ERR_UNSUPPORTED;
      } else {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
          return FP8Q_ERR_CUDA;
      }
      max_units[dev] = n;
    }
  }
  const int64_t units = work_tiles < max_units[dev] ? work_tiles : max_units[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(units * (kPair ? 2 : 1)), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, args) == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// Tile shapes: kDensePair / kGroupedPair select CTA pairs (256 x 256 tiles)
// or single CTAs (128 x 256 tiles) for the dense and grouped GEMMs.
// C (FP32) += result: dense GEMMs only (gradient accumulation).
fp8q_status dispatch_accumulate(int bkind, const CUtensorMap &ta, const CUtensorMap &tb,
                                const CUtensorMap &tc, const GemmArgs &a, int64_t tiles,
                                cudaStream_t s) {
  switch (bkind) {
    case FP8Q_BSCALE_BLOCK:
      return launch<FP8Q_BSCALE_BLOCK, true, false, kDensePair, true>(ta, tb, tc, a, tiles, s);
    case FP8Q_BSCALE_BLOCK_T:
      return launch<FP8Q_BSCALE_BLOCK_T, true, false, kDensePair, true>(ta, tb, tc, a, tiles, s);
    default:
      return launch<FP8Q_BSCALE_ROW, true, false, kDensePair, true>(ta, tb, tc, a, tiles, s);
  }
}

template <bool kGrouped>
fp8q_status dispatch(int bkind, bool f32, const CUtensorMap &ta, const CUtensorMap &tb,
                     const CUtensorMap &tc, const GemmArgs &a, int64_t tiles, cudaStream_t s) {
  if (kGrouped) {
    return f32 ? launch<FP8Q_BSCALE_BLOCK, true, true, kGroupedPair>(ta, tb, tc, a, tiles, s)
               : launch<FP8Q_BSCALE_BLOCK, false, true, kGroupedPair>(ta, tb, tc, a, tiles, s);
  }
  // BF16 rows that end on a 16-byte unit take the tensor-store-only kernels
  const bool tma = !f32 && a.N % 8 == 0;
  switch (bkind) {
    case FP8Q_BSCALE_BLOCK:
      return f32   ? launch<FP8Q_BSCALE_BLOCK, true, false, kDensePair>(ta, tb, tc, a, tiles, s)
             : tma ? launch<FP8Q_BSCALE_BLOCK, false, false, kDensePair, false, true>(
                         ta, tb, tc, a, tiles, s)
                   : launch<FP8Q_BSCALE_BLOCK, false, false, kDensePair>(ta, tb, tc, a, tiles, s);
    case FP8Q_BSCALE_BLOCK_T:
      return f32   ? launch<FP8Q_BSCALE_BLOCK_T, true, false, kDensePair>(ta, tb, tc, a, tiles, s)
             : tma ? launch<FP8Q_BSCALE_BLOCK_T, false, false, kDensePair, false, true>(
                         ta, tb, tc, a, tiles, s)
                   : launch<FP8Q_BSCALE_BLOCK_T, false, false, kDensePair>(ta, tb, tc, a, tiles,
                                                                           s);
    default:
      return f32   ? launch<FP8Q_BSCALE_ROW, true, false, kDensePair>(ta, tb, tc, a, tiles, s)
             : tma ? launch<FP8Q_BSCALE_ROW, false, false, kDensePair, false, true>(
                         ta, tb, tc, a, tiles, s)
                   : launch<FP8Q_BSCALE_ROW, false, false, kDensePair>(ta, tb, tc, a, tiles, s);
  }
}

fp8q_status check_common(const void *a, int64_t lda, const void *b, int64_t ldb, const void *c,
                         int64_t ldc, int out_dtype, int64_t M, int64_t N, int64_t K,
                         const float *sa, int64_t ld_sa) {
  if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP32) return FP8Q_ERR_INVALID;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M >= (1ll << 31) - BM || N >= (1ll << 31) - BN || K >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  if (ldc < N || ld_sa < M) return FP8Q_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8Q_OK;
  if (K > 0 && (lda < K || ldb < K)) return FP8Q_ERR_SHAPE;
  if (!c || (K > 0 && (!a || !b || !sa))) return FP8Q_ERR_INVALID;
  const int64_t esz = out_dtype == FP8Q_OUT_FP32 ? 4 : 2;
  if (!aligned16(c) || (ldc * esz) % 16) return FP8Q_ERR_ALIGN;
  if (K > 0 && (!aligned16(a) || !aligned16(b) || lda % 16 || ldb % 16 || !aligned4(sa)))
    return FP8Q_ERR_ALIGN;
  return FP8Q_OK;
}

}  // namespace
}  // namespace fp8q

using namespace fp8q;

static fp8q_status gemm_entry(const void *a, int64_t lda, const float *sa, int64_t ld_sa,
                              const void *b, int64_t ldb, const float *sb, int64_t ld_sb,
                              int bscale_kind, void *c, int64_t ldc, int out_dtype, int64_t M,
                              int64_t N, int64_t K, void *stream, bool accumulate) {
  if (bscale_kind != FP8Q_BSCALE_BLOCK && bscale_kind != FP8Q_BSCALE_BLOCK_T &&
      bscale_kind != FP8Q_BSCALE_ROW)
    return FP8Q_ERR_INVALID;
  if (fp8q_status st = check_common(a, lda, b, ldb, c, ldc, out_dtype, M, N, K, sa, ld_sa))
    return st;
  if (M == 0 || N == 0) return FP8Q_OK;
  const int64_t KB = K / 128, NB = (N + 127) / 128;
  if (K > 0) {
    if (!sb || !aligned4(sb)) return sb ? FP8Q_ERR_ALIGN : FP8Q_ERR_INVALID;
    if (bscale_kind == FP8Q_BSCALE_BLOCK && ld_sb < KB) return FP8Q_ERR_SHAPE;
    if (bscale_kind == FP8Q_BSCALE_BLOCK_T && ld_sb < NB) return FP8Q_ERR_SHAPE;
    if (bscale_kind == FP8Q_BSCALE_ROW && ld_sb < N) return FP8Q_ERR_SHAPE;
  }
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  if (dev.max_smem_optin < static_cast<int>(smem_bytes(false, kDensePair)))
    return FP8Q_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  // K == 0: no loads happen; describe a dummy 1 x 128 tensor so the maps are valid.
  // Each CTA of a pair loads 128 rows of A and 128 rows (half a tile) of B.
  const void *abase = K > 0 ? a : c;
  const void *bbase = K > 0 ? b : c;
  CUtensorMap tc;
  if (!make_tmap_u8(&ta, abase, K > 0 ? M : 1, K > 0 ? K : 128, K > 0 ? lda : 128, BM) ||
      !make_tmap_u8(&tb, bbase, K > 0 ? N : 1, K > 0 ? K : 128, K > 0 ? ldb : 128,
                    kDensePair ? BN / 2 : BN) ||
      !make_tmap_c(&tc, c, M, N, ldc, out_dtype == FP8Q_OUT_FP32))
    return FP8Q_ERR_CUDA;
  GemmArgs args{};
  args.sa = sa;
  args.ld_sa = ld_sa;
  args.sb = sb;
  args.ld_sb = ld_sb;
  args.c = c;
  args.ldc = ldc;
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.num_kb = static_cast<int>(KB);
  args.tiles_m = static_cast<int>((M + Cfg<kDensePair>::kTileM - 1) / Cfg<kDensePair>::kTileM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.offs = nullptr;
  args.G = 0;
  args.timeout_ns = wait_timeout_ns().load();
  const int64_t tiles = static_cast<int64_t>(args.tiles_m) * args.tiles_n;
  if (tiles >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  if (accumulate)
    return dispatch_accumulate(bscale_kind, ta, tb, tc, args, tiles,
                               static_cast<cudaStream_t>(stream));
  return dispatch<false>(bscale_kind, out_dtype == FP8Q_OUT_FP32, ta, tb, tc, args, tiles,
                         static_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status fp8q_gemm(const void *a, int64_t lda, const float *sa, int64_t ld_sa,
                                 const void *b, int64_t ldb, const float *sb, int64_t ld_sb,
                                 int bscale_kind, void *c, int64_t ldc, int out_dtype, int64_t M,
                                 int64_t N, int64_t K, void *stream) {
  return gemm_entry(a, lda, sa, ld_sa, b, ldb, sb, ld_sb, bscale_kind, c, ldc, out_dtype, M, N, K,
                    stream, false);
}

extern "C" fp8q_status fp8q_gemm_accumulate(const void *a, int64_t lda, const float *sa,
                                            int64_t ld_sa, const void *b, int64_t ldb,
                                            const float *sb, int64_t ld_sb, int bscale_kind,
                                            float *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                            void *stream) {
  return gemm_entry(a, lda, sa, ld_sa, b, ldb, sb, ld_sb, bscale_kind, c, ldc, FP8Q_OUT_FP32, M, N,
                    K, stream, true);
}

extern "C" fp8q_status fp8q_grouped_gemm(const void *a, int64_t lda, const float *sa,
                                         int64_t ld_sa, const void *b, int64_t ldb,
                                         const float *sb, const int32_t *offs, int G, void *c,
                                         int64_t ldc, int out_dtype, int64_t M, int64_t N,
                                         int64_t K, void *stream) {
  if (G < 1 || G > kMaxGroups) return FP8Q_ERR_SHAPE;
  if (fp8q_status st = check_common(a, lda, b, ldb, c, ldc, out_dtype, M, N, K, sa, ld_sa))
    return st;
  if (M == 0 || N == 0) return FP8Q_OK;
  if (!offs) return FP8Q_ERR_INVALID;
  if (!aligned4(offs)) return FP8Q_ERR_ALIGN;
  if (static_cast<int64_t>(G) * N >= (1ll << 31) - BN) return FP8Q_ERR_SHAPE;
  if (K > 0 && (!sb || !aligned4(sb))) return sb ? FP8Q_ERR_ALIGN : FP8Q_ERR_INVALID;
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  if (dev.max_smem_optin < static_cast<int>(smem_bytes(true, kGroupedPair)))
    return FP8Q_ERR_UNSUPPORTED;
  const int64_t KB = K / 128;
  CUtensorMap ta, tb;
  const void *abase = K > 0 ? a : c;
  const void *bbase = K > 0 ? b : c;
  CUtensorMap tc;
  if (!make_tmap_u8(&ta, abase, K > 0 ? M : 1, K > 0 ? K : 128, K > 0 ? lda : 128, BM) ||
      !make_tmap_u8(&tb, bbase, K > 0 ? static_cast<uint64_t>(G) * N : 1, K > 0 ? K : 128,
                    K > 0 ? ldb : 128, kGroupedPair ? BN / 2 : BN) ||
      !make_tmap_c(&tc, c, M, N, ldc, out_dtype == FP8Q_OUT_FP32))
    return FP8Q_ERR_CUDA;
  GemmArgs args{};
  args.sa = sa;
  args.ld_sa = ld_sa;
  args.sb = sb;
  args.ld_sb = KB;
  args.c = c;
  args.ldc = ldc;
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.num_kb = static_cast<int>(KB);
  args.tiles_m = static_cast<int>((M + Cfg<kGroupedPair>::kTileM - 1) / Cfg<kGroupedPair>::kTileM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.offs = offs;
  args.G = G;
  args.timeout_ns = wait_timeout_ns().load();
  // upper bound on tiles: each expert adds at most one partial m-tile
  const int64_t bound = (static_cast<int64_t>(args.tiles_m) + G) * args.tiles_n;
  if (bound >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  return dispatch<true>(FP8Q_BSCALE_BLOCK, out_dtype == FP8Q_OUT_FP32, ta, tb, tc, args, bound,
                        static_cast<cudaStream_t>(stream));
}

extern "C" fp8q_status fp8q_sync_status(void *stream) {
  auto s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP8Q_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return FP8Q_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return FP8Q_ERR_CUDA;
  }
  const fp8q_status q = quant_status_take(s);
  const fp8q_status x = mx_status_take(s);
  if (v != 0) return static_cast<fp8q_status>(v);
  return q != FP8Q_OK ? q : x;
}

extern "C" void fp8q_set_wait_timeout_ns(uint64_t ns) {
  wait_timeout_ns().store(ns ? ns : 2000000000ull);
}

extern "C" fp8q_status fp8q_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  return launch_on(wait_timeout_probe_kernel, dim3(1), dim3(32), 0,
                   static_cast<cudaStream_t>(stream), timeout_ns);
}
