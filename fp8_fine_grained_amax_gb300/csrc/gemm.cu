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
//   warp 1      MMA issuer (one thread): per K-group, 4 x tcgen05.mma
//               (kind::f8f6f4, M=128, N=256, K=32) into one of two TMEM
//               partial buffers, then tcgen05.commit to release the ring slot
//               and to signal the partial.
//   warps 2-3   idle (they complete the first warpgroup).
//   warps 4-11  epilogue: tcgen05.ld the partial (each thread one row, 128
//               columns, 16 at a time), acc += P * sa(m,kb) * sb(n,kb) in FP32
//               registers with packed two-lane FMAs (fma.rn.f32x2), release the
//               TMEM buffer; after the last group, store C as FP32 or
//               round-to-nearest-even BF16.  The scales of group kb+1 are
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

#include <atomic>
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

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kStages = 4;
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
constexpr uint32_t kABytes = BM * BK;
constexpr uint32_t kBBytes = BN * BK;
constexpr uint32_t kIdesc = idesc_e4m3_f32(BM, BN);
constexpr int kGroupM = 16;   // L2 rasterisation band (m-tiles) for the dense GEMM
constexpr int kMaxGroups = 1024;
constexpr uint64_t kDrainNs = 1000000000ull;  // 1 s for draining after an abort

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

// Shared-memory layout (dynamic; tiles 1024-byte aligned for the swizzle).
struct alignas(8) SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t sbfull[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  float sb_row[2][BN];
};

constexpr size_t kTileBytes = static_cast<size_t>(kStages) * (kABytes + kBBytes);

__host__ __device__ constexpr size_t smem_bytes(bool grouped) {
  return 1024 /* alignment slack */ + kTileBytes + sizeof(SmemCtl) +
         (grouped ? 3 * (kMaxGroups + 1) * sizeof(int) : 0);
}

struct Tile {
  int a_row;    // first row of A (and of C) covered by the tile
  int row_end;  // rows >= row_end are not stored
  int b_row;    // first row of B (expert-offset for grouped)
  int n0;       // first output column
  int g;        // expert (grouped) or 0
};

// Grouped tables in shared memory: s_lo[g] / s_hi[g] = clamped row range of
// expert g, s_pre[g] = number of m-tiles of experts before g (s_pre[G] = all).
template <bool kGrouped>
__device__ __forceinline__ Tile tile_of(int t, const GemmArgs &p, const int *s_lo,
                                        const int *s_hi, const int *s_pre) {
  Tile r;
  if (!kGrouped) {
    const int band_tiles = kGroupM * p.tiles_n;
    const int band = t / band_tiles, within = t - band * band_tiles;
    const int mt0 = band * kGroupM;
    const int rows = min(kGroupM, p.tiles_m - mt0);
    const int mt = mt0 + within % rows, nt = within / rows;
    r.a_row = mt * BM;
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
    r.a_row = s_lo[g] + mt * BM;
    r.row_end = s_hi[g];
    r.n0 = nt * BN;
    r.b_row = g * p.N + r.n0;
    r.g = g;
  }
  return r;
}

template <int kBScale, bool kOutF32, bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    fp8q_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages * kABytes;
  SmemCtl *ctl = reinterpret_cast<SmemCtl *>(smem + kTileBytes);
  int *s_lo = reinterpret_cast<int *>(ctl + 1);  // grouped only (see tile_of)
  int *s_hi = s_lo + (kMaxGroups + 1);
  int *s_prefix = s_hi + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &ctl->abort_flag;

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), kEpiWarps);
      mbar_init(smem_u32(&ctl->sbfull[i]), kEpiWarps * 32);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  // grouped: clamp the expert offsets into [0, M] and build the m-tile prefix
  int total_tiles;
  if (kGrouped) {
    for (int g = threadIdx.x; g <= p.G; g += blockDim.x) s_lo[g] = min(max(p.offs[g], 0), p.M);
    __syncthreads();
    if (threadIdx.x == 0) {
      // ranges never overlap: an expert starts no earlier than the previous
      // one ended, and a decreasing offset makes it empty
      int acc = 0, prev_hi = 0;
      for (int g = 0; g < p.G; ++g) {
        const int lo = max(s_lo[g], prev_hi);
        const int hi = max(lo, s_lo[g + 1]);
        s_lo[g] = lo;
        s_hi[g] = hi;
        s_prefix[g] = acc;
        acc += (hi - lo + BM - 1) / BM;
        prev_hi = hi;
      }
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
    const int row_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const int NB = (p.N + 127) / 128;
    const int et = ew * 32 + lane;  // staging slot for per-column scales (< BN stages)
    int tb = 0;
    uint32_t tphase = 0;
    uint32_t sb_iter = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
      const Tile tl = tile_of<kGrouped>(t, p, s_lo, s_hi, s_prefix);
      const int m = tl.a_row + row_in_tile;
      const bool row_in = m < p.M;
      const int ncol0 = tl.n0 + col_base;
      const int nb = ncol0 / 128;
      const float *sb_g = p.sb;
      if (kGrouped) sb_g += static_cast<int64_t>(tl.g) * NB * p.num_kb;
      // scales of K-group kb: sa of this row; sb of this warp's 128 columns
      // (block kinds) or of column n0 + et (per-column kind, staged in smem)
      auto load_sa = [&](int kb) {
        return row_in ? __ldg(p.sa + static_cast<int64_t>(kb) * p.ld_sa + m) : 0.0f;
      };
      auto load_sb = [&](int kb) {
        if (kBScale == FP8Q_BSCALE_BLOCK)
          return nb < NB ? __ldg(sb_g + static_cast<int64_t>(nb) * (kGrouped ? p.num_kb : p.ld_sb) +
                                 kb)
                         : 0.0f;
        if (kBScale == FP8Q_BSCALE_BLOCK_T)
          return nb < NB ? __ldg(p.sb + static_cast<int64_t>(kb) * p.ld_sb + nb) : 0.0f;
        const int n = tl.n0 + et;
        return (et < BN && n < p.N) ? __ldg(p.sb + static_cast<int64_t>(kb) * p.ld_sb + n) : 0.0f;
      };
      uint64_t acc[kEpiCols / 2];  // packed FP32 pairs: columns (2i, 2i+1) of this thread's
#pragma unroll
      for (int j = 0; j < kEpiCols / 2; ++j) acc[j] = 0ull;
      float sa_nx = p.num_kb > 0 ? load_sa(0) : 0.0f;
      float sb_nx = p.num_kb > 0 ? load_sb(0) : 0.0f;

      for (int kb = 0; kb < p.num_kb; ++kb) {
        // the scales of group kb were loaded one iteration ago; fetch kb+1 now
        const float sa_v = sa_nx, sb_v = sb_nx;
        if (kb + 1 < p.num_kb) {
          sa_nx = load_sa(kb + 1);
          sb_nx = load_sb(kb + 1);
        }
        if (kBScale == FP8Q_BSCALE_ROW) {
          // per-column scales, staged through shared memory by all 256 threads
          if (et < BN) ctl->sb_row[sb_iter & 1][et] = sb_v;
          mbar_arrive(smem_u32(&ctl->sbfull[sb_iter & 1]));
          // every lane waits; the warp then agrees (and reconverges) on the outcome
          const bool got = mbar_wait_bounded(smem_u32(&ctl->sbfull[sb_iter & 1]),
                                             (sb_iter >> 1) & 1, abort_flag, &g_status,
                                             p.timeout_ns, FP8Q_ERR_TIMEOUT);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        const uint64_t scale2 = pack_f32x2(sa_v * sb_v, sa_v * sb_v);
        const uint64_t sa2 = pack_f32x2(sa_v, sa_v);
        const bool got = mbar_wait_bounded(smem_u32(&ctl->tfull[tb]), tphase, abort_flag,
                                           &g_status, p.timeout_ns, FP8Q_ERR_TIMEOUT);
        if (!__all_sync(0xffffffffu, got)) {  // tcgen05.ld below needs the whole warp
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(tb * BN + col_base);
#pragma unroll
        for (int ch = 0; ch < kEpiCols / 16; ++ch) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(taddr + ch * 16, r);
          tmem_wait_ld();
          if (kBScale == FP8Q_BSCALE_ROW) {
            const uint64_t *sbr =
                reinterpret_cast<const uint64_t *>(&ctl->sb_row[sb_iter & 1][col_base + ch * 16]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ffma2(acc[ch * 8 + j], pack_u32x2(r[2 * j], r[2 * j + 1]), fmul2(sbr[j], sa2));
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ffma2(acc[ch * 8 + j], pack_u32x2(r[2 * j], r[2 * j + 1]), scale2);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[tb]));
        tb ^= 1;
        if (tb == 0) tphase ^= 1;
        ++sb_iter;
      }
      if (!ok) break;

      // ---- store the tile row (128 columns of row m)
      if (m < tl.row_end && ncol0 < p.N) {
        const bool full = ncol0 + kEpiCols <= p.N;
        if (kOutF32) {
          float *crow = static_cast<float *>(p.c) + static_cast<int64_t>(m) * p.ldc + ncol0;
#pragma unroll
          for (int j = 0; j < kEpiCols; j += 4) {
            const float2 lo = unpack_f32x2(acc[j / 2]), hi = unpack_f32x2(acc[j / 2 + 1]);
            if (full || ncol0 + j + 4 <= p.N) {
              *reinterpret_cast<float4 *>(crow + j) = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
              const float v[4] = {lo.x, lo.y, hi.x, hi.y};
              for (int e = 0; e < 4; ++e)
                if (ncol0 + j + e < p.N) crow[j + e] = v[e];
            }
          }
        } else {
          __nv_bfloat16 *crow =
              static_cast<__nv_bfloat16 *>(p.c) + static_cast<int64_t>(m) * p.ldc + ncol0;
#pragma unroll
          for (int j = 0; j < kEpiCols; j += 8) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 v = unpack_f32x2(acc[j / 2 + e]);
              __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
              w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            if (full || ncol0 + j + 8 <= p.N) {
              *reinterpret_cast<uint4 *>(crow + j) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              for (int e = 0; e < 8; ++e)
                if (ncol0 + j + e < p.N)
                  reinterpret_cast<uint16_t *>(crow)[j + e] =
                      static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
            }
          }
        }
      }
    }
    // teardown (epilogue side): TMEM reads are complete
    __syncwarp();
    tc_fence_before();
    named_barrier_sync(1, kThreads);
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
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        const Tile tl = tile_of<kGrouped>(t, p, s_lo, s_hi, s_prefix);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1, abort_flag, &g_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[stage]);
          mbar_arrive_expect_tx(fb, kABytes + kBBytes);
          tma_load_2d(smem_u32(sA + stage * kABytes), &tmA, fb, kb * BK, tl.a_row);
          tma_load_2d(smem_u32(sB + stage * kBBytes), &tmB, fb, kb * BK, tl.b_row);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // drain: every armed stage's copy must land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (armed & (1u << s)) mbar_wait_drain(smem_u32(&ctl->full[s]), (armed_phase >> s) & 1);
      }
    }
  } else if (warp == 1) {
    // ================================================== MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int tb = 0;
      uint32_t tphase = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->tempty[tb]), tphase ^ 1, abort_flag, &g_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT) ||
              !mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_flag, &g_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * kBBytes));
          const uint32_t d = tmem_base + static_cast<uint32_t>(tb * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, kIdesc, k > 0 ? 1u : 0u);
          mma_commit(smem_u32(&ctl->empty[stage]));
          mma_commit(smem_u32(&ctl->tfull[tb]));
          issued = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
          tb ^= 1;
          if (tb == 0) tphase ^= 1;
        }
      }
      if (!ok && issued) {
        // drain: all MMAs issued so far must finish before TMEM is freed
        mma_commit(smem_u32(&ctl->drain));
        mbar_wait_drain(smem_u32(&ctl->drain), 0);
      }
    }
  }
  // teardown (control side): wait for every warp, then free TMEM
  __syncwarp();
  tc_fence_before();
  named_barrier_sync(1, kThreads);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
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
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D byte tensor [rows][cols] with row pitch ld (bytes), box 128 x box_rows,
// 128-byte swizzle, zero fill outside the tensor.
bool make_tmap_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                  uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

template <int kBScale, bool kOutF32, bool kGrouped>
fp8q_status launch(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &args, int grid,
                   cudaStream_t s) {
  auto kern = fp8q_gemm_kernel<kBScale, kOutF32, kGrouped>;
  static bool attr_set[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_bytes(kGrouped))) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      attr_set[dev] = true;
    }
  }
  kern<<<grid, kThreads, smem_bytes(kGrouped), s>>>(ta, tb, args);
  return launch_status();
}

template <bool kGrouped>
fp8q_status dispatch(int bkind, bool f32, const CUtensorMap &ta, const CUtensorMap &tb,
                     const GemmArgs &a, int grid, cudaStream_t s) {
  if (kGrouped) {
    return f32 ? launch<FP8Q_BSCALE_BLOCK, true, true>(ta, tb, a, grid, s)
               : launch<FP8Q_BSCALE_BLOCK, false, true>(ta, tb, a, grid, s);
  }
  switch (bkind) {
    case FP8Q_BSCALE_BLOCK:
      return f32 ? launch<FP8Q_BSCALE_BLOCK, true, false>(ta, tb, a, grid, s)
                 : launch<FP8Q_BSCALE_BLOCK, false, false>(ta, tb, a, grid, s);
    case FP8Q_BSCALE_BLOCK_T:
      return f32 ? launch<FP8Q_BSCALE_BLOCK_T, true, false>(ta, tb, a, grid, s)
                 : launch<FP8Q_BSCALE_BLOCK_T, false, false>(ta, tb, a, grid, s);
    default:
      return f32 ? launch<FP8Q_BSCALE_ROW, true, false>(ta, tb, a, grid, s)
                 : launch<FP8Q_BSCALE_ROW, false, false>(ta, tb, a, grid, s);
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

extern "C" fp8q_status fp8q_gemm(const void *a, int64_t lda, const float *sa, int64_t ld_sa,
                                 const void *b, int64_t ldb, const float *sb, int64_t ld_sb,
                                 int bscale_kind, void *c, int64_t ldc, int out_dtype, int64_t M,
                                 int64_t N, int64_t K, void *stream) {
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
  if (dev.max_smem_optin < static_cast<int>(smem_bytes(false))) return FP8Q_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  // K == 0: no loads happen; describe a dummy 1 x 128 tensor so the maps are valid
  const void *abase = K > 0 ? a : c;
  const void *bbase = K > 0 ? b : c;
  if (!make_tmap_u8(&ta, abase, K > 0 ? M : 1, K > 0 ? K : 128, K > 0 ? lda : 128, BM) ||
      !make_tmap_u8(&tb, bbase, K > 0 ? N : 1, K > 0 ? K : 128, K > 0 ? ldb : 128, BN))
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
  args.tiles_m = static_cast<int>((M + BM - 1) / BM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.offs = nullptr;
  args.G = 0;
  args.timeout_ns = g_timeout_ns.load();
  const int64_t tiles = static_cast<int64_t>(args.tiles_m) * args.tiles_n;
  if (tiles >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  return dispatch<false>(bscale_kind, out_dtype == FP8Q_OUT_FP32, ta, tb, args, grid,
                         static_cast<cudaStream_t>(stream));
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
  if (dev.max_smem_optin < static_cast<int>(smem_bytes(true))) return FP8Q_ERR_UNSUPPORTED;
  const int64_t KB = K / 128;
  CUtensorMap ta, tb;
  const void *abase = K > 0 ? a : c;
  const void *bbase = K > 0 ? b : c;
  if (!make_tmap_u8(&ta, abase, K > 0 ? M : 1, K > 0 ? K : 128, K > 0 ? lda : 128, BM) ||
      !make_tmap_u8(&tb, bbase, K > 0 ? static_cast<uint64_t>(G) * N : 1, K > 0 ? K : 128,
                    K > 0 ? ldb : 128, BN))
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
  args.tiles_m = static_cast<int>((M + BM - 1) / BM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.offs = offs;
  args.G = G;
  args.timeout_ns = g_timeout_ns.load();
  // upper bound on tiles: each expert adds at most one partial m-tile
  const int64_t bound = (static_cast<int64_t>(args.tiles_m) + G) * args.tiles_n;
  if (bound >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  const int grid = static_cast<int>(bound < dev.sm_count ? bound : dev.sm_count);
  return dispatch<true>(FP8Q_BSCALE_BLOCK, out_dtype == FP8Q_OUT_FP32, ta, tb, args, grid,
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
  return static_cast<fp8q_status>(v);
}

extern "C" void fp8q_set_wait_timeout_ns(uint64_t ns) {
  g_timeout_ns.store(ns ? ns : 2000000000ull);
}

extern "C" fp8q_status fp8q_selftest_wait_timeout(uint64_t timeout_ns, void *stream) {
  DeviceInfo dev;
  if (fp8q_status st = device_info(dev)) return st;
  wait_timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns);
  return launch_status();
}
