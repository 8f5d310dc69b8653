// gemm_mx.cu -- the per-group-scaled FP8 GEMM for power-of-two scales, on the
// tensor cores' block-scaled MMA (sm_103a).
//
//   C[m][n] = sum_kb 2^ea(m,kb) * 2^eb(n,kb) * sum_{k in kb} a[m][k] * b[n][k]
//
// With the method's power-of-two scaling factors (dssusan.co.kr post 91437,
// paragraph 1) every scale is 2^e, and the pages' recommendation that tensor
// cores take the group scales themselves (same post, paragraph 3) is what
// Blackwell's microscaling MMA does ("Deepseek - Not For everyone",
// paragraph 3): tcgen05.mma kind::mxf8f6f4.block_scale multiplies each
// 32-wide K block of A and B by 2^e (UE8M0 exponents held in tensor memory)
// inside the MMA.  The 128-wide group's exponent is used for its four K
// blocks.  Products of powers of two are exact, so the result is the same
// product as the FP32-scale path's, accumulated over the whole K in the FP32
// TMEM accumulator with no per-group fold by the CUDA cores.
//
// Roles (384 threads; CTA pairs, tile 256 x BN, one MMA thread per pair):
//   warp 0      TMA producer: this CTA's 128 rows of A and BN/2 rows of B per
//               K-group into a kStages ring, completing on the leading CTA's
//               "full" barrier.
//   warp 1      MMA issuer (leading CTA): per K-group 4 x tcgen05.mma
//               .cta_group::2 .kind::mxf8f6f4 .block_scale (M=256, N=BN,
//               K=32) into one of kAccBufs TMEM accumulators (BN columns each,
//               alternating by tile), reading the scale exponents of the
//               current scale stage.
//   warps 4-11  scale producers and epilogue.  The TMEM columns after the
//               accumulators hold kSfStages scale stages of 16 columns, each
//               with the exponents of four consecutive K-groups, one byte per
//               group: warps 4-7 write the A exponents of their rows (column
//               +q for lane quarter q), warps 8-11 the B exponents of the
//               tile's BN columns (columns +8.., the same in every lane
//               quarter).  At the end of a tile they read its accumulator
//               (each thread BN/2 columns of its row), release it and store C
//               through a 2 KB shared-memory buffer per warp, 64 bytes of
//               each row at a time, as coalesced 16-byte stores with an L2
//               evict-first policy.
//
// Shipped shape: BN = 256 with one accumulator (columns 0-255) and 16 scale
// stages (columns 256-511).  The epilogue writes scale stages up to 6 ahead
// into the next tile before it drains the current one; with two
// accumulators (any BN that is a multiple of 128 and fits) it drains tile t-1
// while the tensor cores fill tile t.  Narrower tiles measured slower: a
// 224-wide MMA takes about as long as a 256-wide one, and 256 x 128 tiles with
// two accumulators lose more to per-group overhead than they gain.
// A scale that is not a power of two (2^-127 .. 2^127) is a caller error: the
// kernel uses its exponent and records FP8Q_ERR_INVALID in its status word.
// Every wait is bounded in time (as in the FP32-scale GEMM).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fp8q.h"
#include "fp8q_host.cuh"
#include "fp8q_ptx.cuh"

namespace fp8q {

// Device status word of this kernel (read and cleared by fp8q_sync_status).
__device__ int g_mx_status;

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kAccBufs = 1;                     // TMEM accumulators (tiles in flight)
constexpr int kTileM = 2 * BM;                  // C rows per pair tile
constexpr uint32_t kABytes = BM * BK;           // per CTA per stage
constexpr uint32_t kBBytes = (BN / 2) * BK;     // per CTA per stage (half the columns)
constexpr uint32_t kTxBytes = 2 * (kABytes + kBBytes);
constexpr int kStages = 210 * 1024 / (kABytes + kBBytes) < 10
                            ? static_cast<int>(210 * 1024 / (kABytes + kBBytes))
                            : 10;               // operand ring depth
constexpr size_t kRingBytes = static_cast<size_t>(kStages) * (kABytes + kBBytes);
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + kEpiWarps * 32;
constexpr int kLaunchRegs = 168;                // must match ptxas' count (checked by the build)
// Register split: the control warpgroup gives registers back, the epilogue
// warpgroups take them; kernels that prepare per-column scale words in warps
// 2-3 keep more in the control warpgroup for the loads in flight there.
constexpr int kCtlRegs = 40, kEpiRegs = 232;
constexpr int kCtlRegsPrep = 56, kEpiRegsPrep = 224;
static_assert(kCtlRegsPrep + 2 * kEpiRegsPrep <= 3 * kLaunchRegs, "register split must fit");
static_assert(kCtlRegs + 2 * kEpiRegs <= 3 * kLaunchRegs, "register split must fit the launch");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kAccBufs * BN;    // accumulators: columns [0, kAccCols)
constexpr int kSfStages = (512 - kAccCols) / 16 < 16 ? (512 - kAccCols) / 16 : 16;
constexpr uint32_t kSfStageCols = 16;
constexpr uint32_t kSfbOffset = 8;              // B exponents at +8..+14 of a stage
constexpr int kBCols32 = BN / 32;               // 32-column groups of B per tile (7)
constexpr int kEpiCols = BN / 2;                // columns each epilogue thread drains (112)
static_assert(BN % 128 == 0 && kEpiCols % 16 == 0,
              "tile width: whole 128-column scale blocks (and full-rate MMA widths)");
// stages of the next tile written before the previous tile is drained: with
// one accumulator the drain gates the next tile, so a short run-ahead keeps it
// from waiting on the current tile's last stages
constexpr int kRunAhead = kAccBufs == 1 ? 6 : kSfStages;
static_assert(kAccCols + kSfStages * kSfStageCols <= kTmemCols, "TMEM budget");
static_assert(kSfStages >= 2, "the scale ring needs TMEM columns beside the accumulators");
constexpr int kGroupsPerStage = 4;              // one byte per K-group in a 32-bit cell
// Scale producers: true = warps 4-7 write A exponents and warps 8-11 B
// exponents; false = warps 4-7 write both (warps 8-11 only drain).
constexpr bool kSplitSides = true;
constexpr int kProducerWarps = kSplitSides ? 8 : 4;
constexpr int kGroupM = 16;                     // L2 rasterisation band (m-tiles)
constexpr uint64_t kDrainNs = 1000000000ull;

struct MxArgs {
  const float *sa;
  int64_t ld_sa;
  const float *sb;
  int64_t ld_sb;
  void *c;
  int64_t ldc;
  int M, N;
  int num_kb;
  int tiles_m, tiles_n;
  const int32_t *offs;  // grouped only: expert row offsets [G + 1] (device)
  int G;
  uint64_t timeout_ns;
};

// Per-column B scale preparation (dense GEMMs with FP8Q_BSCALE_ROW): every
// scale stage needs 32 FP32 scales per lane (256 columns x 4 K-groups) turned
// into 8 UE8M0 words per lane.  The two otherwise idle warps of the first
// warpgroup (warp 2: column groups 0-3, warp 3: 4-7) load and convert them
// into a shared-memory ring kPrepSlots stages ahead, and the B producer warps,
// which must write the words into their own TMEM lane quarters and which also
// drain the accumulator, only copy ready words.  Loaded by the producers
// themselves, a global load's latency (about a microsecond under the GEMM's
// own L2 traffic) fell on the critical path each time they caught up after a
// drain; block scales (8 values per stage) do not need this.
constexpr int kPrepSlots = 8;
constexpr size_t kPrepBytes = static_cast<size_t>(kPrepSlots) * 8 * 32 * 4;  // [slot][c][lane]

struct alignas(8) MxCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t sfull[kSfStages];   // leading CTA: scale stage written (16 warp arrivals)
  uint64_t sempty[kSfStages];  // every CTA: scale stage consumed by the MMAs
  uint64_t tfull[kAccBufs];    // every CTA: accumulator complete
  uint64_t tempty[kAccBufs];   // leading CTA: accumulator read (16 warp arrivals)
  uint64_t drain;
  uint64_t pready[kPrepSlots];  // every CTA: both preparing warps wrote a stage's B words
  uint64_t pfree[kPrepSlots];   // every CTA: the four B producer warps read them
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kMaxGroups = 1024;
constexpr size_t kGroupTables = 3 * (kMaxGroups + 1) * sizeof(int);
// Output staging: 2 KB per epilogue warp (32 rows x 64 bytes) for coalesced
// stores of the drained accumulator.
constexpr size_t kStageBytes = kEpiWarps * 2048;
constexpr size_t kSmemBytes = 1024 + kRingBytes + kStageBytes + sizeof(MxCtl);

__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kDrainNs) return;
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < ns) {
  }
}

// UE8M0 exponent byte of a power-of-two FP32 scale; `bad` is set for any other
// value (the exponent field is then used, clamped below the NaN code).
__device__ __forceinline__ uint32_t ue8m0_of(float s, bool &bad) {
  const uint32_t b = __float_as_uint(s);
  if (b == 0x00400000u) return 0u;  // 2^-127, the one subnormal power of two in range
  const uint32_t e = (b >> 23) & 0xFFu;
  if ((b & 0x807FFFFFu) != 0u || e == 0u || e == 0xFFu) bad = true;
  return e < 0xFFu ? e : 0xFEu;
}

struct MxTile {
  int m0;       // first row of the pair tile (of A and of C)
  int row_end;  // rows >= row_end are not stored (the expert's end, or M)
  int b_row;    // first row of B (expert g's rows start at g * N)
  int n0;       // first column
  int g;        // expert (grouped) or 0
};

// Dense: bands of kGroupM m-tiles for L2 reuse.  Grouped: expert-major, m-tiles
// fastest; s_lo / s_hi = clamped row range of expert g, s_pre[g] = m-tiles of
// the experts before g.
template <bool kGrouped>
__device__ __forceinline__ MxTile mx_tile_of(int t, const MxArgs &p, const int *s_lo,
                                             const int *s_hi, const int *s_pre) {
  MxTile r;
  if (!kGrouped) {
    const int band_tiles = kGroupM * p.tiles_n;
    const int band = t / band_tiles, within = t - band * band_tiles;
    const int mt0 = band * kGroupM;
    const int rows = min(kGroupM, p.tiles_m - mt0);
    r.m0 = (mt0 + within % rows) * kTileM;
    r.row_end = p.M;
    r.n0 = (within / rows) * BN;
    r.b_row = r.n0;
    r.g = 0;
  } else {
    int lo = 0, hi = p.G;  // largest g with s_pre[g] * tiles_n <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] * p.tiles_n <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int mtiles = s_pre[g + 1] - s_pre[g];
    const int local = t - s_pre[g] * p.tiles_n;
    r.m0 = s_lo[g] + (local % mtiles) * kTileM;
    r.row_end = s_hi[g];
    r.n0 = (local / mtiles) * BN;
    r.b_row = g * p.N + r.n0;
    r.g = g;
  }
  return r;
}

template <int kBScale, bool kOutF32, bool kAccum, bool kGrouped = false>
__global__ void __launch_bounds__(kThreads, 1)
    fp8q_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const MxArgs p) {
  // per-column B scales of a dense GEMM are prepared in warps 2-3
  constexpr bool kPrep = kBScale == FP8Q_BSCALE_ROW && !kGrouped;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages * kABytes;
  uint8_t *sC = smem + kRingBytes;  // output staging (1024-byte aligned)
  uint32_t *prep_b = reinterpret_cast<uint32_t *>(sC + kStageBytes);  // [slot][8][32]
  MxCtl *ctl = reinterpret_cast<MxCtl *>(sC + kStageBytes + (kPrep ? kPrepBytes : 0));
  int *s_lo = reinterpret_cast<int *>(ctl + 1);  // grouped only (see mx_tile_of)
  int *s_hi = s_lo + (kMaxGroups + 1);
  int *s_pre = s_hi + (kMaxGroups + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = &ctl->abort_flag;
  const uint32_t rank = cluster_ctarank();  // 0 = the CTA that issues the MMAs
  const int tile_first = static_cast<int>(blockIdx.x >> 1);
  const int tile_step = static_cast<int>(gridDim.x >> 1);
  const int nst = (p.num_kb + kGroupsPerStage - 1) / kGroupsPerStage;  // scale stages per tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&ctl->full[i]), 1);
      mbar_init(smem_u32(&ctl->empty[i]), 1);
    }
    for (int i = 0; i < kSfStages; ++i) {
      mbar_init(smem_u32(&ctl->sfull[i]), 2 * kProducerWarps);
      mbar_init(smem_u32(&ctl->sempty[i]), 1);
    }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(smem_u32(&ctl->tfull[i]), 1);
      mbar_init(smem_u32(&ctl->tempty[i]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    for (int i = 0; i < kPrepSlots; ++i) {
      mbar_init(smem_u32(&ctl->pready[i]), 2);
      mbar_init(smem_u32(&ctl->pfree[i]), 4);
    }
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
    tc_fence_before();
  }
  __syncwarp();
  cluster_sync_all();
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
        s_pre[g] = acc;
        acc += (hi - lo + kTileM - 1) / kTileM;
        prev_hi = hi;
      }
      s_pre[p.G] = acc;
    }
    __syncthreads();
    total_tiles = s_pre[p.G] * p.tiles_n;
  } else {
    total_tiles = p.tiles_m * p.tiles_n;
  }
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPrep ? kEpiRegsPrep : kEpiRegs));
    // ================================================== scale producers + epilogue
    const int ew = warp - 4;
    const int q = warp & 3;          // lane quarter this warp may access
    const bool producer = kSplitSides || ew < 4;
    const bool do_a = producer && (!kSplitSides || ew < 4);   // writes A exponents
    const bool do_b = producer && (!kSplitSides || ew >= 4);  // writes B exponents
    const int col_half = ew >> 2;    // epilogue: columns [kEpiCols * col_half, +kEpiCols)
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int row_in_tile = static_cast<int>(rank) * BM + q * 32 + lane;
    const uint32_t sfull0 = mapa_shared(smem_u32(&ctl->sfull[0]), 0);
    const uint32_t tempty0 = mapa_shared(smem_u32(&ctl->tempty[0]), 0);
    int ss = 0;           // next scale stage slot to write
    uint32_t sphase = 0;  // its phase
    uint32_t tphase = 0;  // bit b: phase of tfull[b]
    bool ok = true;

    // Scale production walks a cursor over (tile, stage) in the order the MMA
    // consumes stages.  The raw FP32 scales of the stage at the cursor were
    // loaded one stage earlier: a global load takes about a microsecond under
    // the GEMM's own L2 traffic, as long as the tensor cores take to consume a
    // stage, so loading them at use would put that latency on the critical path.
    //   A warps: raw[0..3] = sa of this thread's row, K-groups 4 js .. 4 js + 3.
    //   B warps, per-column scales: raw[4 c + j] = sb of column n0 + 32 c + lane.
    //   B warps, block scales: raw[4 h + j] = the scale of 128-column block h
    //   of the tile (column group c lies in block c / 4).
    constexpr int kRawB = kBScale == FP8Q_BSCALE_ROW ? kBCols32 * kGroupsPerStage
                                                     : (BN / 128) * kGroupsPerStage;
    // split: a warp loads one side, from raw[0]; combined: A at [0, 4), B after
    constexpr int kOffB = kSplitSides ? 0 : kGroupsPerStage;
    static_assert(!kPrep || kSplitSides, "prepared B words assume split sides");
    constexpr int kRaw = kPrep ? kGroupsPerStage
                         : kSplitSides ? (kRawB > kGroupsPerStage ? kRawB : kGroupsPerStage)
                                       : kGroupsPerStage + kRawB;
    const int NB = (p.N + 127) / 128;
    auto load_raw = [&](int t, int js, float (&r)[kRaw]) {
      if (kPrep && !do_a) return;  // the B words come from warps 2-3
      const MxTile tl = mx_tile_of<kGrouped>(t, p, s_lo, s_hi, s_pre);
      const int kb0 = js * kGroupsPerStage;
#pragma unroll
      for (int i = 0; i < kRaw; ++i) r[i] = 1.0f;
      if (do_a) {
        const int m = tl.m0 + row_in_tile;
#pragma unroll
        for (int j = 0; j < kGroupsPerStage; ++j)
          if (kb0 + j < p.num_kb && m < p.M)
            r[j] = __ldg(p.sa + static_cast<int64_t>(kb0 + j) * p.ld_sa + m);
        if (kSplitSides) return;
      }
      float *rb = r + kOffB;
      if (!do_b) {
      } else if (kBScale == FP8Q_BSCALE_ROW) {
#pragma unroll
        for (int c = 0; c < kBCols32; ++c) {
          const int n = tl.n0 + 32 * c + lane;
#pragma unroll
          for (int j = 0; j < kGroupsPerStage; ++j)
            if (kb0 + j < p.num_kb && n < p.N)
              rb[4 * c + j] = __ldg(p.sb + static_cast<int64_t>(kb0 + j) * p.ld_sb + n);
        }
      } else {
        // columns past N in a partial block read zero-filled B rows, so the
        // block's own scale is as good as any for them
        const float *sbg = kGrouped ? p.sb + static_cast<int64_t>(tl.g) * NB * p.num_kb : p.sb;
#pragma unroll
        for (int h = 0; h < BN / 128; ++h) {
          const int nb = tl.n0 / 128 + h;
#pragma unroll
          for (int j = 0; j < kGroupsPerStage; ++j)
            if (kb0 + j < p.num_kb && nb < NB)
              rb[4 * h + j] = kBScale == FP8Q_BSCALE_BLOCK
                                  ? __ldg(sbg + static_cast<int64_t>(nb) * p.ld_sb + kb0 + j)
                                  : __ldg(p.sb + static_cast<int64_t>(kb0 + j) * p.ld_sb + nb);
        }
      }
    };
    float raw[kRaw];
    int gp = 0;                          // stages produced (prepared-word ring position)
    int cur_t = tile_first, cur_js = 0;  // production cursor
    if (cur_t < total_tiles) load_raw(cur_t, 0, raw);

    // Write the stage at the cursor into slot ss and advance the cursor.
    auto produce = [&]() -> bool {
      int nt = cur_t, njs = cur_js + 1;
      if (njs == nst) {
        nt += tile_step;
        njs = 0;
      }
      if (!producer) {  // only walks the cursor, in step with the producers
        cur_t = nt;
        cur_js = njs;
        return true;
      }
      float nxt[kRaw];
      if (nt < total_tiles) load_raw(nt, njs, nxt);
      // prepared words of this stage (warps 2-3), copied to registers and
      // released before the wait for the TMEM scale slot
      uint32_t pw[8];
      if (kPrep && do_b) {
        const int pslot = gp % kPrepSlots;
        const bool ready = mbar_wait_bounded(
            smem_u32(&ctl->pready[pslot]), static_cast<uint32_t>(gp / kPrepSlots) & 1u,
            abort_flag, &g_mx_status, p.timeout_ns, FP8Q_ERR_TIMEOUT);
        if (!__all_sync(0xffffffffu, ready)) return false;
#pragma unroll
        for (int c = 0; c < 8; ++c) pw[c] = prep_b[(pslot * 8 + c) * 32 + lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->pfree[pslot]));
        ++gp;
      }
      const bool got = mbar_wait_bounded(smem_u32(&ctl->sempty[ss]), sphase ^ 1, abort_flag,
                                         &g_mx_status, p.timeout_ns, FP8Q_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, got)) return false;  // tcgen05.st needs the whole warp
      tc_fence_after();
      const uint32_t col = kAccCols + static_cast<uint32_t>(ss) * kSfStageCols;
      bool bad = false;
      if (do_a) {
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < kGroupsPerStage; ++j) w |= ue8m0_of(raw[j], bad) << (8 * j);
        tmem_st_32x32b_x1(tmem_base + lane_addr + col + static_cast<uint32_t>(q), w);
      }
      if (do_b && !(kSplitSides && do_a)) {
        uint32_t w[8];
        if (kPrep) {
#pragma unroll
          for (int c = 0; c < 8; ++c) w[c] = pw[c];
        } else if (kBScale == FP8Q_BSCALE_ROW) {  // one word per 32-column group
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t word = 0x7F7F7F7Fu;  // column group past the tile: unused, 2^0
            if (c < kBCols32) {
              word = 0;
#pragma unroll
              for (int j = 0; j < kGroupsPerStage; ++j)
                word |= ue8m0_of(raw[kOffB + 4 * c + j], bad) << (8 * j);
            }
            w[c] = word;
          }
        } else {  // one word per 128-column block, repeated for its 4 column groups
          uint32_t wb[BN / 128];
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < kGroupsPerStage; ++j)
              word |= ue8m0_of(raw[kOffB + 4 * h + j], bad) << (8 * j);
            wb[h] = word;
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) w[c] = c < kBCols32 ? wb[c / 4] : 0x7F7F7F7Fu;
        }
        tmem_st_32x32b_x8(tmem_base + lane_addr + col + kSfbOffset, w);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(&g_mx_status, 0, FP8Q_ERR_INVALID);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(sfull0 + static_cast<uint32_t>(ss) * 8u);
      if (++ss == kSfStages) {
        ss = 0;
        sphase ^= 1;
      }
#pragma unroll
      for (int i = 0; i < kRaw; ++i) raw[i] = nxt[i];
      cur_t = nt;
      cur_js = njs;
      return true;
    };

    // Read tile t's accumulator (buffer buf_acc), release it, store C through the
    // warp's shared-memory buffer (coalesced 16-byte stores).
    auto drain = [&](int t, int buf_acc) -> bool {
      const bool got = mbar_wait_bounded(smem_u32(&ctl->tfull[buf_acc]), (tphase >> buf_acc) & 1u,
                                         abort_flag, &g_mx_status, p.timeout_ns,
                                         FP8Q_ERR_TIMEOUT);
      if (!__all_sync(0xffffffffu, got)) return false;
      tphase ^= 1u << buf_acc;
      tc_fence_after();
      constexpr int kChunks = kEpiCols / 16;
      const uint32_t taddr = tmem_base + lane_addr +
                             static_cast<uint32_t>(buf_acc * BN + col_half * kEpiCols);
      const MxTile tl = mx_tile_of<kGrouped>(t, p, s_lo, s_hi, s_pre);
      const int ncol0 = tl.n0 + col_half * kEpiCols;
      const int wrow0 = tl.m0 + row_in_tile - lane;
      const bool warp_ok = wrow0 < tl.row_end && ncol0 < p.N;  // warp-uniform
      const uint32_t buf = smem_u32(sC) + static_cast<uint32_t>(ew) * 2048u;
      if (kOutF32 && kPrep) {
        // FP32 out, per-column scales: these warps hold no raw scales, so the
        // whole row of kEpiCols values is read first and the accumulator is
        // released before any store; stores go 64 bytes (16 columns) of each
        // row at a time through the warp's buffer
        uint32_t v[kChunks][16];
#pragma unroll
        for (int i = 0; i < kChunks; ++i) tmem_ld_32x32b_x16(taddr + i * 16, v[i]);
        tmem_wait_ld_tied(v[0]);
#pragma unroll
        for (int i = 1; i < kChunks; ++i) reg_tie(v[i]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(buf_acc) * 8u);
        if (warp_ok) {
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
            const int col = ncol0 + i * 16;
            if (col >= p.N) break;
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u[q] = make_uint4(v[i][4 * q], v[i][4 * q + 1], v[i][4 * q + 2], v[i][4 * q + 3]);
            warp_store_block64<4, kAccum>(buf, u, p.c, p.ldc, wrow0, tl.row_end, col, p.N, lane);
          }
        }
      } else if (kOutF32) {
        // FP32 out: two halves of kEpiCols / 2 columns, the first stored while
        // the second is read, which halves the registers the drain holds; the
        // accumulator is released after the last TMEM read.  Stores go 64
        // bytes (16 columns) of each row at a time through the warp's buffer.
        constexpr int kHalf = kChunks / 2;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t v[kHalf][16];
#pragma unroll
          for (int i = 0; i < kHalf; ++i) tmem_ld_32x32b_x16(taddr + (hf * kHalf + i) * 16, v[i]);
          tmem_wait_ld_tied(v[0]);
#pragma unroll
          for (int i = 1; i < kHalf; ++i) reg_tie(v[i]);
          if (hf == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(buf_acc) * 8u);
          }
          if (!warp_ok) continue;
#pragma unroll
          for (int i = 0; i < kHalf; ++i) {
            const int col = ncol0 + (hf * kHalf + i) * 16;
            if (col >= p.N) break;
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u[q] = make_uint4(v[i][4 * q], v[i][4 * q + 1], v[i][4 * q + 2], v[i][4 * q + 3]);
            warp_store_block64<4, kAccum>(buf, u, p.c, p.ldc, wrow0, tl.row_end, col, p.N, lane);
          }
        }
      } else {  // BF16 out: 64 bytes (32 columns) of each row at a time
        uint32_t v[kChunks][16];
#pragma unroll
        for (int i = 0; i < kChunks; ++i) tmem_ld_32x32b_x16(taddr + i * 16, v[i]);
        tmem_wait_ld_tied(v[0]);
#pragma unroll
        for (int i = 1; i < kChunks; ++i) reg_tie(v[i]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(buf_acc) * 8u);
        if (warp_ok) {
#pragma unroll
          for (int i = 0; i < kChunks; i += 2) {
            const int col = ncol0 + i * 16;
            if (col >= p.N) break;
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c0 = i * 16 + 2 * e;
              __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[c0 / 16][c0 % 16]),
                                                       __uint_as_float(v[c0 / 16][c0 % 16 + 1]));
              w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            uint4 u[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              u[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            warp_store_block64<2, false>(buf, u, p.c, p.ldc, wrow0, tl.row_end, col, p.N, lane);
          }
        }
      }
      return true;
    };

    // Tile t's accumulator is read at the top of the next iteration, while the
    // tensor cores fill the other buffer with tile t + step; the scale stages
    // of the next tile are written ahead (up to kSfStages of them: stage js of
    // the next tile reuses the slot of this tile's stage nst + js - kSfStages,
    // so no wait depends on the next tile's own MMAs).
    int prev_t = -1, prev_buf = 0;
    int i = 0;
    for (int t = tile_first; ok && t < total_tiles; t += tile_step, ++i) {
      if (prev_t >= 0 && !(ok = drain(prev_t, prev_buf))) break;
      while (ok && cur_t == t) ok = produce();  // the rest of this tile's stages
      const int lim = nst < kRunAhead ? nst : kRunAhead;
      while (ok && cur_t == t + tile_step && cur_t < total_tiles && cur_js < lim) ok = produce();
      prev_t = t;
      prev_buf = i % kAccBufs;
    }
    if (ok && prev_t >= 0) ok = drain(prev_t, prev_buf);
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    return;
  }

  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPrep ? kCtlRegsPrep : kCtlRegs));
  if (warp == 0) {
    // ================================================== TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      for (int t = tile_first; ok && t < total_tiles; t += tile_step) {
        const MxTile tl = mx_tile_of<kGrouped>(t, p, s_lo, s_hi, s_pre);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1, abort_flag,
                                 &g_mx_status, p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[stage]);
          if (rank == 0) mbar_arrive_expect_tx(fb, kTxBytes);
          const uint32_t fb0 = mapa_shared(fb, 0);
          tma_load_2d_pair(smem_u32(sA + stage * kABytes), &tmA, fb0, kb * BK,
                           tl.m0 + static_cast<int>(rank) * BM);
          tma_load_2d_pair(smem_u32(sB + stage * kBBytes), &tmB, fb0, kb * BK,
                           tl.b_row + static_cast<int>(rank) * (BN / 2));
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          for (int s = 0; s < kStages; ++s)
            if (armed & (1u << s)) mbar_wait_drain(smem_u32(&ctl->full[s]), (armed_phase >> s) & 1);
        }
        spin_ns(1000000);
      }
    }
  } else if (kPrep && (warp == 2 || warp == 3)) {
    // ================================================== per-column B scale words
    // warp 2 prepares column groups 0-3, warp 3 groups 4-7, of scale stage g
    // (consumption order) into slot g % kPrepSlots
    const int c0 = (warp - 2) * 4;
    int g = 0;
    bool ok = true;
    for (int t = tile_first; ok && t < total_tiles; t += tile_step) {
      const MxTile tl = mx_tile_of<kGrouped>(t, p, s_lo, s_hi, s_pre);
      for (int js = 0; js < nst; ++js, ++g) {
        const int kb0 = js * kGroupsPerStage;
        const int slot = g % kPrepSlots;
        // loads first: their latency overlaps the wait for the slot
        float v[4 * kGroupsPerStage];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int n = tl.n0 + 32 * (c0 + c) + lane;
#pragma unroll
          for (int j = 0; j < kGroupsPerStage; ++j)
            v[4 * c + j] = kb0 + j < p.num_kb && n < p.N
                               ? __ldg(p.sb + static_cast<int64_t>(kb0 + j) * p.ld_sb + n)
                               : 1.0f;
        }
        const bool got = mbar_wait_bounded(
            smem_u32(&ctl->pfree[slot]), (static_cast<uint32_t>(g / kPrepSlots) & 1u) ^ 1u,
            abort_flag, &g_mx_status, p.timeout_ns, FP8Q_ERR_TIMEOUT);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        bool bad = false;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w = 0;
#pragma unroll
          for (int j = 0; j < kGroupsPerStage; ++j) w |= ue8m0_of(v[4 * c + j], bad) << (8 * j);
          prep_b[(slot * 8 + c0 + c) * 32 + lane] = c0 + c < kBCols32 ? w : 0x7F7F7F7Fu;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicCAS(&g_mx_status, 0, FP8Q_ERR_INVALID);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->pready[slot]));
      }
    }
  } else if (warp == 1) {
    // ================================================== MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int ss = 0;
      uint32_t sphase = 0;
      uint32_t tphase = 0;  // bit b: phase of tempty[b]
      bool ok = true, issued = false;
      int i = 0;
      for (int t = tile_first; ok && t < total_tiles; t += tile_step, ++i) {
        // this tile's accumulator must have been read out (both CTAs)
        const int buf = i % kAccBufs;
        if (!mbar_wait_bounded(smem_u32(&ctl->tempty[buf]), ((tphase >> buf) & 1u) ^ 1u,
                               abort_flag, &g_mx_status, p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
          ok = false;
          break;
        }
        tphase ^= 1u << buf;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          const uint32_t j = static_cast<uint32_t>(kb % kGroupsPerStage);
          if (j == 0) {
            if (!mbar_wait_bounded(smem_u32(&ctl->sfull[ss]), sphase, abort_flag, &g_mx_status,
                                   p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
              ok = false;
              break;
            }
          }
          if (!mbar_wait_bounded(smem_u32(&ctl->full[stage]), phase, abort_flag, &g_mx_status,
                                 p.timeout_ns, FP8Q_ERR_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(sA + stage * kABytes));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + stage * kBBytes));
          const uint32_t sfa = tmem_base + kAccCols + static_cast<uint32_t>(ss) * kSfStageCols;
          const uint32_t idesc = idesc_mx_e4m3(kTileM, BN, j, j);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_mx_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, sfa, sfa + kSfbOffset,
                        (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair_multicast(smem_u32(&ctl->empty[stage]), 0x3);
          if (j == kGroupsPerStage - 1 || kb == p.num_kb - 1) {
            mma_commit_pair_multicast(smem_u32(&ctl->sempty[ss]), 0x3);
            if (++ss == kSfStages) {
              ss = 0;
              sphase ^= 1;
            }
          }
          issued = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(smem_u32(&ctl->tfull[buf]), 0x3);
      }
      if (!ok && issued) {
        mma_commit_pair_multicast(smem_u32(&ctl->drain), 0x1);
        mbar_wait_drain(smem_u32(&ctl->drain), 0);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host
template <int kBScale, bool kOutF32, bool kAccum, bool kGrouped = false>
fp8q_status launch_mx(const CUtensorMap &ta, const CUtensorMap &tb, const MxArgs &args,
                      int64_t tiles, cudaStream_t s) {
  auto kern = fp8q_gemm_mx_kernel<kBScale, kOutF32, kAccum, kGrouped>;
  constexpr size_t smem = kSmemBytes + (kGrouped ? kGroupTables : 0) +
                          (kBScale == FP8Q_BSCALE_ROW && !kGrouped ? kPrepBytes : 0);
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  static int max_pairs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP8Q_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // CTA pairs
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (max_pairs[dev] == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem)) != cudaSuccess)
        return FP8Q_ERR_CUDA;
      int n = 0;
      cfg.gridDim = dim3(2, 1, 1);
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1)
        return FP8Q_ERR_UNSUPPORTED;
      max_pairs[dev] = n;
    }
  }
  const int64_t pairs = tiles < max_pairs[dev] ? tiles : max_pairs[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, args) == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <bool kAccum>
fp8q_status dispatch_mx(int bkind, bool f32, const CUtensorMap &ta, const CUtensorMap &tb,
                        const MxArgs &a, int64_t tiles, cudaStream_t s) {
  if (kAccum) {
    switch (bkind) {
      case FP8Q_BSCALE_BLOCK: return launch_mx<FP8Q_BSCALE_BLOCK, true, true>(ta, tb, a, tiles, s);
      case FP8Q_BSCALE_BLOCK_T:
        return launch_mx<FP8Q_BSCALE_BLOCK_T, true, true>(ta, tb, a, tiles, s);
      default: return launch_mx<FP8Q_BSCALE_ROW, true, true>(ta, tb, a, tiles, s);
    }
  }
  switch (bkind) {
    case FP8Q_BSCALE_BLOCK:
      return f32 ? launch_mx<FP8Q_BSCALE_BLOCK, true, false>(ta, tb, a, tiles, s)
                 : launch_mx<FP8Q_BSCALE_BLOCK, false, false>(ta, tb, a, tiles, s);
    case FP8Q_BSCALE_BLOCK_T:
      return f32 ? launch_mx<FP8Q_BSCALE_BLOCK_T, true, false>(ta, tb, a, tiles, s)
                 : launch_mx<FP8Q_BSCALE_BLOCK_T, false, false>(ta, tb, a, tiles, s);
    default:
      return f32 ? launch_mx<FP8Q_BSCALE_ROW, true, false>(ta, tb, a, tiles, s)
                 : launch_mx<FP8Q_BSCALE_ROW, false, false>(ta, tb, a, tiles, s);
  }
}

fp8q_status mx_entry(const void *a, int64_t lda, const float *sa, int64_t ld_sa, const void *b,
                     int64_t ldb, const float *sb, int64_t ld_sb, int bkind, void *c, int64_t ldc,
                     int out_dtype, int64_t M, int64_t N, int64_t K, void *stream, bool accum) {
  if (bkind != FP8Q_BSCALE_BLOCK && bkind != FP8Q_BSCALE_BLOCK_T && bkind != FP8Q_BSCALE_ROW)
    return FP8Q_ERR_INVALID;
  if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP32) return FP8Q_ERR_INVALID;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M >= (1ll << 31) - kTileM || N >= (1ll << 31) - BN || K >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  if (ldc < N || ld_sa < M) return FP8Q_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8Q_OK;
  if (!c) return FP8Q_ERR_INVALID;
  const int64_t esz = out_dtype == FP8Q_OUT_FP32 ? 4 : 2;
  if (!aligned16(c) || (ldc * esz) % 16) return FP8Q_ERR_ALIGN;
  const int64_t KB = K / 128, NB = (N + 127) / 128;
  auto st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  if (fp8q_status e = device_info(dev)) return e;
  if (K == 0) {  // empty sum: C = 0 (or C unchanged when accumulating)
    if (accum) return FP8Q_OK;
    return cudaMemset2DAsync(c, static_cast<size_t>(ldc * esz), 0, static_cast<size_t>(N * esz),
                             static_cast<size_t>(M), st) == cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
  }
  if (lda < K || ldb < K) return FP8Q_ERR_SHAPE;
  if (!a || !b || !sa || !sb) return FP8Q_ERR_INVALID;
  if (!aligned16(a) || !aligned16(b) || lda % 16 || ldb % 16 || !aligned4(sa) || !aligned4(sb))
    return FP8Q_ERR_ALIGN;
  if (bkind == FP8Q_BSCALE_BLOCK && ld_sb < KB) return FP8Q_ERR_SHAPE;
  if (bkind == FP8Q_BSCALE_BLOCK_T && ld_sb < NB) return FP8Q_ERR_SHAPE;
  if (bkind == FP8Q_BSCALE_ROW && ld_sb < N) return FP8Q_ERR_SHAPE;
  if (dev.max_smem_optin < static_cast<int>(kSmemBytes + kPrepBytes)) return FP8Q_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, M, K, lda, 128, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, N, K, ldb, 128, BN / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8Q_ERR_CUDA;
  MxArgs args{};
  args.sa = sa;
  args.ld_sa = ld_sa;
  args.sb = sb;
  args.ld_sb = ld_sb;
  args.c = c;
  args.ldc = ldc;
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.num_kb = static_cast<int>(KB);
  args.tiles_m = static_cast<int>((M + kTileM - 1) / kTileM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.timeout_ns = wait_timeout_ns().load();
  const int64_t tiles = static_cast<int64_t>(args.tiles_m) * args.tiles_n;
  if (tiles >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  return accum ? dispatch_mx<true>(bkind, true, ta, tb, args, tiles, st)
               : dispatch_mx<false>(bkind, out_dtype == FP8Q_OUT_FP32, ta, tb, args, tiles, st);
}

}  // namespace

fp8q_status mx_status_take(cudaStream_t s) {
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP8Q_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mx_status, sizeof(int)) != cudaSuccess) return FP8Q_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_mx_status, &zero, sizeof(int)) != cudaSuccess) return FP8Q_ERR_CUDA;
  }
  return static_cast<fp8q_status>(v);
}

}  // namespace fp8q

using namespace fp8q;

extern "C" fp8q_status fp8q_gemm_pow2(const void *a, int64_t lda, const float *sa, int64_t ld_sa,
                                      const void *b, int64_t ldb, const float *sb, int64_t ld_sb,
                                      int bscale_kind, void *c, int64_t ldc, int out_dtype,
                                      int64_t M, int64_t N, int64_t K, void *stream) {
  return mx_entry(a, lda, sa, ld_sa, b, ldb, sb, ld_sb, bscale_kind, c, ldc, out_dtype, M, N, K,
                  stream, false);
}

extern "C" fp8q_status fp8q_gemm_pow2_accumulate(const void *a, int64_t lda, const float *sa,
                                                 int64_t ld_sa, const void *b, int64_t ldb,
                                                 const float *sb, int64_t ld_sb, int bscale_kind,
                                                 float *c, int64_t ldc, int64_t M, int64_t N,
                                                 int64_t K, void *stream) {
  return mx_entry(a, lda, sa, ld_sa, b, ldb, sb, ld_sb, bscale_kind, c, ldc, FP8Q_OUT_FP32, M, N,
                  K, stream, true);
}

extern "C" fp8q_status fp8q_grouped_gemm_pow2(const void *a, int64_t lda, const float *sa,
                                              int64_t ld_sa, const void *b, int64_t ldb,
                                              const float *sb, const int32_t *offs, int G,
                                              void *c, int64_t ldc, int out_dtype, int64_t M,
                                              int64_t N, int64_t K, void *stream) {
  if (G < 1 || G > kMaxGroups) return FP8Q_ERR_SHAPE;
  if (out_dtype != FP8Q_OUT_BF16 && out_dtype != FP8Q_OUT_FP32) return FP8Q_ERR_INVALID;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0) return FP8Q_ERR_SHAPE;
  if (M >= (1ll << 31) - kTileM || K >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  if (static_cast<int64_t>(G) * N >= (1ll << 31) - BN) return FP8Q_ERR_SHAPE;
  if (ldc < N || ld_sa < M) return FP8Q_ERR_SHAPE;
  if (M == 0 || N == 0) return FP8Q_OK;
  if (!c || !offs) return FP8Q_ERR_INVALID;
  const int64_t esz = out_dtype == FP8Q_OUT_FP32 ? 4 : 2;
  if (!aligned16(c) || (ldc * esz) % 16 || !aligned4(offs)) return FP8Q_ERR_ALIGN;
  auto st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  if (fp8q_status e = device_info(dev)) return e;
  if (K == 0) return FP8Q_ERR_SHAPE;  // an expert's empty sum is not written by this path
  if (lda < K || ldb < K) return FP8Q_ERR_SHAPE;
  if (!a || !b || !sa || !sb) return FP8Q_ERR_INVALID;
  if (!aligned16(a) || !aligned16(b) || lda % 16 || ldb % 16 || !aligned4(sa) || !aligned4(sb))
    return FP8Q_ERR_ALIGN;
  if (dev.max_smem_optin < static_cast<int>(kSmemBytes + kGroupTables)) return FP8Q_ERR_UNSUPPORTED;
  const int64_t KB = K / 128;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, a, M, K, lda, 128, BM,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, b, static_cast<uint64_t>(G) * N, K, ldb,
                    128, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return FP8Q_ERR_CUDA;
  MxArgs args{};
  args.sa = sa;
  args.ld_sa = ld_sa;
  args.sb = sb;
  args.ld_sb = KB;
  args.c = c;
  args.ldc = ldc;
  args.M = static_cast<int>(M);
  args.N = static_cast<int>(N);
  args.num_kb = static_cast<int>(KB);
  args.tiles_m = static_cast<int>((M + kTileM - 1) / kTileM);
  args.tiles_n = static_cast<int>((N + BN - 1) / BN);
  args.offs = offs;
  args.G = G;
  args.timeout_ns = wait_timeout_ns().load();
  // upper bound on tiles: each expert adds at most one partial m-tile
  const int64_t bound = (static_cast<int64_t>(args.tiles_m) + G) * args.tiles_n;
  if (bound >= (1ll << 31)) return FP8Q_ERR_SHAPE;
  return out_dtype == FP8Q_OUT_FP32
             ? launch_mx<FP8Q_BSCALE_BLOCK, true, false, true>(ta, tb, args, bound, st)
             : launch_mx<FP8Q_BSCALE_BLOCK, false, false, true>(ta, tb, args, bound, st);
}
