// fp8q_ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, TMA (bulk tensor
// copies), tcgen05 (TMEM allocation, MMA, commit, TMEM loads), E4M3 packing.
// Every wrapper is a single documented PTX instruction (or a short fixed
// sequence); nothing here is taken from a vendor library.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace fp8q {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA / tensor-core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with the given parity has completed.  The suspend-time
// hint (1 us) lets the hardware park the waiting thread until the phase
// completes instead of returning at once; the callers' loops still bound the
// total wait.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Returns true when the phase completed; false when the CTA's
// abort flag is raised or `limit_ns` has passed (then it raises the abort
// flag itself and records `code` in the device status word).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag,
                                                  int *status_word, uint64_t limit_ns,
                                                  int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicExch(status_word, code);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
// 2-D tiled bulk tensor copy global -> shared, completing on an mbarrier.
// c0 is the innermost (contiguous) coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const void *tmap, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// 2-D tiled bulk tensor copy shared -> global (the box is clipped at the
// tensor's bounds), tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const void *tmap, uint32_t smem_src, int32_t c0,
                                             int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(smem_src)
      : "memory");
}
// L2 policy that makes the written lines the first to go: for a GEMM's C,
// which no one reads back while the operands are still being reused.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_store_2d_hint(const void *tmap, uint32_t smem_src, int32_t c0,
                                                  int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(smem_src), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void st_global_v4_hint(void *ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void st_global_b64_hint(void *ptr, uint64_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(ptr), "l"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four 8x8 16-bit matrices from shared memory, transposed: lanes 8i..8i+7
// give the addresses of the 8 rows (16 bytes each) of matrix i; thread t
// receives, for matrix i, elements (row 2(t%4), column t/4) in the low half
// and (row 2(t%4)+1, column t/4) in the high half of r[i].
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t smem_row_addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_row_addr)
               : "memory");
}

// Two 16x16 byte matrices from shared memory, transposed: lanes 16i..16i+15
// give the addresses of the 16 rows (16 bytes each) of matrix i; lane 4g + t
// receives, for matrix i, rows 4t..4t+3 of column g in the bytes of
// r[2i] (row 4t in the low byte) and the same rows of column g + 8 in r[2i+1].
__device__ __forceinline__ void ldmatrix_b8_x2_trans(uint32_t smem_row_addr, uint32_t *r) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_row_addr)
               : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}
__device__ __forceinline__ void st_shared_b64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared.b64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// One warp writes a block of 32 rows x 64 bytes of a row-major matrix C, row r
// of the block held by lane r as four 16-byte units u[0..3], through a 2 KB
// shared-memory buffer `buf`: the units go in under a 64-byte XOR swizzle
// (unit q of row r at q ^ ((r >> 1) & 3), conflict-free) and come back four
// lanes per row, so each 16-byte global store writes eight whole 64-byte row
// segments instead of 32 scattered pieces, with an L2 evict-first hint.  The
// block starts at (row0, col0); rows >= row_end and columns >= n are left
// alone.  kEsz: element size (2 or 4); kAccum (FP32 only): C += values, one
// FP32 addition per element.
template <int kEsz, bool kAccum>
__device__ __forceinline__ void warp_store_block64(uint32_t buf, const uint4 (&u)[4], void *c,
                                                   int64_t ldc, int row0, int row_end, int col0,
                                                   int n, int lane) {
  static_assert(!kAccum || kEsz == 4, "C += is FP32 only");
  constexpr int kUnitCols = 16 / kEsz;
  __syncwarp();  // the buffer's previous block has been read back
  const uint32_t swz = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) st_shared_v4(buf + lane * 64 + 16 * (q ^ swz), u[q]);
  __syncwarp();
  const int unit = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i;
    uint4 v = ld_shared_v4(buf + r * 64 + 16 * (unit ^ ((r >> 1) & 3)));
    const int row = row0 + r, col = col0 + unit * kUnitCols;
    if (row >= row_end || col >= n) continue;
    uint8_t *dst = static_cast<uint8_t *>(c) + (static_cast<int64_t>(row) * ldc + col) * kEsz;
    if (col + kUnitCols <= n) {
      if (kAccum) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        v.x = __float_as_uint(__fadd_rn(old.x, __uint_as_float(v.x)));
        v.y = __float_as_uint(__fadd_rn(old.y, __uint_as_float(v.y)));
        v.z = __float_as_uint(__fadd_rn(old.z, __uint_as_float(v.z)));
        v.w = __float_as_uint(__fadd_rn(old.w, __uint_as_float(v.w)));
      }
      st_global_v4_hint(dst, v, l2_evict_first_policy());
    } else {
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      for (int e = 0; e < kUnitCols && col + e < n; ++e) {
        if (kEsz == 4) {
          float *d = reinterpret_cast<float *>(dst) + e;
          *d = kAccum ? __fadd_rn(*d, __uint_as_float(w[e])) : __uint_as_float(w[e]);
        } else {
          reinterpret_cast<uint16_t *>(dst)[e] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
        }
      }
    }
  }
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, issued by one thread.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (count 1) on an mbarrier once all tcgen05 operations issued so far by
// this thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for this thread's outstanding tcgen05.ld, with the given registers
// passed through the wait: the loaded values are only defined after it, and
// tying them to the instruction keeps their uses from being scheduled above it.
__device__ __forceinline__ void tmem_wait_ld_tied(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
// Ties more registers to the wait just issued (an empty volatile statement
// that the compiler keeps in order after it).
__device__ __forceinline__ void reg_tie(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 16 TMEM lanes x 8 columns per repetition, four repetitions (32 columns):
// thread t receives, for repetition k, r[4k], r[4k+1] = lane t/4, columns
// 8k + 2(t%4) and 8k + 2(t%4) + 1, and r[4k+2], r[4k+3] = the same columns of
// lane t/4 + 8 (lanes counted from the address's lane field).
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand tile
// laid out by TMA with 128-byte swizzling: rows of 128 bytes, 8-row atoms of
// 1024 bytes stacked along M/N (stride byte offset 1024).  The leading byte
// offset is unused for this layout (the MMA's K extent, 32 bytes, stays
// inside one 128-byte row) and is set to 1.  Bits 46-48 hold the fixed value
// 0b001; bits 61-63 the swizzle mode (2 = 128-byte).  The tile base must be
// 1024-byte aligned; the start address may then be advanced in 32-byte steps
// along K within the row.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                      // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                      // fixed 0b001
  d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f8f6f4: D FP32, A and B E4M3, both K-major,
// shape M x N (M = 128 here; N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format: F32
         | (0u << 7)                                 // A format: E4M3
         | (0u << 10)                                // B format: E4M3
         | (0u << 15) | (0u << 16)                   // A, B K-major
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ---------------------------------------------------------------- packed FP32 pairs
// sm_100+ executes two FP32 FMAs / multiplies per instruction on register
// pairs (fma.rn.f32x2, mul.rn.f32x2); each lane is an ordinary IEEE FP32
// operation rounded to nearest.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t pack_u32x2(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// acc = a * b + acc, per lane
__device__ __forceinline__ void ffma2(uint64_t &acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ---------------------------------------------------------------- E4M3
// Two FP32 -> two E4M3 bytes (round to nearest-even, saturate to +-448):
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  return pack_e4m3x2(a, b) | (pack_e4m3x2(c, d) << 16);
}

// ---------------------------------------------------------------- scales
// Scale of one group from its max-abs value (FP32 mode: s = a/448, inv =
// 448/a, IEEE divisions; POW2 mode: s = 2^e with the smallest e such that
// 448 * 2^e >= a), where a = max(amax, 2^-116).
__device__ __forceinline__ void group_scale(float amax, bool pow2, float &s, float &inv) {
  const float a = fmaxf(amax, 0x1p-116f);
  if (!pow2) {
    s = __fdiv_rn(a, 448.0f);
    inv = __fdiv_rn(448.0f, a);
    return;
  }
  // a = 1.m * 2^E; 448 = 1.75 * 2^8.  For 1.m <= 1.75, e = E - 8; else E - 7.
  // e is clamped to 127 (an infinite max-abs, reachable only when a value
  // overflowed FP32 before quantisation, also gives 127); the floor on a
  // keeps e >= -124, so s is always a normal FP32.  inv = 2^-e is normal for
  // e <= 126 and the subnormal 2^-127 for e = 127.
  const uint32_t bits = __float_as_uint(a);
  const int E = static_cast<int>((bits >> 23) & 0xFF) - 127;
  const uint32_t mant = bits & 0x7FFFFF;
  int e = E - 8 + (mant > 0x600000u ? 1 : 0);
  if (E > 127) e = 127;
  e = max(-126, min(127, e));
  s = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  inv = e <= 126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23)
                 : __uint_as_float(0x00400000u);
}

// Two E4M3 codes (low byte first) -> two FP16 values (exact: every E4M3 value
// is an FP16 value), packed low half first.
__device__ __forceinline__ uint32_t decode_e4m3x2(uint16_t codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes),
                                                   __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFF)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max of |lo|, |hi| of a packed BF16 pair, as FP32 (exact).
__device__ __forceinline__ float absmax_bf16x2(uint32_t w) {
  return fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w)));
}

}  // namespace fp8q

namespace fp8q {

// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs running tcgen05 with .cta_group::2: one MMA (M=256)
// uses both CTAs' shared memory and writes both CTAs' tensor memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// All threads of all CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (may be the peer's).
// Default (CTA-scope release) semantics: the only thing the arrive publishes is
// that this CTA's tcgen05.ld of an accumulator has completed, which the
// tcgen05.fence::before_thread_sync ahead of it already orders.  A
// cluster-scope release here costs a full memory barrier on every K-group.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMEM allocation for a CTA pair (issued by one warp in each CTA of the pair).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs]^T,
// M = 256 (128 rows per CTA), issued by one thread of the pair.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (count 1) on the mbarrier at the same offset in every CTA of
// `cta_mask` once all tcgen05 operations issued so far by this thread are done.
__device__ __forceinline__ void mma_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is
// signalled on an mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const void *tmap,
                                                 uint32_t bar_cluster_addr, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar_cluster_addr)
      : "memory");
}

}  // namespace fp8q

namespace fp8q {

// ---------------------------------------------------------------- block-scaled MMA
// tcgen05.mma ... kind::mxf8f6f4.block_scale.scale_vec::1X: each 32-wide K
// block of a row of A and of a row of B carries an unsigned 8-bit power-of-two
// exponent (UE8M0, bias 127, 255 = NaN) held in tensor memory.  Layout in TMEM
// (established by a probe with single-instruction, exactly representable
// results): the scale of row r of A (r < 128, per CTA) is at lane r, column
// sfa + r/32; the scale of row n of B (n < 256) is at column sfb + n/32 of
// lane 32*(r/32) + n%32 for the D rows r it multiplies, i.e. replicated in
// each 32-lane quarter.  The byte within the 32-bit cell is selected by the
// instruction descriptor's scale-factor ids, so one cell can carry four
// consecutive K blocks' exponents.  The same layout holds in each CTA of a
// pair (each CTA holds its own rows' A scales and all of the tile's B scales).

// Instruction descriptor for kind::mxf8f6f4 with UE8M0 scales: A, B E4M3
// K-major, D FP32 (implied), shape M x N; a_id / b_id pick the scale byte.
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int M, int N, uint32_t a_id, uint32_t b_id) {
  return (b_id << 4)                                 // B scale-factor byte
         | (0u << 7) | (0u << 10)                    // A, B: E4M3
         | (0u << 15) | (0u << 16)                   // A, B K-major
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (1u << 23)                                // scale type UE8M0
         | (static_cast<uint32_t>(M >> 4) << 24)     // M / 16
         | (a_id << 29);                             // A scale-factor byte
}

// D[tmem of both CTAs] (+)= (A . 2^sfa) * (B . 2^sfb)^T, M = 256 across the pair.
__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Register -> TMEM stores: thread i of the warp writes lane (base lane + i),
// 1 or 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st_32x32b_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace fp8q
