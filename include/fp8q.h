/*
 * fp8q.h -- C ABI of libfp8q: fine-grained FP8 (E4M3) quantisation and the
 * per-group-scaled FP8 GEMM on one sm_103a GPU.
 *
 * The operations follow the FP8 training recipe of DeepSeek-V3 as described
 * on these pages:
 *   - dssusan.co.kr board post 91437 (an excerpt of the DeepSeek-V3 report's
 *     FP8 section): paragraph 1 (power-of-two scaling factors for some
 *     activations), paragraph 2 (max-abs computed online per 1x128 activation
 *     tile and per 128x128 weight block; the scaling factor follows from it),
 *     paragraph 3 (Figure 6: per-group scaling factors along the GEMM's inner
 *     dimension K, applied as dequantisation, FP32 accumulation), paragraph 4
 *     (Figure 7 (a): 1x128 per token per 128 channels, 128x128 per 128 input
 *     by 128 output channels; 1x128 tiles become 128x1 tiles in the backward
 *     pass);
 *   - "Deepseek - Not For everyone" (xn--jj0bz6z98ct0a29q.com post 278251),
 *     paragraph 4: the max-abs is mapped onto the largest finite FP8 value;
 *   - youlimart.com FAQ post 597629, paragraph 2 (Figure 6): Fprop, Dgrad and
 *     Wgrad all run in FP8, taking FP8 inputs and producing BF16 or FP32;
 *   - "FP8 mixed precision -- где и как DeepSeek снизили точность
 *     вычислений?" (Data Science by ODS.ai): E4M3 for every tensor, FP32
 *     accumulation of the tensor-core partial sums.
 *
 * Conventions for every call:
 *   - Tensors are row-major; every leading dimension (ld*) is in ELEMENTS of
 *     that tensor's type.  E4M3 tensors are raw bytes (1 byte per element),
 *     BF16 tensors raw 16-bit patterns.
 *   - All pointers are DEVICE pointers owned by the caller; the library never
 *     allocates or frees device memory, and keeps none of the caller's
 *     pointers after a call returns (the only device address it keeps is that
 *     of its own static scratch array, see fp8q_quant_tensor_noalloc).  Calls
 *     are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).
 *   - E4M3 means the OCP "E4M3FN" encoding (bias 7, largest finite 448, NaN
 *     0x7F/0xFF, no infinity).  Values are rounded to nearest-even and
 *     saturated to +-448.
 *   - Scales s are FP32 with dequantised value = decode(q) * s.  For a group
 *     with max-abs value amax, a = max(amax, 2^-116) and
 *       FP8Q_SCALE_FP32: s = a / 448, codes E4M3(x * (448 / a)), both FP32
 *                        divisions rounded to nearest;
 *       FP8Q_SCALE_POW2: s = 2^e, e the smallest integer with 448 * 2^e >= a,
 *                        codes E4M3(x * 2^-e).
 *     Inputs must be finite; NaN/Inf inputs give unspecified codes.
 *   - Argument errors are returned synchronously and nothing is launched.
 *     A device-side failure (a bounded wait that gave up) is recorded in a
 *     device status word and returned by fp8q_sync_status().
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8q_status {
  FP8Q_OK = 0,
  FP8Q_ERR_INVALID = 1,     /* null pointer where one is required, unknown enum */
  FP8Q_ERR_SHAPE = 2,       /* negative size, K/T not a multiple of 128, ld too small */
  FP8Q_ERR_ALIGN = 3,       /* pointer or leading dimension breaks a 16-byte rule */
  FP8Q_ERR_UNSUPPORTED = 4, /* current device is not sm_103, or too little shared memory */
  FP8Q_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  FP8Q_ERR_TIMEOUT = 6      /* a device-side wait gave up (reported by fp8q_sync_status) */
} fp8q_status;

enum { FP8Q_SCALE_FP32 = 0, FP8Q_SCALE_POW2 = 1 };
enum { FP8Q_OUT_BF16 = 0, FP8Q_OUT_FP32 = 1 };
/* Layout of the B-operand scales of fp8q_gemm. */
enum {
  FP8Q_BSCALE_BLOCK = 0,   /* one per 128x128 block:  sb[(n/128) * ld_sb + k/128] */
  FP8Q_BSCALE_BLOCK_T = 1, /* one per 128x128 block, grid transposed:
                              sb[(k/128) * ld_sb + n/128] (Dgrad reading a weight's grid) */
  FP8Q_BSCALE_ROW = 2      /* one per row n per 128-K group (128x1 tiles, Wgrad):
                              sb[(k/128) * ld_sb + n] */
};

/*
 * Activation quantisation, 1x128 tiles: one scale per row (token) m per 128
 * columns (channels) ([dssusan] paragraph 2 and paragraph 4, Figure 7 (a)(1)).
 *   x   BF16 [M][ldx], reads columns [0, K).       K % 128 == 0, M >= 0.
 *   q   E4M3 [M][ldq], writes columns [0, K).
 *   sa  FP32, MN-major: scale of (m, group g) at sa[g * ld_sa + m], ld_sa >= M.
 * Alignment: x and q 16-byte aligned, ldx % 8 == 0, ldq % 16 == 0.
 */
fp8q_status fp8q_quant_act(const void *x, int64_t M, int64_t K, int64_t ldx,
                           void *q, int64_t ldq, float *sa, int64_t ld_sa,
                           int scale_mode, void *stream);

/*
 * Activation quantisation for the backward pass, 128x1 tiles: one scale per
 * column (channel) c per 128 rows (tokens) ([dssusan] paragraph 4: 1x128
 * tiles become 128x1 tiles).  The codes are written TRANSPOSED so the token
 * dimension is contiguous, i.e. K-major for the Wgrad GEMM.
 *   x      BF16 [T][ldx], columns [0, C).           T % 128 == 0, C % 8 == 0,
 *          T <= 65535 * 128, C <= 2^31 - 128 (else FP8Q_ERR_SHAPE).
 *   qT     E4M3 [C][ldqT], qT[c][t] = code of x[t][c].
 *   sT     FP32, scale of (t-group tg, c) at sT[tg * ld_sT + c], ld_sT >= C.
 *   q_rows optional (NULL to skip): the 1x128 quantisation of the same x,
 *          computed from the same read: E4M3 [T][ldq_rows] and
 *          s_rows[g * ld_s_rows + t] exactly as fp8q_quant_act would write
 *          them.  Requires C % 128 == 0; s_rows must then be non-NULL.
 * Alignment: x, qT (and q_rows) 16-byte aligned; ldx % 8, ldqT % 16,
 * ldq_rows % 16 == 0.
 */
fp8q_status fp8q_quant_act_T(const void *x, int64_t T, int64_t C, int64_t ldx,
                             void *qT, int64_t ldqT, float *sT, int64_t ld_sT,
                             void *q_rows, int64_t ldq_rows, float *s_rows,
                             int64_t ld_s_rows, int scale_mode, void *stream);

/*
 * 128x1 requantisation of FP8-cached activations: the forward pass keeps its
 * activations as 1x128-quantised E4M3 ([dssusan] paragraph 2: cached
 * activations are stored in low precision), and the backward pass needs the
 * same tensor in 128x1 tiles ([dssusan] paragraph 4).  Each cached value is
 * dequantised with one FP32 multiply, x = fl32(decode(q[t][c]) * s_rows(t, c)),
 * then quantised exactly as fp8q_quant_act_T quantises x.
 *   q       E4M3 [T][ldq], columns [0, C).          T % 128 == 0, C % 128 == 0,
 *           T <= 65535 * 128, C <= 2^31 - 1 (else FP8Q_ERR_SHAPE).
 *   s_rows  FP32 1x128 scales of q: s_rows[(c/128) * ld_s_rows + t], ld_s_rows >= T.
 *   qT      E4M3 [C][ldqT], qT[c][t];  sT FP32 sT[(t/128) * ld_sT + c].
 * Alignment: q, qT 16-byte aligned; ldq % 16 == 0, ldqT % 16 == 0.
 */
fp8q_status fp8q_requant_act_T(const void *q, int64_t T, int64_t C, int64_t ldq,
                               const float *s_rows, int64_t ld_s_rows, void *qT, int64_t ldqT,
                               float *sT, int64_t ld_sT, int scale_mode, void *stream);

/*
 * Weight quantisation, 128x128 blocks: one scale per 128 rows (output
 * channels) x 128 columns (input channels) ([dssusan] paragraph 4, Figure
 * 7 (a)(2)).  A last partial block of rows covers only the rows that exist.
 *   w   BF16 [N][ldw], columns [0, K).              K % 128 == 0, N >= 0.
 *   q   E4M3 [N][ldq].
 *   qT  optional (NULL to skip): E4M3 [K][ldqT], qT[k][n] = q[n][k] -- the
 *       K-major B operand of the Dgrad GEMM (dX = dY * W).
 *   sb  FP32 [ceil(N/128)][ld_sb], block (nb, kb) at sb[nb * ld_sb + kb],
 *       ld_sb >= K/128.
 * Alignment: w, q, qT 16-byte aligned; ldw % 8, ldq % 16, ldqT % 16 == 0.
 */
fp8q_status fp8q_quant_weight(const void *w, int64_t N, int64_t K, int64_t ldw,
                              void *q, int64_t ldq, void *qT, int64_t ldqT,
                              float *sb, int64_t ld_sb, int scale_mode,
                              void *stream);

/*
 * Per-tensor quantisation, for comparison with the fine-grained quantisers:
 * one scale for the whole tensor from its max-abs value, by the same rule as
 * a group's.  This is the standard practice the pages contrast with the
 * method ("Deepseek - Not For everyone", paragraph 4: mapping the tensor's
 * max-abs onto the FP8 maximum makes the result sensitive to outliers).
 * Two passes: per-64-row partial max-abs values go to `workspace`, then every
 * slab reduces them and quantises.
 *   x  BF16 [M][ldx], columns [0, K), K % 8 == 0;  q E4M3 [M][ldq];
 *   s  one FP32 (device) -- the tensor's scale.
 *   workspace  device scratch of at least fp8q_quant_tensor_workspace_bytes(M, K)
 *              bytes, 4-byte aligned, owned by the caller; its contents on entry
 *              do not matter.
 * Alignment: x, q 16-byte aligned; ldx % 8, ldq % 8 == 0.
 */
int64_t fp8q_quant_tensor_workspace_bytes(int64_t M, int64_t K);
fp8q_status fp8q_quant_tensor(const void *x, int64_t M, int64_t K, int64_t ldx,
                              void *q, int64_t ldq, float *s, void *workspace,
                              int64_t workspace_bytes, int scale_mode, void *stream);

/*
 * fp8q_quant_tensor with no workspace argument and no allocation.  The
 * sources describe no such call: it is a library convenience for callers that
 * cannot allocate device memory when they quantise (code inside an
 * allocator's or pool's callbacks, or a runtime whose device memory is all
 * handed to its own pools).  The scratch is a fixed 4 KB array in the
 * library's static device memory, one per device, so:
 *   - M <= 65536 (1024 partials of 64 rows); larger M returns FP8Q_ERR_SHAPE
 *     and launches nothing.  Every other argument, result and error is as for
 *     fp8q_quant_tensor.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that call before any stream capture.  The
 *     address is remembered with the id of the CUDA context it belongs to and
 *     looked up again when another context is current, e.g. after
 *     cudaDeviceReset or after the primary context was released and created
 *     again (the first call after that is again a set-up call).
 *   - Every call on a device uses the same array.  Calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     and may return wrong scales; calls ordered on one stream do not.
 * The call makes no cudaMalloc or cudaFree and allocates no other memory.
 */
fp8q_status fp8q_quant_tensor_noalloc(const void *x, int64_t M, int64_t K, int64_t ldx,
                                      void *q, int64_t ldq, float *s, int scale_mode,
                                      void *stream);

/*
 * FP8 GEMM with per-group scaling along K ([dssusan] paragraph 3, Figure 6;
 * [youlimart] paragraph 2):
 *   C[m][n] = sum over 128-wide groups kb of
 *             sa(m,kb) * sb(n,kb) * sum_{k in kb} decode(a[m][k]) * decode(b[n][k])
 * The inner sums run on the tensor cores into an FP32 partial per group; each
 * partial is scaled and added into an FP32 accumulator by separate warps.
 * The result is stored as FP32, or rounded to nearest-even BF16.
 *   a   E4M3 [M][lda] (K-major), sa FP32 at sa[kb * ld_sa + m], ld_sa >= M.
 *   b   E4M3 [N][ldb] (K-major), sb FP32 laid out per bscale_kind (see enum).
 *   c   [M][ldc] BF16 or FP32 per out_dtype.
 *   K % 128 == 0; M, N >= 0 (tails are masked).  K == 0 writes zeros.
 * Alignment: a, b, c 16-byte aligned; lda % 16 == 0, ldb % 16 == 0,
 * ldc * sizeof(out) % 16 == 0.
 * Fprop: a = quantised activations, b = quantised weight, BLOCK scales.
 * Dgrad: a = quantised dY, b = the weight's qT, BLOCK_T over the weight's sb.
 * Wgrad: a = dY's qT, b = X's qT, sa = dY's sT, sb = X's sT with ROW scales.
 */
fp8q_status fp8q_gemm(const void *a, int64_t lda, const float *sa,
                      int64_t ld_sa, const void *b, int64_t ldb,
                      const float *sb, int64_t ld_sb, int bscale_kind, void *c,
                      int64_t ldc, int out_dtype, int64_t M, int64_t N,
                      int64_t K, void *stream);

/*
 * Gradient accumulation form of fp8q_gemm: C += the same product, C FP32.
 * Weight gradients are kept in FP32 and summed over micro-batches
 * ([dssusan] paragraph 2: weight gradients stay in FP32); each element
 * receives one FP32 addition, fl32(C_old + result).  Arguments and rules as
 * fp8q_gemm with out_dtype = FP8Q_OUT_FP32.
 */
fp8q_status fp8q_gemm_accumulate(const void *a, int64_t lda, const float *sa,
                                 int64_t ld_sa, const void *b, int64_t ldb,
                                 const float *sb, int64_t ld_sb, int bscale_kind,
                                 float *c, int64_t ldc, int64_t M, int64_t N,
                                 int64_t K, void *stream);

/*
 * fp8q_gemm for power-of-two scales, on the tensor cores' block-scaled MMA.
 * The method allows scaling factors that are integral powers of two
 * ([dssusan] paragraph 1) and recommends tensor cores that take the group
 * scales themselves ([dssusan] paragraph 3); Blackwell's microscaling MMA
 * ("Deepseek - Not For everyone", paragraph 3) multiplies each 32-wide K
 * block of A and B by a power of two inside the MMA.  This call computes the
 * same product as fp8q_gemm, with the K-group scales applied by the MMA and
 * the sum over all K-groups accumulated in FP32 by the tensor cores (no
 * per-group FP32 fold by the CUDA cores).
 *   Arguments, layouts, alignment and return codes: as fp8q_gemm.
 *   Precondition: every scale the product reads (sa of rows < M, sb of
 *   columns < N, K-groups < K/128) is a power of two 2^e, -127 <= e <= 127 --
 *   what the quantisers produce with FP8Q_SCALE_POW2.  Any other value is
 *   used by its binary exponent alone, and the kernel records
 *   FP8Q_ERR_INVALID in a device status word that fp8q_sync_status reports.
 *   K == 0 writes zeros (fp8q_gemm_pow2) or leaves C unchanged (_accumulate).
 * Tiles are 256 x 256 (a pair of CTAs per tile).
 */
fp8q_status fp8q_gemm_pow2(const void *a, int64_t lda, const float *sa,
                           int64_t ld_sa, const void *b, int64_t ldb,
                           const float *sb, int64_t ld_sb, int bscale_kind,
                           void *c, int64_t ldc, int out_dtype, int64_t M,
                           int64_t N, int64_t K, void *stream);

/* C (FP32) += the fp8q_gemm_pow2 product; as fp8q_gemm_accumulate otherwise. */
fp8q_status fp8q_gemm_pow2_accumulate(const void *a, int64_t lda, const float *sa,
                                      int64_t ld_sa, const void *b, int64_t ldb,
                                      const float *sb, int64_t ld_sb, int bscale_kind,
                                      float *c, int64_t ldc, int64_t M, int64_t N,
                                      int64_t K, void *stream);

/*
 * Grouped FP8 GEMM for MoE experts: rows [offs[g], offs[g+1]) of A (tokens
 * sorted by expert, top-1 routing) are multiplied by expert g's weight.
 *   a     E4M3 [M][lda], sa at sa[kb * ld_sa + m] as in fp8q_gemm.
 *   b     E4M3 [G][N][ldb] (expert g's rows start at b + g*N*ldb).
 *   sb    FP32 [G][ceil(N/128)][K/128] (BLOCK layout per expert).
 *   offs  int32 DEVICE array [G+1]: 0 <= offs[0] <= ... <= offs[G] <= M.
 *         Empty experts are allowed.  Rows outside [offs[0], offs[G]) are
 *         not written.  Offsets that break the ordering are clamped into
 *         [0, M] and a decreasing step is treated as an empty expert.
 *   c     [M][ldc] BF16 or FP32.
 *   1 <= G <= 1024; other rules as fp8q_gemm.
 */
fp8q_status fp8q_grouped_gemm(const void *a, int64_t lda, const float *sa,
                              int64_t ld_sa, const void *b, int64_t ldb,
                              const float *sb, const int32_t *offs, int G,
                              void *c, int64_t ldc, int out_dtype, int64_t M,
                              int64_t N, int64_t K, void *stream);

/*
 * fp8q_grouped_gemm for power-of-two scales, on the block-scaled MMA (see
 * fp8q_gemm_pow2): the same arguments, layouts and results, with the same
 * precondition on the scales.  Tiles are 256 rows x 256 columns (a CTA pair);
 * K must be a positive multiple of 128 (K == 0 returns FP8Q_ERR_SHAPE).
 */
fp8q_status fp8q_grouped_gemm_pow2(const void *a, int64_t lda, const float *sa,
                                   int64_t ld_sa, const void *b, int64_t ldb,
                                   const float *sb, const int32_t *offs, int G,
                                   void *c, int64_t ldc, int out_dtype, int64_t M,
                                   int64_t N, int64_t K, void *stream);

/*
 * Plain FP32 -> E4M3 conversion of n values (round to nearest-even, saturate
 * to +-448, NaN -> 0x7F), with no scaling.  The quantisers use the same
 * conversion; this entry exposes it so it can be checked on every FP32 bit
 * pattern.  x: FP32 [n], q: E4M3 [n]; both 16-byte aligned.
 */
fp8q_status fp8q_cast_e4m3(const float *x, int64_t n, void *q, void *stream);

/*
 * Synchronise `stream`, then read and clear this device's status word.
 * Returns FP8Q_ERR_TIMEOUT if a kernel's bounded wait gave up since the last
 * call, FP8Q_ERR_CUDA if synchronisation failed, else FP8Q_OK.
 */
fp8q_status fp8q_sync_status(void *stream);

/*
 * Set the time limit, in nanoseconds, of every device-side wait launched
 * afterwards from this process (default 2e9 = 2 s; 0 restores the default).
 */
void fp8q_set_wait_timeout_ns(uint64_t ns);

/*
 * Diagnostic: launch one CTA that waits, with the bounded wait the GEMM uses,
 * on a barrier that nothing ever completes, for at most timeout_ns.  The wait
 * must give up, record FP8Q_ERR_TIMEOUT in the status word and return; the
 * caller then reads it with fp8q_sync_status().
 */
fp8q_status fp8q_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* Human-readable name of a status code (static storage). */
const char *fp8q_status_string(fp8q_status s);

/* ABI version of this header (major * 100 + minor). */
int fp8q_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
