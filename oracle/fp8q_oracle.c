/*
 * fp8q_oracle.c -- CPU oracle for fine-grained FP8 quantisation and the
 * per-group-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library: everything here is written
 * out from the definitions below, plainly and slowly, so that a reader can
 * check it against the source pages by eye.
 *
 * Sources (web pages on DeepSeek-V3's FP8 training recipe):
 *   [dssusan]  dssusan.co.kr board post 91437 (spun excerpt of the DeepSeek-V3
 *              report's FP8 section): paragraph 2 (online max-abs per 1x128
 *              activation tile / 128x128 weight block, then the scaling
 *              factor); paragraph 3 (Figure 6: per-group scaling along the
 *              inner dimension K, multiplied in as dequantisation, FP32
 *              accumulation); paragraph 4 (Figure 7 (a): 1x128 per token per
 *              128 channels, 128x128 per 128 input x 128 output channels;
 *              1x128 tiles become 128x1 tiles in the backward pass);
 *              paragraph 1 (power-of-2 scaling factors).
 *   [notforeveryone] "Deepseek - Not For everyone" (xn--jj0bz6z98ct0a29q.com
 *              post 278251), paragraph 4: the max-abs value is mapped to the
 *              largest representable FP8 value.
 *   [ods]      "FP8 mixed precision -- где и как DeepSeek снизили точность
 *              вычислений?" (Data Science by ODS.ai): E4M3 for every tensor;
 *              1x128 tiles for activations, 128x128 blocks for weights;
 *              FP32 accumulation of the GEMM partial results.
 *   [youlimart] youlimart.com FAQ post 597629, paragraph 2 (Figure 6): the
 *              GEMMs take FP8 inputs and produce BF16 or FP32 outputs.
 *
 * Where the pages leave a step open, the plainest reading is taken; each such
 * reading is marked READING below.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        -pthread (no FMA contraction, IEEE single/double arithmetic).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------
 * Threads: a plain parallel-for over independent output items.  No blocking
 * or reordering of any sum: each item is computed exactly as the serial code
 * would compute it.
 * ------------------------------------------------------------------------ */
typedef void (*item_fn)(int64_t i, void *ctx);

typedef struct {
  item_fn fn;
  void *ctx;
  int64_t n;
  int t, nt;
} par_job;

static void *par_worker(void *arg) {
  par_job *j = (par_job *)arg;
  int64_t lo = j->n * j->t / j->nt, hi = j->n * (j->t + 1) / j->nt;
  for (int64_t i = lo; i < hi; ++i) j->fn(i, j->ctx);
  return NULL;
}

int oracle_num_threads(void) {
  const char *env = getenv("ORACLE_THREADS");
  if (env && atoi(env) > 0) return atoi(env);
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static void par_for(int64_t n, item_fn fn, void *ctx) {
  int nt = oracle_num_threads();
  if (nt > 256) nt = 256;
  if (n < nt) nt = (int)(n > 0 ? n : 1);
  if (nt == 1) {
    for (int64_t i = 0; i < n; ++i) fn(i, ctx);
    return;
  }
  pthread_t th[256];
  par_job jobs[256];
  for (int t = 0; t < nt; ++t) {
    jobs[t] = (par_job){fn, ctx, n, t, nt};
    if (pthread_create(&th[t], NULL, par_worker, &jobs[t]) != 0) {
      par_worker(&jobs[t]); /* run it here if a thread cannot be made */
      th[t] = 0;
    }
  }
  for (int t = 0; t < nt; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------
 * Number formats.
 * ------------------------------------------------------------------------ */

/* BF16 -> FP32 is exact: the 16 stored bits are the top half of the FP32. */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/*
 * E4M3 ("E4M3FN" in the OCP 8-bit floating point definition), the only FP8
 * format the method uses ([ods]: E4M3 for Fprop, Dgrad and Wgrad alike).
 * Bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa.
 * Exponent field 0: subnormal, value m * 2^-9.  Otherwise (1 + m/8) * 2^(e-7).
 * S.1111.111 is NaN; there is no infinity; the largest finite value is
 * S.1111.110 = 448.
 */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 0x7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return s ? -mag : mag;
}

/*
 * FP32 -> E4M3, rounding to nearest with ties to even, then saturating to the
 * largest finite magnitude (448) instead of overflowing to NaN.
 * READING: the pages name the format (E4M3) and the target of the scaling
 * (the largest finite FP8 value, [notforeveryone] paragraph 4) but not the
 * rounding; round-to-nearest-even with saturation is the format's standard
 * conversion.  NaN in gives the NaN code 0x7F.
 */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E; /* saturate: nothing lies above 448 */
  /* Spacing of the E4M3 grid: 2^-9 below 2^-5 (subnormals and the first
   * normal binade), 2^(E-3) in the binade [2^E, 2^(E+1)) for E >= -6. */
  int E = -6;
  if (a >= 0x1p-6) {
    int ex;
    (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
    E = ex - 1;
  }
  double quantum = ldexp(1.0, E - 3);
  double n = rint(a / quantum); /* exact scaling; rint: nearest, ties to even */
  double mag = n * quantum;
  if (mag > 448.0) mag = 448.0;
  if (mag < 0x1p-6) return sign | (uint8_t)(mag / 0x1p-9); /* code 0..7 */
  int ex;
  double f = frexp(mag, &ex);
  int Eo = ex - 1;                         /* mag = (2f) * 2^Eo, 2f in [1,2) */
  int mant = (int)((2.0 * f - 1.0) * 8.0); /* exact: 2f has <= 4 bits */
  return sign | (uint8_t)(((Eo + 7) << 3) | mant);
}

typedef struct {
  const float *x;
  uint8_t *q;
} enc_ctx;

static void enc_item(int64_t i, void *c) {
  enc_ctx *e = (enc_ctx *)c;
  for (int64_t j = i * 65536; j < (i + 1) * 65536; ++j)
    e->q[j] = oracle_e4m3_encode(e->x[j]);
}

/* Encode n floats; n must be a multiple of 65536 for the threaded part, the
 * remainder is encoded serially. */
void oracle_e4m3_encode_array(const float *x, int64_t n, uint8_t *q) {
  enc_ctx c = {x, q};
  int64_t chunks = n / 65536;
  par_for(chunks, enc_item, &c);
  for (int64_t j = chunks * 65536; j < n; ++j) q[j] = oracle_e4m3_encode(x[j]);
}

/* ------------------------------------------------------------------------
 * Scale of one group from its max-abs value ([dssusan] paragraph 2: the
 * max-abs is computed online for each 1x128 tile / 128x128 block and the
 * scaling factor follows from it; [notforeveryone] paragraph 4: the max-abs
 * is mapped onto the largest finite FP8 value, 448).
 *
 * READING (floor): a = max(amax, 2^-116) so that an all-zero group still has
 * a finite, normal scale and reciprocal; the floor only touches groups whose
 * max-abs is below ~1.2e-35.
 *
 * FP32 mode:  s = a / 448 and inv = 448 / a, each one IEEE single-precision
 *             division rounded to nearest; the stored scale is s and the
 *             codes are E4M3(fl32(x * inv)).
 * POW2 mode ([dssusan] paragraph 1: for some activations the scaling
 *             factors are whole powers of two):
 *             READING: e is the smallest integer with 448 * 2^e >= a (round
 *             the scale up, so no element exceeds 448); s = 2^e, inv = 2^-e.
 *             e is clamped to [-127, 127] (never reached for finite BF16).
 * ------------------------------------------------------------------------ */
void oracle_group_scale(float amax, int pow2, float *s, float *inv) {
  float a = amax > 0x1p-116f ? amax : 0x1p-116f;
  if (!pow2) {
    *s = a / 448.0f;
    *inv = 448.0f / a;
    return;
  }
  int e = -127;
  while (e < 127 && ldexp(448.0, e) < (double)a) ++e;
  *s = (float)ldexp(1.0, e);
  *inv = (float)ldexp(1.0, -e);
}

/* ------------------------------------------------------------------------
 * Activation quantisation, 1x128 tiles: one scale per token (row m) per 128
 * channels (group g) ([dssusan] paragraph 4, Figure 7 (a)(1)).
 * x: BF16 bits, [M][K] with row stride ldx.  K % 128 == 0.
 * q: E4M3 codes [M][K], row stride ldq.
 * sa: scales, stored MN-major: sa[g * ld_sa + m]  (one column of M scales per
 *     128-wide K group; layout choice of this library, not of the pages).
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *x;
  int64_t M, K, ldx, ldq, ld_sa;
  uint8_t *q;
  float *sa;
  int pow2;
} qa_ctx;

static void quant_act_row(int64_t m, void *c) {
  qa_ctx *p = (qa_ctx *)c;
  for (int64_t g = 0; g < p->K / 128; ++g) {
    const uint16_t *xg = p->x + m * p->ldx + g * 128;
    float amax = 0.0f;
    for (int j = 0; j < 128; ++j) {
      float v = fabsf(bf16_to_f32(xg[j]));
      if (v > amax) amax = v;
    }
    float s, inv;
    oracle_group_scale(amax, p->pow2, &s, &inv);
    p->sa[g * p->ld_sa + m] = s;
    for (int j = 0; j < 128; ++j) {
      float prod = bf16_to_f32(xg[j]) * inv;
      p->q[m * p->ldq + g * 128 + j] = oracle_e4m3_encode(prod);
    }
  }
}

void oracle_quant_act(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                      uint8_t *q, int64_t ldq, float *sa, int64_t ld_sa,
                      int pow2) {
  qa_ctx c = {x, M, K, ldx, ldq, ld_sa, q, sa, pow2};
  par_for(M, quant_act_row, &c);
}

/* ------------------------------------------------------------------------
 * Activation quantisation for the backward pass, 128x1 tiles: one scale per
 * channel c per 128 tokens ([dssusan] paragraph 4: the 1x128 tiles are
 * converted to 128x1 tiles in the backward pass).  The codes are written
 * transposed so that the token dimension T (the GEMM's K for Wgrad) is
 * contiguous.
 * x: BF16 [T][C], row stride ldx.  T % 128 == 0.
 * qT: E4M3 [C][T], row stride ldqT.   sT: sT[tg * ld_sT + c].
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *x;
  int64_t T, C, ldx, ldqT, ld_sT;
  uint8_t *qT;
  float *sT;
  int pow2;
} qt_ctx;

static void quant_act_T_channel(int64_t c, void *cx) {
  qt_ctx *p = (qt_ctx *)cx;
  for (int64_t tg = 0; tg < p->T / 128; ++tg) {
    float amax = 0.0f;
    for (int j = 0; j < 128; ++j) {
      float v = fabsf(bf16_to_f32(p->x[(tg * 128 + j) * p->ldx + c]));
      if (v > amax) amax = v;
    }
    float s, inv;
    oracle_group_scale(amax, p->pow2, &s, &inv);
    p->sT[tg * p->ld_sT + c] = s;
    for (int j = 0; j < 128; ++j) {
      int64_t t = tg * 128 + j;
      float prod = bf16_to_f32(p->x[t * p->ldx + c]) * inv;
      p->qT[c * p->ldqT + t] = oracle_e4m3_encode(prod);
    }
  }
}

void oracle_quant_act_T(const uint16_t *x, int64_t T, int64_t C, int64_t ldx,
                        uint8_t *qT, int64_t ldqT, float *sT, int64_t ld_sT,
                        int pow2) {
  qt_ctx c = {x, T, C, ldx, ldqT, ld_sT, qT, sT, pow2};
  par_for(C, quant_act_T_channel, &c);
}

/* ------------------------------------------------------------------------
 * Weight quantisation, 128x128 blocks: one scale per 128 output channels
 * (rows n) x 128 input channels (columns k) ([dssusan] paragraph 4, Figure
 * 7 (a)(2)).
 * w: BF16 [N][K], row stride ldw.  K % 128 == 0; READING: a last, partial
 * block of rows covers only the rows that exist.
 * q: E4M3 [N][K], row stride ldq.  sb[nb * (K/128) + kb], nb < ceil(N/128).
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *w;
  int64_t N, K, ldw, ldq;
  uint8_t *q;
  float *sb;
  int pow2;
} qw_ctx;

static void quant_weight_block(int64_t idx, void *cx) {
  qw_ctx *p = (qw_ctx *)cx;
  int64_t KB = p->K / 128;
  int64_t nb = idx / KB, kb = idx % KB;
  int64_t n0 = nb * 128, n1 = n0 + 128 < p->N ? n0 + 128 : p->N;
  float amax = 0.0f;
  for (int64_t n = n0; n < n1; ++n)
    for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
      float v = fabsf(bf16_to_f32(p->w[n * p->ldw + k]));
      if (v > amax) amax = v;
    }
  float s, inv;
  oracle_group_scale(amax, p->pow2, &s, &inv);
  p->sb[nb * KB + kb] = s;
  for (int64_t n = n0; n < n1; ++n)
    for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
      float prod = bf16_to_f32(p->w[n * p->ldw + k]) * inv;
      p->q[n * p->ldq + k] = oracle_e4m3_encode(prod);
    }
}

void oracle_quant_weight(const uint16_t *w, int64_t N, int64_t K, int64_t ldw,
                         uint8_t *q, int64_t ldq, float *sb, int pow2) {
  qw_ctx c = {w, N, K, ldw, ldq, q, sb, pow2};
  par_for(((N + 127) / 128) * (K / 128), quant_weight_block, &c);
}

/* ------------------------------------------------------------------------
 * The FP8 GEMM with per-group scaling along K ([dssusan] paragraph 3, Figure
 * 6: the per-group scaling factors along the inner dimension K are
 * multiplied in as the dequantisation step and the sum is kept in full FP32
 * precision; [youlimart] paragraph 2: BF16 or FP32 outputs).
 *
 * The method reaches, up to rounding order, the plain product of the
 * dequantised operands, so the oracle is that definition evaluated in double:
 *     C[m][n] = sum_k  a[m][k] * b[n][k],
 *     a[m][k] = decode(qa[m][k]) * sa(m, k/128),
 *     b[n][k] = decode(qb[n][k]) * sb(n, k/128).
 * It also returns absdot[m][n] = sum_k |a[m][k] * b[n][k]|, the scale of the
 * tolerance bound.
 *
 * A scale: sa[(k/128) * ld_sa + m].
 * B scale, by kind:
 *   0  one per 128x128 block        sb[(n/128) * ld_sb + k/128]
 *   1  one per 128x128 block, grid stored transposed
 *                                   sb[(k/128) * ld_sb + n/128]
 *   2  one per row n per 128-K group (128x1 tiles, Wgrad)
 *                                   sb[(k/128) * ld_sb + n]
 * Computed for the rows listed in `rows` (all N columns each); out rows are
 * packed: c[i * N + n] for rows[i].
 * ------------------------------------------------------------------------ */
static double b_scale(const float *sb, int kind, int64_t ld_sb, int64_t n,
                      int64_t kb) {
  if (kind == 0) return sb[(n / 128) * ld_sb + kb];
  if (kind == 1) return sb[kb * ld_sb + n / 128];
  return sb[kb * ld_sb + n];
}

typedef struct {
  const uint8_t *qa;
  int64_t lda;
  const float *sa;
  int64_t ld_sa;
  const uint8_t *qb;
  int64_t ldb;
  const float *sb;
  int bkind;
  int64_t ld_sb, N, K;
  const int64_t *rows;
  double *c, *absdot;
  double lut[256];
} gemm_ctx;

static void gemm_item(int64_t idx, void *cx) {
  gemm_ctx *p = (gemm_ctx *)cx;
  int64_t i = idx / p->N, n = idx % p->N;
  int64_t m = p->rows[i];
  double acc = 0.0, mag = 0.0;
  for (int64_t k = 0; k < p->K; ++k) {
    double a = p->lut[p->qa[m * p->lda + k]] * (double)p->sa[(k / 128) * p->ld_sa + m];
    double b = p->lut[p->qb[n * p->ldb + k]] * b_scale(p->sb, p->bkind, p->ld_sb, n, k / 128);
    acc += a * b;
    mag += fabs(a * b);
  }
  p->c[i * p->N + n] = acc;
  if (p->absdot) p->absdot[i * p->N + n] = mag;
}

void oracle_gemm_rows(const uint8_t *qa, int64_t lda, const float *sa,
                      int64_t ld_sa, const uint8_t *qb, int64_t ldb,
                      const float *sb, int bkind, int64_t ld_sb, int64_t N,
                      int64_t K, const int64_t *rows, int64_t nrows, double *c,
                      double *absdot) {
  gemm_ctx *p = (gemm_ctx *)malloc(sizeof(gemm_ctx));
  if (!p) return;
  *p = (gemm_ctx){qa, lda, sa, ld_sa, qb, ldb, sb, bkind, ld_sb, N, K, rows, c, absdot, {0}};
  for (int v = 0; v < 256; ++v) p->lut[v] = oracle_e4m3_decode((uint8_t)v);
  par_for(nrows * N, gemm_item, p);
  free(p);
}

/* ------------------------------------------------------------------------
 * Grouped GEMM for MoE experts: the GEMM above, applied per expert g to the
 * rows [offs[g], offs[g+1]) of A (tokens sorted by expert) with that expert's
 * weight qb[g] ([N][K]) and block scales sb[g] ([ceil(N/128)][K/128]).
 * READING: top-1 routing, so each row belongs to exactly one expert; empty
 * experts are legal.  A row outside [offs[0], offs[G]) gives zeros.
 * ------------------------------------------------------------------------ */
typedef struct {
  gemm_ctx base;
  const int32_t *offs;
  int G;
} ggemm_ctx;

static void ggemm_item(int64_t idx, void *cx) {
  ggemm_ctx *gp = (ggemm_ctx *)cx;
  const gemm_ctx *p = &gp->base;
  int64_t i = idx / p->N, n = idx % p->N;
  int64_t m = p->rows[i];
  int g = -1;
  for (int e = 0; e < gp->G; ++e)
    if (m >= gp->offs[e] && m < gp->offs[e + 1]) g = e;
  if (g < 0) {
    p->c[i * p->N + n] = 0.0;
    if (p->absdot) p->absdot[i * p->N + n] = 0.0;
    return;
  }
  int64_t NB = (p->N + 127) / 128, KB = p->K / 128;
  double acc = 0.0, mag = 0.0;
  const uint8_t *qb = p->qb + (int64_t)g * p->N * p->K;
  const float *sb = p->sb + (int64_t)g * NB * KB;
  for (int64_t k = 0; k < p->K; ++k) {
    double a = p->lut[p->qa[m * p->lda + k]] * (double)p->sa[(k / 128) * p->ld_sa + m];
    double b = p->lut[qb[n * p->K + k]] * (double)sb[(n / 128) * KB + k / 128];
    acc += a * b;
    mag += fabs(a * b);
  }
  p->c[i * p->N + n] = acc;
  if (p->absdot) p->absdot[i * p->N + n] = mag;
}

void oracle_grouped_gemm_rows(const uint8_t *qa, int64_t lda, const float *sa,
                              int64_t ld_sa, const uint8_t *qb,
                              const float *sb, const int32_t *offs, int G,
                              int64_t N, int64_t K, const int64_t *rows,
                              int64_t nrows, double *c, double *absdot) {
  ggemm_ctx *gp = (ggemm_ctx *)malloc(sizeof(ggemm_ctx));
  if (!gp) return;
  gp->base = (gemm_ctx){qa, lda, sa, ld_sa, qb, K, sb, 0, 0, N, K, rows, c, absdot, {0}};
  for (int v = 0; v < 256; ++v) gp->base.lut[v] = oracle_e4m3_decode((uint8_t)v);
  gp->offs = offs;
  gp->G = G;
  par_for(nrows * N, ggemm_item, gp);
  free(gp);
}

/* ------------------------------------------------------------------------
 * Context only: the unquantised product of the BF16 inputs in double,
 * C[m][n] = sum_k x[m][k] * w[n][k], for the listed rows.  Used to report
 * the error of the FP8 path against a BF16 GEMM; it pins nothing.
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint16_t *x, *w;
  int64_t ldx, ldw, N, K;
  const int64_t *rows;
  double *c;
} bgemm_ctx;

static void bgemm_item(int64_t idx, void *cx) {
  bgemm_ctx *p = (bgemm_ctx *)cx;
  int64_t i = idx / p->N, n = idx % p->N, m = p->rows[i];
  double acc = 0.0;
  for (int64_t k = 0; k < p->K; ++k)
    acc += (double)bf16_to_f32(p->x[m * p->ldx + k]) * (double)bf16_to_f32(p->w[n * p->ldw + k]);
  p->c[i * p->N + n] = acc;
}

void oracle_bf16_gemm_rows(const uint16_t *x, int64_t ldx, const uint16_t *w,
                           int64_t ldw, int64_t N, int64_t K,
                           const int64_t *rows, int64_t nrows, double *c) {
  bgemm_ctx p = {x, w, ldx, ldw, N, K, rows, c};
  par_for(nrows * N, bgemm_item, &p);
}

/* ------------------------------------------------------------------------
 * 128x1 requantisation from FP8-cached activations.  The forward pass keeps
 * its activations in FP8 ([dssusan] paragraph 2, compressing cached
 * activations; "Deepseek - Not For everyone" paragraph 3, caching activations
 * in FP8 for the Linear's backward pass) as 1x128 tiles, and the backward
 * pass needs the same tensor as 128x1 tiles ([dssusan] paragraph 4).
 * READING: dequantise each cached value with one FP32 multiply rounded to
 * nearest, x = fl32(decode(q) * s_row), then apply the 128x1 rule above to
 * those FP32 values.
 * q: E4M3 [T][C] (row stride ldq), s_rows: 1x128 scales s_rows[g * ld_s + t].
 * qT: E4M3 [C][T] (row stride ldqT), sT[tg * ld_sT + c].  T % 128 == 0,
 * C % 128 == 0.
 * ------------------------------------------------------------------------ */
typedef struct {
  const uint8_t *q;
  const float *s_rows;
  int64_t T, C, ldq, ld_s, ldqT, ld_sT;
  uint8_t *qT;
  float *sT;
  int pow2;
  double lut[256];
} rq_ctx;

static float dequant_f32(const rq_ctx *p, int64_t t, int64_t c) {
  float v = (float)p->lut[p->q[t * p->ldq + c]];
  return v * p->s_rows[(c / 128) * p->ld_s + t]; /* one FP32 multiply */
}

static void requant_T_channel(int64_t c, void *cx) {
  rq_ctx *p = (rq_ctx *)cx;
  for (int64_t tg = 0; tg < p->T / 128; ++tg) {
    float amax = 0.0f;
    for (int j = 0; j < 128; ++j) {
      float v = fabsf(dequant_f32(p, tg * 128 + j, c));
      if (v > amax) amax = v;
    }
    float s, inv;
    oracle_group_scale(amax, p->pow2, &s, &inv);
    p->sT[tg * p->ld_sT + c] = s;
    for (int j = 0; j < 128; ++j) {
      int64_t t = tg * 128 + j;
      float prod = dequant_f32(p, t, c) * inv;
      p->qT[c * p->ldqT + t] = oracle_e4m3_encode(prod);
    }
  }
}

void oracle_requant_act_T(const uint8_t *q, int64_t T, int64_t C, int64_t ldq,
                          const float *s_rows, int64_t ld_s, uint8_t *qT,
                          int64_t ldqT, float *sT, int64_t ld_sT, int pow2) {
  rq_ctx *p = (rq_ctx *)malloc(sizeof(rq_ctx));
  if (!p) return;
  *p = (rq_ctx){q, s_rows, T, C, ldq, ld_s, ldqT, ld_sT, qT, sT, pow2, {0}};
  for (int v = 0; v < 256; ++v) p->lut[v] = oracle_e4m3_decode((uint8_t)v);
  par_for(C, requant_T_channel, p);
  free(p);
}

/* ------------------------------------------------------------------------
 * Per-tensor quantisation, for comparison only: the standard practice the
 * pages contrast with fine-grained scaling ("Deepseek - Not For everyone",
 * paragraph 4: the max-abs of the whole tensor is mapped onto the largest FP8
 * value, which makes the result sensitive to outliers).  One scale for the
 * whole [M][K] tensor from its max-abs, by the same rule as a group's.
 * ------------------------------------------------------------------------ */
void oracle_quant_tensor(const uint16_t *x, int64_t M, int64_t K, int64_t ldx, uint8_t *q,
                         int64_t ldq, float *s_out, int pow2) {
  float amax = 0.0f;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k) {
      float v = fabsf(bf16_to_f32(x[m * ldx + k]));
      if (v > amax) amax = v;
    }
  float s, inv;
  oracle_group_scale(amax, pow2, &s, &inv);
  *s_out = s;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k)
      q[m * ldq + k] = oracle_e4m3_encode(bf16_to_f32(x[m * ldx + k]) * inv);
}
