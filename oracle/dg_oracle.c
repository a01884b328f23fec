/*
 * CPU oracle for the fine-grained-scaled FP8 GEMM family (dense NT, M-grouped
 * contiguous, M-grouped masked, K-grouped).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Everything here is the plain definition, in FP64:
 *   - E4M3 codes decode by the OCP OFP8 v1.0 E4M3 rule (bias 7, no infinities,
 *     S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9).
 *   - Quantisation: a scale s = 2^e per 1x128 row group (activations, LHS) or
 *     per 128x128 block (weights, RHS), e the smallest integer with
 *     448 * 2^e >= amax of the group, values cast to E4M3 with
 *     round-to-nearest-even, saturating at +-448.
 *     Fine-grained scaling: "DeepGEMM: kernels GEMM FP8 limpos e eficientes por
 *     meio de scaling granular" (pt.news.hada.io), title and section
 *     "Interface GEMM e restrições de layout"; the launch report on feifmx.com
 *     (Feb 2025), paragraph on fine-grained scaling from DeepSeek-V3.
 *   - UE8M0 packing, four 8-bit exponents per 32-bit word, MN-major: same page,
 *     section "Interface GEMM e restrições de layout" (SM100 scale format,
 *     transposed TMA-aligned LHS scales).
 *   - GEMM D = C + A @ B.T (NT): same page, same section.
 *   - Contiguous M-grouped layout and masked M-grouped layout: same page,
 *     section "GEMM denso e grouped".
 *   - K-grouped (weight-gradient) layout, experts stacked along K: same page,
 *     same section; the reading of its operand layout is stated beside
 *     or_gemm_k_grouped below.
 *
 * Evaluation order of the GEMM: for each 128-wide K block the products of the
 * decoded codes are summed in FP64 (exact: every product is a multiple of
 * 2^-18 below 448^2, 128 of them stay far below 2^53 units), the block sum is
 * multiplied by the two power-of-two scales (exact), and the block results are
 * added in FP64 in increasing K order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_BLOCK_K 128
#define OR_E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* E4M3 (OCP OFP8 v1.0)                                                      */
/* ------------------------------------------------------------------------ */

static double g_e4m3[256];
static double g_pos_mag[127]; /* magnitudes of codes 0x00..0x7E, ascending */
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
  for (int code = 0; code < 256; ++code) {
    int sign = (code >> 7) & 1;
    int exp_field = (code >> 3) & 0xF;
    int man = code & 0x7;
    double mag;
    if (exp_field == 0xF && man == 0x7) {
      mag = NAN;
    } else if (exp_field == 0) {
      mag = ldexp((double)man, -9); /* m/8 * 2^(1-7) */
    } else {
      mag = ldexp(1.0 + man / 8.0, exp_field - 7);
    }
    g_e4m3[code] = sign ? -mag : mag;
  }
  for (int code = 0; code < 127; ++code) g_pos_mag[code] = g_e4m3[code];
}

static void ensure_tables(void) { pthread_once(&g_once, build_tables); }

double or_e4m3_decode(uint8_t code) {
  ensure_tables();
  return g_e4m3[code];
}

void or_e4m3_table(double* out256) {
  ensure_tables();
  memcpy(out256, g_e4m3, sizeof(g_e4m3));
}

/* Round-to-nearest-even onto the E4M3 grid, saturating at +-448.  The
 * magnitude grid (codes 0..126) is increasing in the code, so the nearest
 * value is found by binary search; a tie goes to the even code (mantissa LSB
 * zero).  NaN maps to the positive NaN code 0x7F.  The sign is kept, so a
 * negative value that rounds to zero gives 0x80. */
uint8_t or_e4m3_encode(double x) {
  ensure_tables();
  if (isnan(x)) return 0x7F;
  int neg = signbit(x) ? 1 : 0;
  double mag = fabs(x);
  int code;
  if (mag >= OR_E4M3_MAX) {
    code = 0x7E;
  } else {
    /* largest lo with g_pos_mag[lo] <= mag */
    int lo = 0, hi = 126;
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (g_pos_mag[mid] <= mag) lo = mid; else hi = mid - 1;
    }
    if (g_pos_mag[lo] == mag) {
      code = lo;
    } else {
      double below = g_pos_mag[lo], above = g_pos_mag[lo + 1];
      double d_lo = mag - below, d_hi = above - mag;
      if (d_lo < d_hi) code = lo;
      else if (d_hi < d_lo) code = lo + 1;
      else code = (lo % 2 == 0) ? lo : lo + 1;
    }
  }
  return (uint8_t)(neg ? (code | 0x80) : code);
}

/* ------------------------------------------------------------------------ */
/* Scale rule                                                                */
/* ------------------------------------------------------------------------ */

/* Smallest integer e with 448 * 2^e >= amax, clamped to the UE8M0 range
 * [-127, 127].  amax == 0 (an all-zero group) gives e = 0, scale 1. */
int or_scale_exponent(double amax) {
  if (!(amax > 0.0)) return 0;
  int e;
  frexp(amax / OR_E4M3_MAX, &e); /* first guess, fixed exactly below */
  while (ldexp(OR_E4M3_MAX, e) < amax) ++e;
  while (ldexp(OR_E4M3_MAX, e - 1) >= amax) --e;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* ------------------------------------------------------------------------ */
/* Threading helper: split [0, n) in contiguous chunks over worker threads.   */
/* ------------------------------------------------------------------------ */

static int g_threads = 0;

void or_set_threads(int n) { g_threads = n; }

int or_get_threads(void) {
  if (g_threads > 0) return g_threads;
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

typedef void (*or_range_fn)(void* ctx, int64_t begin, int64_t end);

typedef struct {
  or_range_fn fn;
  void* ctx;
  int64_t begin, end;
} or_job;

static void* or_job_main(void* p) {
  or_job* j = (or_job*)p;
  j->fn(j->ctx, j->begin, j->end);
  return NULL;
}

static void parallel_for(int64_t n, or_range_fn fn, void* ctx) {
  int t = or_get_threads();
  if (t > 256) t = 256;
  if (n < t) t = (int)(n > 0 ? n : 1);
  if (t <= 1) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t th[256];
  or_job jobs[256];
  int64_t chunk = (n + t - 1) / t;
  int started = 0;
  for (int i = 0; i < t; ++i) {
    int64_t b = i * chunk, e = b + chunk < n ? b + chunk : n;
    if (b >= e) break;
    jobs[i].fn = fn; jobs[i].ctx = ctx; jobs[i].begin = b; jobs[i].end = e;
    if (pthread_create(&th[i], NULL, or_job_main, &jobs[i]) != 0) {
      or_job_main(&jobs[i]); /* run inline if a thread cannot start */
      th[i] = 0;
    }
    started = i + 1;
  }
  for (int i = 0; i < started; ++i)
    if (th[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* Quantisation                                                              */
/* ------------------------------------------------------------------------ */

typedef struct {
  const float* x;
  int64_t rows, cols;
  int block_rows;
  uint8_t* q;
  int32_t* sf_exp;   /* [ceil(rows/block_rows), cols/128] */
  double* sf_scale;  /* same shape, 2^e; may be NULL */
} quant_ctx;

static void quant_range(void* p, int64_t rb_begin, int64_t rb_end) {
  quant_ctx* c = (quant_ctx*)p;
  int64_t kblocks = c->cols / OR_BLOCK_K;
  for (int64_t rb = rb_begin; rb < rb_end; ++rb) {
    int64_t r0 = rb * c->block_rows;
    int64_t r1 = r0 + c->block_rows < c->rows ? r0 + c->block_rows : c->rows;
    for (int64_t kb = 0; kb < kblocks; ++kb) {
      int64_t c0 = kb * OR_BLOCK_K;
      double amax = 0.0;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t j = c0; j < c0 + OR_BLOCK_K; ++j) {
          double v = fabs((double)c->x[r * c->cols + j]);
          if (v > amax) amax = v;
        }
      int e = or_scale_exponent(amax);
      c->sf_exp[rb * kblocks + kb] = e;
      if (c->sf_scale) c->sf_scale[rb * kblocks + kb] = ldexp(1.0, e);
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t j = c0; j < c0 + OR_BLOCK_K; ++j)
          c->q[r * c->cols + j] = or_e4m3_encode(ldexp((double)c->x[r * c->cols + j], -e));
    }
  }
}

/* x: FP32 [rows, cols] row-major, cols % 128 == 0.  block_rows = 1 gives the
 * 1x128 activation grouping, 128 the 128x128 weight blocks (the last block
 * along rows covers only the rows that exist).  Returns 0, or -1 on bad
 * arguments. */
int or_quantize(const float* x, int64_t rows, int64_t cols, int block_rows,
                uint8_t* q, int32_t* sf_exp, double* sf_scale) {
  ensure_tables();
  if (!x || !q || !sf_exp || rows < 0 || cols < 0 || cols % OR_BLOCK_K != 0) return -1;
  if (block_rows != 1 && block_rows != 128) return -1;
  quant_ctx c = {x, rows, cols, block_rows, q, sf_exp, sf_scale};
  int64_t rblocks = (rows + block_rows - 1) / block_rows;
  parallel_for(rblocks, quant_range, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* UE8M0 packing (SM100 scale layout)                                         */
/* ------------------------------------------------------------------------ */

/* sf_exp: [groups, ceil(mn/block_rows), kblocks] exponents.
 * packed: [groups, ceil(kblocks/4), mn_pad] int32, mn_pad = mn rounded up to a
 * multiple of 4 (16 bytes).  Word (g, j, r) holds in byte t (t = 0..3, least
 * significant first) the biased exponent e + 127 of K block 4j + t for row r
 * (for block_rows = 128, the exponent of row r's 128-row block).  Bytes past
 * the last K block and rows in [mn, mn_pad) are zero. */
int or_pack_ue8m0(const int32_t* sf_exp, int64_t groups, int64_t mn, int64_t kblocks,
                  int block_rows, int32_t* packed) {
  if (!sf_exp || !packed || groups < 0 || mn < 0 || kblocks < 0) return -1;
  if (block_rows != 1 && block_rows != 128) return -1;
  int64_t mn_pad = (mn + 3) / 4 * 4;
  int64_t kpacks = (kblocks + 3) / 4;
  int64_t mn_blocks = (mn + block_rows - 1) / block_rows;
  for (int64_t g = 0; g < groups; ++g)
    for (int64_t j = 0; j < kpacks; ++j)
      for (int64_t r = 0; r < mn_pad; ++r) {
        uint32_t word = 0;
        if (r < mn) {
          for (int t = 0; t < 4; ++t) {
            int64_t kb = 4 * j + t;
            if (kb >= kblocks) break;
            int32_t e = sf_exp[(g * mn_blocks + r / block_rows) * kblocks + kb];
            uint32_t biased = (uint32_t)(e + 127) & 0xFFu;
            word |= biased << (8 * t);
          }
        }
        packed[(g * kpacks + j) * mn_pad + r] = (int32_t)word;
      }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* GEMM                                                                       */
/* ------------------------------------------------------------------------ */

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof(f));
  return (double)f;
}

/* One output row: o[n] = c[n] + sum_kb (sum_{k in kb} dec(a[k]) dec(b[n,k])) * sa[kb] * sb[n/128, kb]
 * a: K codes of the row; sa: K/128 scales of the row; b: [N, K] codes;
 * sb: [ceil(N/128), K/128] scales; c: N bf16 values or NULL. */
static void gemm_row(const uint8_t* a, const double* sa, const uint8_t* b, const double* sb,
                     const uint16_t* c, int64_t N, int64_t K, double* o) {
  int64_t kblocks = K / OR_BLOCK_K;
  for (int64_t n = 0; n < N; ++n) {
    double acc = c ? bf16_bits_to_double(c[n]) : 0.0;
    const uint8_t* brow = b + n * K;
    for (int64_t kb = 0; kb < kblocks; ++kb) {
      double inner = 0.0;
      for (int64_t k = kb * OR_BLOCK_K; k < (kb + 1) * OR_BLOCK_K; ++k)
        inner += g_e4m3[a[k]] * g_e4m3[brow[k]];
      acc += inner * sa[kb] * sb[(n / OR_BLOCK_K) * kblocks + kb];
    }
    o[n] = acc;
  }
}

typedef struct {
  const uint8_t* qa; const double* sa;
  const uint8_t* qb; const double* sb;
  const uint16_t* c;
  int64_t N, K;
  const int64_t* rows; /* NULL: row i is i */
  double* o;
} dense_ctx;

static void dense_range(void* p, int64_t i0, int64_t i1) {
  dense_ctx* c = (dense_ctx*)p;
  int64_t kblocks = c->K / OR_BLOCK_K;
  for (int64_t i = i0; i < i1; ++i) {
    int64_t m = c->rows ? c->rows[i] : i;
    gemm_row(c->qa + m * c->K, c->sa + m * kblocks, c->qb, c->sb,
             c->c ? c->c + m * c->N : NULL, c->N, c->K, c->o + i * c->N);
  }
}

/* Dense NT: o[M,N] = C + dequant(A) @ dequant(B)^T.
 * qa: [M,K] E4M3 codes, sa: [M, K/128] scales; qb: [N,K] codes,
 * sb: [ceil(N/128), K/128] scales; c: [M,N] bf16 bits or NULL. */
int or_gemm_nt(const uint8_t* qa, const double* sa, const uint8_t* qb, const double* sb,
               const uint16_t* c, int64_t M, int64_t N, int64_t K, double* o) {
  ensure_tables();
  if (!qa || !sa || !qb || !sb || !o || M < 0 || N < 0 || K % OR_BLOCK_K != 0) return -1;
  dense_ctx ctx = {qa, sa, qb, sb, c, N, K, NULL, o};
  parallel_for(M, dense_range, &ctx);
  return 0;
}

/* Same as or_gemm_nt for a chosen list of rows: o[i, :] is row rows[i]. */
int or_gemm_nt_rows(const uint8_t* qa, const double* sa, const uint8_t* qb, const double* sb,
                    const uint16_t* c, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                    double* o) {
  ensure_tables();
  if (!qa || !sa || !qb || !sb || !o || !rows || N < 0 || K % OR_BLOCK_K != 0) return -1;
  dense_ctx ctx = {qa, sa, qb, sb, c, N, K, rows, o};
  parallel_for(nrows, dense_range, &ctx);
  return 0;
}

typedef struct {
  const uint8_t* qa; const double* sa;
  const uint8_t* qb; const double* sb;
  const int32_t* group_of_row; /* per output row: group id, or -1 = not written */
  int64_t num_groups, N, K;
  const int64_t* rows;
  double* o;
  uint8_t* written;
} grouped_ctx;

static void grouped_range(void* p, int64_t i0, int64_t i1) {
  grouped_ctx* c = (grouped_ctx*)p;
  int64_t kblocks = c->K / OR_BLOCK_K;
  int64_t nblocks = (c->N + OR_BLOCK_K - 1) / OR_BLOCK_K;
  for (int64_t i = i0; i < i1; ++i) {
    int64_t r = c->rows ? c->rows[i] : i;
    int32_t g = c->group_of_row[r];
    if (g < 0 || g >= c->num_groups) {
      c->written[i] = 0;
      for (int64_t n = 0; n < c->N; ++n) c->o[i * c->N + n] = 0.0;
      continue;
    }
    c->written[i] = 1;
    gemm_row(c->qa + r * c->K, c->sa + r * kblocks, c->qb + (int64_t)g * c->N * c->K,
             c->sb + (int64_t)g * nblocks * kblocks, NULL, c->N, c->K, c->o + i * c->N);
  }
}

/* M-grouped contiguous: the token rows of all experts are concatenated along
 * M; m_indices[r] is the expert of row r, or -1 for a padding row, which is not
 * written.  qa: [m_sum,K], sa: [m_sum,K/128]; qb: [G,N,K],
 * sb: [G, ceil(N/128), K/128]; o: [m_sum, N]; written: [m_sum] (1 = row
 * computed).  An index outside [0, G) is treated like -1.  rows (optional)
 * restricts the evaluation to a list of rows; o and written are then indexed
 * by list position. */
int or_gemm_contiguous(const uint8_t* qa, const double* sa, const uint8_t* qb, const double* sb,
                       const int32_t* m_indices, int64_t m_sum, int64_t num_groups, int64_t N,
                       int64_t K, const int64_t* rows, int64_t nrows, double* o, uint8_t* written) {
  ensure_tables();
  if (!qa || !sa || !qb || !sb || !m_indices || !o || !written || N < 0 ||
      K % OR_BLOCK_K != 0)
    return -1;
  grouped_ctx ctx = {qa, sa, qb, sb, m_indices, num_groups, N, K, rows, o, written};
  parallel_for(rows ? nrows : m_sum, grouped_range, &ctx);
  return 0;
}

/* M-grouped masked: group g owns rows [g*cap, (g+1)*cap) of A [G,cap,K] and of
 * the output [G,cap,N]; only its first masked_m[g] rows are computed and
 * written (masked_m is clamped to [0, cap]).  rows (optional) as above, as
 * flat indices g*cap + r. */
int or_gemm_masked(const uint8_t* qa, const double* sa, const uint8_t* qb, const double* sb,
                   const int32_t* masked_m, int64_t num_groups, int64_t cap, int64_t N, int64_t K,
                   const int64_t* rows, int64_t nrows, double* o, uint8_t* written) {
  ensure_tables();
  if (!qa || !sa || !qb || !sb || !masked_m || !o || !written || N < 0 || cap < 0 ||
      K % OR_BLOCK_K != 0)
    return -1;
  int64_t total = num_groups * cap;
  int32_t* group_of_row = (int32_t*)malloc((size_t)(total > 0 ? total : 1) * sizeof(int32_t));
  if (!group_of_row) return -2;
  for (int64_t g = 0; g < num_groups; ++g) {
    int64_t valid = masked_m[g];
    if (valid < 0) valid = 0;
    if (valid > cap) valid = cap;
    for (int64_t r = 0; r < cap; ++r) group_of_row[g * cap + r] = r < valid ? (int32_t)g : -1;
  }
  grouped_ctx ctx = {qa, sa, qb, sb, group_of_row, num_groups, N, K, rows, o, written};
  parallel_for(rows ? nrows : total, grouped_range, &ctx);
  free(group_of_row);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* K-grouped layout (MoE weight gradients)                                    */
/* ------------------------------------------------------------------------ */
/* "DeepGEMM: kernels GEMM FP8 limpos e eficientes por meio de scaling
 * granular" (pt.news.hada.io), section "GEMM denso e grouped": a grouped API
 * along K for the weight backward of MoE models, M and N fixed, named
 * k_grouped_fp8_gemm_tn_contiguous.  The page gives no more; the reading
 * taken here: the experts' token rows are stacked along K (each expert's
 * segment a multiple of 128 rows), A is stored [sum_k, M] and B [sum_k, N]
 * ("TN": both with the reduction axis outermost), every 128-row block of one
 * column carries one power-of-two scale (the same fine-grained grouping, along
 * the reduction axis), and expert g produces
 *   D[g] = C[g] + A_g^T B_g   (FP32 [M, N]).                                */

typedef struct {
  const float* x;
  int64_t rows, cols;
  uint8_t* q;
  int32_t* sf_exp;   /* [rows/128, cols] */
  double* sf_scale;  /* same shape, 2^e; may be NULL */
} quant_cols_ctx;

static void quant_cols_range(void* p, int64_t rb_begin, int64_t rb_end) {
  quant_cols_ctx* c = (quant_cols_ctx*)p;
  for (int64_t rb = rb_begin; rb < rb_end; ++rb) {
    int64_t r0 = rb * OR_BLOCK_K;
    for (int64_t j = 0; j < c->cols; ++j) {
      double amax = 0.0;
      for (int64_t r = r0; r < r0 + OR_BLOCK_K; ++r) {
        double v = fabs((double)c->x[r * c->cols + j]);
        if (v > amax) amax = v;
      }
      int e = or_scale_exponent(amax);
      c->sf_exp[rb * c->cols + j] = e;
      if (c->sf_scale) c->sf_scale[rb * c->cols + j] = ldexp(1.0, e);
      for (int64_t r = r0; r < r0 + OR_BLOCK_K; ++r)
        c->q[r * c->cols + j] = or_e4m3_encode(ldexp((double)c->x[r * c->cols + j], -e));
    }
  }
}

/* x: FP32 [rows, cols] row-major, rows % 128 == 0: one scale per 128 rows of
 * each column (the reduction axis is the row axis).  Returns 0, or -1. */
int or_quantize_cols(const float* x, int64_t rows, int64_t cols, uint8_t* q, int32_t* sf_exp,
                     double* sf_scale) {
  ensure_tables();
  if (!x || !q || !sf_exp || rows < 0 || cols < 0 || rows % OR_BLOCK_K != 0) return -1;
  quant_cols_ctx c = {x, rows, cols, q, sf_exp, sf_scale};
  parallel_for(rows / OR_BLOCK_K, quant_cols_range, &c);
  return 0;
}

typedef struct {
  const uint8_t* qa; const double* sa;
  const uint8_t* qb; const double* sb;
  const int64_t* kb_start; /* [G + 1] first K block of each expert */
  int64_t M, N;
  const float* c;
  const int64_t* rows;
  double* o;
} kgrouped_ctx;

static void kgrouped_range(void* p, int64_t i0, int64_t i1) {
  kgrouped_ctx* c = (kgrouped_ctx*)p;
  double* inner = (double*)malloc((size_t)(c->N > 0 ? c->N : 1) * sizeof(double));
  if (!inner) return;
  for (int64_t i = i0; i < i1; ++i) {
    int64_t flat = c->rows ? c->rows[i] : i; /* g * M + m */
    int64_t g = flat / c->M, m = flat % c->M;
    double* acc = c->o + i * c->N;
    for (int64_t n = 0; n < c->N; ++n) acc[n] = c->c ? (double)c->c[flat * c->N + n] : 0.0;
    for (int64_t kb = c->kb_start[g]; kb < c->kb_start[g + 1]; ++kb) {
      for (int64_t n = 0; n < c->N; ++n) inner[n] = 0.0;
      for (int64_t k = kb * OR_BLOCK_K; k < (kb + 1) * OR_BLOCK_K; ++k) {
        double av = g_e4m3[c->qa[k * c->M + m]];
        const uint8_t* brow = c->qb + k * c->N;
        for (int64_t n = 0; n < c->N; ++n) inner[n] += av * g_e4m3[brow[n]];
      }
      double sam = c->sa[kb * c->M + m];
      for (int64_t n = 0; n < c->N; ++n) acc[n] += inner[n] * sam * c->sb[kb * c->N + n];
    }
  }
  free(inner);
}

/* K-grouped TN: qa [sum_k, M] codes, sa [sum_k/128, M] scales; qb [sum_k, N]
 * codes, sb [sum_k/128, N] scales; ks [G] rows per expert (each >= 0 and a
 * multiple of 128, summing to sum_k); c [G, M, N] FP32 or NULL.
 * o [G, M, N] = C + per expert sum over its K blocks, in increasing K order,
 * of (exact FP64 inner sum over the block) * sa * sb.  rows (optional) lists
 * flat indices g * M + m; o is then [nrows, N].  Returns 0, or -1. */
int or_gemm_k_grouped(const uint8_t* qa, const double* sa, const uint8_t* qb, const double* sb,
                      const int32_t* ks, int64_t num_groups, int64_t M, int64_t N, int64_t sum_k,
                      const float* c, const int64_t* rows, int64_t nrows, double* o) {
  ensure_tables();
  if (!qa || !sa || !qb || !sb || !ks || !o || num_groups < 0 || M < 0 || N < 0 || sum_k < 0 ||
      sum_k % OR_BLOCK_K != 0)
    return -1;
  int64_t* kb_start = (int64_t*)malloc((size_t)(num_groups + 1) * sizeof(int64_t));
  if (!kb_start) return -2;
  kb_start[0] = 0;
  for (int64_t g = 0; g < num_groups; ++g) {
    if (ks[g] < 0 || ks[g] % OR_BLOCK_K != 0) {
      free(kb_start);
      return -1;
    }
    kb_start[g + 1] = kb_start[g] + ks[g] / OR_BLOCK_K;
  }
  if (kb_start[num_groups] * OR_BLOCK_K != sum_k) {
    free(kb_start);
    return -1;
  }
  if (rows)
    for (int64_t i = 0; i < nrows; ++i)
      if (rows[i] < 0 || rows[i] >= num_groups * M) {
        free(kb_start);
        return -1;
      }
  kgrouped_ctx ctx = {qa, sa, qb, sb, kb_start, M, N, c, rows, o};
  parallel_for(rows ? nrows : num_groups * M, kgrouped_range, &ctx);
  free(kb_start);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* BF16 rounding of an FP64 value (round to nearest, ties to even), used to
 * state the exact expected output of cases whose FP32 accumulation is exact. */
/* ------------------------------------------------------------------------ */

uint16_t or_bf16_rne(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double mag = fabs(x);
  if (mag == 0.0) return sign;
  /* bf16: 8 significant bits, exponent range of FP32 */
  int e;
  frexp(mag, &e);              /* mag = f * 2^e, f in [0.5, 1) */
  int exp_unbiased = e - 1;    /* mag in [2^(e-1), 2^e) */
  if (exp_unbiased < -126) exp_unbiased = -126; /* subnormal spacing */
  double ulp = ldexp(1.0, exp_unbiased - 7);
  double q = mag / ulp;        /* exact: scaling by a power of two */
  double fl = floor(q);
  double rem = q - fl;
  double r;
  if (rem > 0.5) r = fl + 1.0;
  else if (rem < 0.5) r = fl;
  else r = fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
  double val = r * ulp;
  if (val >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80); /* overflow to inf */
  float f = (float)val; /* exact: val has 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof(u));
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the Python wrapper.                                      */
/* ------------------------------------------------------------------------ */

void or_e4m3_encode_array(const double* x, int64_t n, uint8_t* out) {
  ensure_tables();
  for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i]);
}

void or_bf16_rne_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_rne(x[i]);
}
