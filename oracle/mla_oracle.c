/*
 * fp64 CPU oracle for sequence-sharded MLA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code with
 * the CUDA path: it has its own bf16 and e4m3 decoding, its own page gather
 * and its own softmax.  It is deliberately plain and slow.
 *
 * What it computes (page "Decode Context Parallelism", sections 4.1 and 5.3;
 * page "Kimi K3 in vLLM: Specialized CuTe DSL Decode on NVIDIA GB300",
 * section 1):
 *
 *   For request b, query position i, head h, over the gathered token set T:
 *     s_t  = scale * sum_{d<576} q[b,i,h,d] * K_t[d]          (absorbed form)
 *     lse  = ln sum_{t in T} exp(s_t)
 *     out  = sum_{t in T} exp(s_t - lse) * K_t[0:512]            (V = c_kv)
 *     y    = out . W_UV[h]   (512 -> 128, optional v-projection)
 *
 *   K_t is row (t mod 64) of page block_table[b][t / 64] of the latent cache,
 *   laid out [c_kv(512) | k_rope(64)].  fp8 caches are decoded exactly as
 *   e4m3(code) * scale_t.
 *
 *   T = { t < L_b }, intersected with { t <= L_b - q_len + i } when causal
 *   (query i of a 1+N verify step sees the committed context plus drafts up
 *   to itself), and with the shard's positions when a shard is requested:
 *     interleaved:  t mod N == s
 *     contiguous:   s*c <= t < min((s+1)*c, L_b),  c = ceil(L_b / N)
 *   ("Decode Context Parallelism" section 4: each GPU owns a chunk of token
 *   positions of the same sequence).  An empty T gives lse = -inf, out = 0.
 *
 *   The LSE merge of shards ("Decode Context Parallelism" section 4.1, the
 *   reweighting of partial outputs by their LSE) is:
 *     M = max_s lse_s,  w_s = exp(lse_s - M),
 *     lse = M + ln sum_s w_s,  out = sum_s w_s out_s / sum_s w_s.
 *
 * The softmax is the two-pass textbook form (max, then sum), not the online
 * form, so that it shares no structure with the kernel.
 *
 * Parity pins (tests/test_oracle_pins.py): brute force in extended precision
 * without max subtraction, for bf16 caches and for fp8 caches with
 * row-varying token scales; single-token (bf16 and fp8) and identical-key
 * closed forms; the
 * sharded-then-merged result equals the unsharded one for every N and both
 * layouts; block-table page permutation invariance; causal row i equals a
 * q_len = 1 query at context L - q_len + 1 + i; e4m3 decoding against the
 * closed form and torch's float8_e4m3fn; W_UV against a library matmul.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_QK 576
#define D_V 512
#define D_UV 128
#define PAGE 64

enum { ORACLE_OK = 0, ORACLE_BAD_PAGE = -1, ORACLE_NOMEM = -2, ORACLE_BAD_ARG = -3 };
enum { LAYOUT_INTERLEAVED = 0, LAYOUT_CONTIGUOUS = 1 };

/* bf16 bit pattern -> value (exact). */
static double bf16_value(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OCP e4m3 ("fn") code -> value: bias 7, no infinities, S.1111.111 is NaN.
 *   exponent field 0:   (m / 8) * 2^-6
 *   otherwise:          (1 + m / 8) * 2^(e - 7)                              */
static double e4m3_value(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

void oracle_e4m3_decode(const uint8_t* codes, size_t n, double* out) {
  for (size_t k = 0; k < n; ++k) out[k] = e4m3_value(codes[k]);
}

void oracle_bf16_decode(const uint16_t* bits, size_t n, double* out) {
  for (size_t k = 0; k < n; ++k) out[k] = bf16_value(bits[k]);
}

typedef struct {
  const void* kv;
  const float* scale;   /* fp8 only */
  int fp8;
  int num_pages;
  const int32_t* block_table;
  int max_pages;
} cache_view;

/* Copy K_t (all 576 dims) of request b into dst as doubles. */
static int gather_row(const cache_view* cv, int b, long t, double* dst) {
  long slot = t / PAGE;
  if (slot >= cv->max_pages) return ORACLE_BAD_PAGE;
  int32_t page = cv->block_table[(size_t)b * cv->max_pages + slot];
  if (page < 0 || page >= cv->num_pages) return ORACLE_BAD_PAGE;
  size_t row = (size_t)page * PAGE + (size_t)(t % PAGE);
  if (cv->fp8) {
    const uint8_t* src = (const uint8_t*)cv->kv + row * D_QK;
    double s = (double)cv->scale[row];
    for (int d = 0; d < D_QK; ++d) dst[d] = e4m3_value(src[d]) * s;
  } else {
    const uint16_t* src = (const uint16_t*)cv->kv + row * D_QK;
    for (int d = 0; d < D_QK; ++d) dst[d] = bf16_value(src[d]);
  }
  return ORACLE_OK;
}

/* Is token t of a request with context L in the set seen by query i? */
static int token_visible(long t, long L, int q_len, int i, int causal, int shard,
                         int nshards, int layout) {
  if (t < 0 || t >= L) return 0;
  if (causal && t > L - q_len + i) return 0;
  if (shard < 0) return 1;
  if (layout == LAYOUT_INTERLEAVED) return (t % nshards) == shard;
  long c = (L + nshards - 1) / nshards;
  return t >= (long)shard * c && t < (long)(shard + 1) * c;
}

/* Shard that owns token t of a context of L tokens (-1 if t is outside). */
int oracle_token_owner(long t, long L, int nshards, int layout) {
  for (int s = 0; s < nshards; ++s)
    if (token_visible(t, L, 1, 0, 0, s, nshards, layout)) return s;
  return -1;
}

/*
 * Attention for a list of query rows.  Row index r encodes
 * (b * q_len + i) * H + h.  rows == NULL means all B*q_len*H rows in order.
 * shard < 0 selects the unsharded token set.
 *
 * q_lens (may be NULL): request b carries q_lens[b] <= q_len query tokens;
 * its rows i >= q_lens[b] are padding and see no token, and its causal
 * query i sees t <= L - q_lens[b] + i.  This is a batch of verify steps
 * with different draft counts padded to one q_len ("GLM-5.2" deployment
 * post, sections 2.1-2.2: 1 + N tokens per request per step).
 */
int oracle_attend(const uint16_t* q, int B, int q_len, int H, const void* kv,
                  const float* kv_scale, int kv_fp8, int num_pages,
                  const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                  const int32_t* q_lens, int causal, double softmax_scale, int shard,
                  int nshards, int layout, const int64_t* rows, int64_t n_rows, double* out,
                  double* lse) {
  if (B <= 0 || q_len <= 0 || H <= 0) return ORACLE_BAD_ARG;
  if (shard >= 0 && (nshards <= 0 || shard >= nshards)) return ORACLE_BAD_ARG;
  cache_view cv = {kv, kv_scale, kv_fp8, num_pages, block_table, max_pages};
  int64_t total = (int64_t)B * q_len * H;
  if (rows == NULL) n_rows = total;
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t k = 0; k < n_rows; ++k) {
    int64_t r = rows ? rows[k] : k;
    int h = (int)(r % H);
    int i = (int)((r / H) % q_len);
    int b = (int)(r / ((int64_t)H * q_len));
    long L = seq_lens[b];
    int qn = q_lens ? q_lens[b] : q_len;
    if (i >= qn) { /* padding row */
      double* o0 = out + (size_t)k * D_V;
      for (int c = 0; c < D_V; ++c) o0[c] = 0.0;
      lse[k] = -INFINITY;
      continue;
    }
    double qv[D_QK], kt[D_QK];
    const uint16_t* qrow = q + (size_t)r * D_QK;
    for (int d = 0; d < D_QK; ++d) qv[d] = bf16_value(qrow[d]);
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!s) {
#pragma omp atomic write
      status = ORACLE_NOMEM;
      continue;
    }
    /* pass 1: logits of visible tokens, and their maximum */
    double m = -INFINITY;
    int bad = 0;
    for (long t = 0; t < L; ++t) {
      if (!token_visible(t, L, qn, i, causal, shard, nshards, layout)) continue;
      if (gather_row(&cv, b, t, kt) != ORACLE_OK) { bad = 1; break; }
      double acc = 0.0;
      for (int d = 0; d < D_QK; ++d) acc += qv[d] * kt[d];
      s[t] = softmax_scale * acc;
      if (s[t] > m) m = s[t];
    }
    double* o = out + (size_t)k * D_V;
    for (int c = 0; c < D_V; ++c) o[c] = 0.0;
    if (bad) {
#pragma omp atomic write
      status = ORACLE_BAD_PAGE;
      free(s);
      continue;
    }
    if (m == -INFINITY) { /* empty token set */
      lse[k] = -INFINITY;
      free(s);
      continue;
    }
    /* pass 2: normaliser */
    double z = 0.0;
    for (long t = 0; t < L; ++t)
      if (token_visible(t, L, qn, i, causal, shard, nshards, layout)) z += exp(s[t] - m);
    double l = m + log(z);
    lse[k] = l;
    /* pass 3: probability-weighted sum of the latent values */
    for (long t = 0; t < L; ++t) {
      if (!token_visible(t, L, qn, i, causal, shard, nshards, layout)) continue;
      gather_row(&cv, b, t, kt);
      double p = exp(s[t] - l);
      for (int c = 0; c < D_V; ++c) o[c] += p * kt[c];
    }
    free(s);
  }
  return status;
}

/* Row of token t of request b for KV head kh in a GQA cache, or NULL if the
 * block-table entry is missing or out of range. */
static const uint16_t* gqa_row(const uint16_t* cache, const int32_t* block_table, int max_pages,
                               int num_pages, int Hkv, int D, int b, int kh, long t) {
  long slot = t / PAGE;
  if (slot >= max_pages) return NULL;
  int32_t page = block_table[(size_t)b * max_pages + slot];
  if (page < 0 || page >= num_pages) return NULL;
  return cache + (((size_t)page * PAGE + (size_t)(t % PAGE)) * Hkv + kh) * D;
}

/*
 * Grouped-query attention (GQA) over a paged cache, the second backend of
 * "Decode Context Parallelism" (section 5.4): the cache stores Hkv KV heads
 * of width D, separate K and V,
 *   k_cache, v_cache: bf16 [num_pages][64][Hkv][D],
 * and query head h attends with KV head h / (H / Hkv) -- the KV heads are
 * broadcast over their groups of H / Hkv consecutive query heads.  Token
 * sets, sharding, causal masking and the two-pass softmax are those of
 * oracle_attend; rows r = (b * q_len + i) * H + h, out [n_rows][D].
 */
int oracle_gqa_attend(const uint16_t* q, int B, int q_len, int H, int Hkv, int D,
                      const uint16_t* k_cache, const uint16_t* v_cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                      int causal, double softmax_scale, int shard, int nshards, int layout,
                      const int64_t* rows, int64_t n_rows, double* out, double* lse) {
  if (B <= 0 || q_len <= 0 || H <= 0 || Hkv <= 0 || D <= 0 || H % Hkv != 0)
    return ORACLE_BAD_ARG;
  if (shard >= 0 && (nshards <= 0 || shard >= nshards)) return ORACLE_BAD_ARG;
  const int group = H / Hkv;
  int64_t total = (int64_t)B * q_len * H;
  if (rows == NULL) n_rows = total;
  int status = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t k = 0; k < n_rows; ++k) {
    int64_t r = rows ? rows[k] : k;
    int h = (int)(r % H);
    int i = (int)((r / H) % q_len);
    int b = (int)(r / ((int64_t)H * q_len));
    int kh = h / group;
    long L = seq_lens[b];
    double* o = out + (size_t)k * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!qv || !s) {
      free(qv);
      free(s);
#pragma omp atomic write
      status = ORACLE_NOMEM;
      continue;
    }
    const uint16_t* qrow = q + (size_t)r * D;
    for (int d = 0; d < D; ++d) qv[d] = bf16_value(qrow[d]);
    double m = -INFINITY;
    int bad = 0;
    for (long t = 0; t < L; ++t) {
      if (!token_visible(t, L, q_len, i, causal, shard, nshards, layout)) continue;
      const uint16_t* kr = gqa_row(k_cache, block_table, max_pages, num_pages, Hkv, D, b, kh, t);
      if (!kr) { bad = 1; break; }
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += qv[d] * bf16_value(kr[d]);
      s[t] = softmax_scale * acc;
      if (s[t] > m) m = s[t];
    }
    if (bad) {
#pragma omp atomic write
      status = ORACLE_BAD_PAGE;
    } else if (m == -INFINITY) {
      lse[k] = -INFINITY;
    } else {
      double z = 0.0;
      for (long t = 0; t < L; ++t)
        if (token_visible(t, L, q_len, i, causal, shard, nshards, layout)) z += exp(s[t] - m);
      double l = m + log(z);
      lse[k] = l;
      for (long t = 0; t < L; ++t) {
        if (!token_visible(t, L, q_len, i, causal, shard, nshards, layout)) continue;
        const uint16_t* vr = gqa_row(v_cache, block_table, max_pages, num_pages, Hkv, D, b, kh, t);
        double p = exp(s[t] - l);
        for (int c = 0; c < D; ++c) o[c] += p * bf16_value(vr[c]);
      }
    }
    free(qv);
    free(s);
  }
  return status;
}

/* LSE merge of N shard partials.  outs: [N][rows][512], lses: [N][rows]. */
void oracle_lse_merge(const double* outs, const double* lses, int nshards, int64_t rows,
                      int dim, double* out, double* lse) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int s = 0; s < nshards; ++s) {
      double v = lses[(size_t)s * rows + r];
      if (v > M) M = v;
    }
    double* o = out + (size_t)r * dim;
    for (int c = 0; c < dim; ++c) o[c] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int s = 0; s < nshards; ++s) {
      double w = exp(lses[(size_t)s * rows + r] - M);
      wsum += w;
      const double* os = outs + ((size_t)s * rows + r) * dim;
      for (int c = 0; c < dim; ++c) o[c] += w * os[c];
    }
    for (int c = 0; c < dim; ++c) o[c] /= wsum;
    lse[r] = M + log(wsum);
  }
}

/* Per-head value up-projection: y[r] = out[r] . W_UV[head[r]]  (512 -> 128). */
void oracle_project_wuv(const double* out, const int32_t* head_of_row,
                        const uint16_t* w_uv, int64_t rows, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* w = w_uv + (size_t)head_of_row[r] * D_V * D_UV;
    const double* o = out + (size_t)r * D_V;
    double* yr = y + (size_t)r * D_UV;
    for (int j = 0; j < D_UV; ++j) {
      double acc = 0.0;
      for (int c = 0; c < D_V; ++c) acc += o[c] * bf16_value(w[(size_t)c * D_UV + j]);
      yr[j] = acc;
    }
  }
}

/* Threads the OpenMP runtime will use (reported next to CPU timings). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for later calls: n > 0 sets n, n == 0 restores the count the
 * process started with (CPU timings at 1 core and at all cores). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  extern void omp_set_num_threads(int);
  static int initial = 0;
  if (initial == 0) initial = omp_get_max_threads();
  omp_set_num_threads(n > 0 ? n : initial);
#else
  (void)n;
#endif
}
