/*
 * mla_oracle.c -- float64 CPU oracle for MLA speculative-verify decode.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct reference
 * that the CUDA path is checked against. Nothing in the product library links,
 * includes or calls it; only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark load it. It shares no code, header, table or constant
 * with the GPU path.
 *
 * What it computes (sglang PR #33650 "[Kimi-K3] Allow DSPARK verify on
 * cutedsl_mla (fold_sq)", "Which decode backend?" section: MQA with one latent
 * KV head, query heads H per rank, q verify tokens; the kernel name "HQk576"
 * in the GPU-timeline section gives the 576-wide key):
 *
 *   request b has ctx = seq_len_b keys (the q verify tokens included) and
 *   q = q_len_b verify tokens. Verify token i in [0, q) sees the first
 *   n_i = ctx - q + i + 1 keys (causal rule over the verify rows).
 *   Key j lives in physical cache row page_table[b][j / P] * P + j % P.
 *   Khat_j = the 576 stored values of that row (times kv_scale for an fp8
 *   e4m3 cache, times 1 for bf16). V_j = Khat_j[0:512].
 *   s_j = sm_scale * sum_{d<576} Q[b,i,h,d] * Khat_j[d]
 *   m = max_j s_j,  l = sum_j exp(s_j - m)
 *   O[b,i,h,:] = sum_j exp(s_j - m) V_j / l,   LSE = m + ln l  (natural log)
 *
 * Three evaluation orders, all float64, all reaching the same result up to
 * rounding (the pages' claim that folding only changes how often the KV cache
 * is read, not the result: PR #33650 "Why" paragraph; the split-KV partial +
 * reduction of the GPU-timeline section):
 *   MODE_DIRECT : every (i, h) row on its own, scores fully materialised.
 *   MODE_FOLDED : fold_sq -- F = largest divisor of q with H*F <= 128; the q
 *                 tokens form q/F groups of F*H packed rows; each group reads
 *                 every key once and updates all of its rows with an online
 *                 (running max) softmax, masking rows that may not see the key.
 *   MODE_SPLIT  : the key range [0, ctx) is cut at caller-given boundaries;
 *                 each chunk yields a partial (O_s, LSE_s) (a chunk a causal
 *                 row cannot see yields LSE_s = -inf, O_s = 0) and the partials
 *                 are merged: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D_QK 576
#define D_V 512

enum { MODE_DIRECT = 0, MODE_FOLDED = 1, MODE_SPLIT = 2 };
enum { KV_BF16 = 0, KV_FP8_E4M3 = 1 };

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, exponent 0 is subnormal (m/8 * 2^-6). */
double mla_oracle_e4m3_to_double(uint8_t b) {
  int sign = (b >> 7) & 1, e = (b >> 3) & 0xF, m = b & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

typedef struct {
  const uint16_t* q;            /* [total_q, H, 576] bf16 bits */
  const void* kv;               /* [rows, 576] bf16 bits or e4m3 bytes */
  int kv_dtype;
  double kv_scale;
  const int32_t* page_table;    /* [batch, pt_stride] */
  int pt_stride, page_size;
  const int32_t* seq_lens, *q_lens;
  int batch, H;
  double sm_scale;
} problem_t;

static double kv_elem(const problem_t* p, int64_t row, int d) {
  if (p->kv_dtype == KV_BF16) return bf16_to_double(((const uint16_t*)p->kv)[row * D_QK + d]);
  return p->kv_scale * mla_oracle_e4m3_to_double(((const uint8_t*)p->kv)[row * D_QK + d]);
}

static int64_t phys_row(const problem_t* p, int b, int j) {
  int page = p->page_table[(int64_t)b * p->pt_stride + j / p->page_size];
  return (int64_t)page * p->page_size + j % p->page_size;
}

/* Khat_j for key j of request b, fetched into k[576]. */
static void load_key(const problem_t* p, int b, int j, double* k) {
  int64_t r = phys_row(p, b, j);
  for (int d = 0; d < D_QK; ++d) k[d] = kv_elem(p, r, d);
}

static double dot_qk(const problem_t* p, int64_t qrow, const double* k) {
  const uint16_t* qv = p->q + qrow * D_QK;
  double s = 0.0;
  for (int d = 0; d < D_QK; ++d) s += bf16_to_double(qv[d]) * k[d];
  return s * p->sm_scale;
}

/* Softmax attention of one query row over keys [j0, j1) of request b.
 * Writes the normalised O and LSE; an empty range gives O = 0, LSE = -inf. */
static void attend_range(const problem_t* p, int b, int64_t qrow, int j0, int j1, double* o, double* lse) {
  for (int d = 0; d < D_V; ++d) o[d] = 0.0;
  if (j1 <= j0) { *lse = -INFINITY; return; }
  int n = j1 - j0;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double k[D_QK];
  double m = -INFINITY;
  for (int j = j0; j < j1; ++j) {
    load_key(p, b, j, k);
    s[j - j0] = dot_qk(p, qrow, k);
    if (s[j - j0] > m) m = s[j - j0];
  }
  double l = 0.0;
  for (int j = j0; j < j1; ++j) {
    double w = exp(s[j - j0] - m);
    l += w;
    load_key(p, b, j, k);
    for (int d = 0; d < D_V; ++d) o[d] += w * k[d];
  }
  for (int d = 0; d < D_V; ++d) o[d] /= l;
  *lse = m + log(l);
  free(s);
}

/* fold_sq factor: the largest divisor F of q with H * F <= 128 (PR #33650,
 * "Why" paragraph). H > 128 leaves no fold (F = 1). */
int mla_oracle_fold_factor(int q, int H) {
  int best = 1;
  for (int f = 1; f <= q; ++f)
    if (q % f == 0 && (int64_t)H * f <= 128) best = f;
  return best;
}

static void prefix_q(const problem_t* p, int64_t* cu) {
  cu[0] = 0;
  for (int b = 0; b < p->batch; ++b) cu[b + 1] = cu[b] + p->q_lens[b];
}

static void run_direct(const problem_t* p, const int64_t* cu, double* out, double* lse, int nthreads) {
  int64_t total_rows = cu[p->batch] * p->H;
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t r = 0; r < total_rows; ++r) {
    int64_t tok = r / p->H;
    int b = 0;
    while (cu[b + 1] <= tok) ++b;
    int i = (int)(tok - cu[b]);
    int ctx = p->seq_lens[b], q = p->q_lens[b];
    int n_i = ctx - q + i + 1;
    attend_range(p, b, r, 0, n_i, out + r * D_V, lse + r);
  }
}

/* One fold group: F tokens x H heads, every key read once, online softmax. */
static void fold_group(const problem_t* p, int b, int64_t tok0, int i0, int F, double* out, double* lse) {
  int H = p->H, R = F * H;
  int ctx = p->seq_lens[b], q = p->q_lens[b];
  double* m = (double*)malloc(sizeof(double) * R);
  double* l = (double*)malloc(sizeof(double) * R);
  double* acc = (double*)calloc((size_t)R * D_V, sizeof(double));
  double k[D_QK];
  for (int r = 0; r < R; ++r) { m[r] = -INFINITY; l[r] = 0.0; }
  for (int j = 0; j < ctx; ++j) {
    load_key(p, b, j, k);
    for (int r = 0; r < R; ++r) {
      int f = r / H;               /* packed row r = f * H + h */
      int i = i0 + f;
      if (j >= ctx - q + i + 1) continue;  /* causal mask */
      int64_t qrow = (tok0 + f) * H + (r % H);
      double s = dot_qk(p, qrow, k);
      double mn = s > m[r] ? s : m[r];
      double a = exp(m[r] - mn), w = exp(s - mn);  /* exp(-inf) = 0 on the first key */
      l[r] = l[r] * a + w;
      for (int d = 0; d < D_V; ++d) acc[(size_t)r * D_V + d] = acc[(size_t)r * D_V + d] * a + w * k[d];
      m[r] = mn;
    }
  }
  for (int r = 0; r < R; ++r) {
    int f = r / H;
    int64_t qrow = (tok0 + f) * H + (r % H);
    for (int d = 0; d < D_V; ++d) out[qrow * D_V + d] = acc[(size_t)r * D_V + d] / l[r];
    lse[qrow] = m[r] + log(l[r]);
  }
  free(m); free(l); free(acc);
}

static void run_folded(const problem_t* p, const int64_t* cu, double* out, double* lse, int nthreads) {
  /* enumerate (request, group) work items */
  int64_t n_items = 0;
  for (int b = 0; b < p->batch; ++b) n_items += p->q_lens[b] / mla_oracle_fold_factor(p->q_lens[b], p->H);
  int* ib = (int*)malloc(sizeof(int) * (n_items + 1));
  int* ig = (int*)malloc(sizeof(int) * (n_items + 1));
  int64_t t = 0;
  for (int b = 0; b < p->batch; ++b) {
    int F = mla_oracle_fold_factor(p->q_lens[b], p->H);
    for (int g = 0; g < p->q_lens[b] / F; ++g) { ib[t] = b; ig[t] = g; ++t; }
  }
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t it = 0; it < n_items; ++it) {
    int b = ib[it], g = ig[it];
    int F = mla_oracle_fold_factor(p->q_lens[b], p->H);
    fold_group(p, b, cu[b] + (int64_t)g * F, g * F, F, out, lse);
  }
  free(ib); free(ig);
}

/* bounds: CSR list per request; bounds[off[b] .. off[b+1]) are increasing key
 * positions starting at 0 and ending at ctx_b. */
static void run_split(const problem_t* p, const int64_t* cu, const int32_t* bounds, const int32_t* off,
                      double* out, double* lse, int nthreads) {
  /* partials for every (row, chunk) */
  int64_t total_chunks_rows = 0;
  int64_t* row_chunk_base = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cu[p->batch] + 1));
  for (int b = 0; b < p->batch; ++b) {
    int nch = off[b + 1] - off[b] - 1;
    for (int64_t tok = cu[b]; tok < cu[b + 1]; ++tok) {
      row_chunk_base[tok] = total_chunks_rows;
      total_chunks_rows += (int64_t)nch * p->H;
    }
  }
  double* po = (double*)malloc(sizeof(double) * (size_t)total_chunks_rows * D_V);
  double* pl = (double*)malloc(sizeof(double) * (size_t)total_chunks_rows);
  /* work items: (token, chunk) -- each computes H rows over one chunk */
  int64_t n_items = 0;
  for (int b = 0; b < p->batch; ++b) n_items += (int64_t)(off[b + 1] - off[b] - 1) * p->q_lens[b];
  (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t it = 0; it < n_items; ++it) {
    int64_t rem = it;
    int b = 0;
    while (rem >= (int64_t)(off[b + 1] - off[b] - 1) * p->q_lens[b]) { rem -= (int64_t)(off[b + 1] - off[b] - 1) * p->q_lens[b]; ++b; }
    int nch = off[b + 1] - off[b] - 1;
    int i = (int)(rem / nch), c = (int)(rem % nch);
    int ctx = p->seq_lens[b], q = p->q_lens[b];
    int n_i = ctx - q + i + 1;
    int j0 = bounds[off[b] + c], j1 = bounds[off[b] + c + 1];
    if (j1 > n_i) j1 = n_i;
    int64_t tok = cu[b] + i;
    for (int h = 0; h < p->H; ++h) {
      int64_t slot = row_chunk_base[tok] + (int64_t)c * p->H + h;
      attend_range(p, b, tok * p->H + h, j0, j1, po + slot * D_V, pl + slot);
    }
  }
  /* merge */
#pragma omp parallel for schedule(static) num_threads(nthreads)
  for (int64_t tok = 0; tok < cu[p->batch]; ++tok) {
    int b = 0;
    while (cu[b + 1] <= tok) ++b;
    int nch = off[b + 1] - off[b] - 1;
    for (int h = 0; h < p->H; ++h) {
      double mx = -INFINITY;
      for (int c = 0; c < nch; ++c) {
        double v = pl[row_chunk_base[tok] + (int64_t)c * p->H + h];
        if (v > mx) mx = v;
      }
      double sum = 0.0;
      for (int c = 0; c < nch; ++c) {
        double v = pl[row_chunk_base[tok] + (int64_t)c * p->H + h];
        if (v != -INFINITY) sum += exp(v - mx);
      }
      double L = mx + log(sum);
      double* o = out + (tok * p->H + h) * D_V;
      for (int d = 0; d < D_V; ++d) o[d] = 0.0;
      for (int c = 0; c < nch; ++c) {
        int64_t slot = row_chunk_base[tok] + (int64_t)c * p->H + h;
        if (pl[slot] == -INFINITY) continue;
        double w = exp(pl[slot] - L);
        for (int d = 0; d < D_V; ++d) o[d] += w * po[slot * D_V + d];
      }
      lse[tok * p->H + h] = L;
    }
  }
  free(po); free(pl); free(row_chunk_base);
}

/* Entry point. Returns 0 on success, a negative value on bad arguments. */
int mla_oracle_decode(const uint16_t* q, const void* kv, int kv_dtype, double kv_scale,
                      const int32_t* page_table, int pt_stride, int page_size,
                      const int32_t* seq_lens, const int32_t* q_lens, int batch, int H,
                      double sm_scale, int mode, const int32_t* split_bounds, const int32_t* split_off,
                      double* out, double* lse, int nthreads) {
  if (!q || !kv || !page_table || !seq_lens || !q_lens || !out || !lse) return -1;
  if (batch < 0 || H < 1 || page_size < 1) return -1;
  if (kv_dtype != KV_BF16 && kv_dtype != KV_FP8_E4M3) return -1;
  for (int b = 0; b < batch; ++b) {
    if (q_lens[b] < 1 || seq_lens[b] < q_lens[b]) return -2;
    if ((seq_lens[b] + page_size - 1) / page_size > pt_stride) return -2;
  }
  if (mode == MODE_SPLIT) {
    if (!split_bounds || !split_off) return -1;
    for (int b = 0; b < batch; ++b) {
      int n = split_off[b + 1] - split_off[b];
      if (n < 2 || split_bounds[split_off[b]] != 0 || split_bounds[split_off[b + 1] - 1] != seq_lens[b]) return -3;
      for (int c = split_off[b]; c + 1 < split_off[b + 1]; ++c)
        if (split_bounds[c + 1] < split_bounds[c]) return -3;
    }
  }
  if (nthreads < 1) nthreads = 1;
  problem_t p = {q, kv, kv_dtype, kv_scale, page_table, pt_stride, page_size, seq_lens, q_lens, batch, H, sm_scale};
  int64_t* cu = (int64_t*)malloc(sizeof(int64_t) * (size_t)(batch + 1));
  prefix_q(&p, cu);
  if (mode == MODE_DIRECT) run_direct(&p, cu, out, lse, nthreads);
  else if (mode == MODE_FOLDED) run_folded(&p, cu, out, lse, nthreads);
  else if (mode == MODE_SPLIT) run_split(&p, cu, split_bounds, split_off, out, lse, nthreads);
  else { free(cu); return -1; }
  free(cu);
  return 0;
}
