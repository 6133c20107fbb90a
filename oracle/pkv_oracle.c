/*
 * pkv_oracle.c - plain, slow, obviously correct CPU oracle for the paged
 * KV-cache attention step: store_kv, decode attention, extend (chunked
 * prefill) attention and the log-sum-exp merge of two partial states.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call this file. It shares no code,
 * header, table or constant with the CUDA library, and includes none of it.
 *
 * Arithmetic: every input is a bf16 bit pattern, widened exactly to double.
 * Dot products, exponentials, logarithms and sums are taken in double, in
 * plain loop order, with a naive two-pass softmax (max first, then sums).
 * Nothing is blocked, fused or reordered.
 *
 * Where each step comes from (page title, section):
 *  - "Code Notes: mini-sglang", Engine Layer table, BaseKVCachePool row: the
 *    KV pool is one tensor of shape
 *    (2, num_layers, num_pages, page_size, heads, head_dim), index 0 holding
 *    K and index 1 holding V, and store_kv() writes it at out_loc indices.
 *  - same page, Scheduler Layer table, TableManager row: the page_table has
 *    one row per request, mapping the request's KV cache; CacheManager row:
 *    the allocator hands out free token positions (slots).
 *  - same page, Engine Layer table, BaseAttnBackend row: prefill and decode
 *    are separate attention calls over that cache.
 *  - same page, Scheduler Layer table, PrefillManager row, and
 *    "Introduction", Key Features (Chunked Prefill): a long prompt is split
 *    into chunks, each attending over the KV of what came before it.
 *  - "Introduction", Key Features (Radix Cache): requests with a common
 *    prefix reuse its KV entries, so several page_table rows name the same
 *    slots. Nothing here needs to know; it only follows the rows.
 *
 * Readings where the pages are silent (each one is used below):
 *  R1 slot = page * page_size + offset; out_loc holds such flat slots.
 *  R2 a page_table entry for page_size P > 1 is the physical page id of the
 *     row's logical page i / P; the key sits at offset i % P of that page.
 *     For P = 1 an entry is the slot itself.
 *  R3 q head h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 *  R4 softmax scale is an argument; lse is the natural-log log-sum-exp of the
 *     scaled scores.
 *  R5 decode: the query of request b sees keys 0 .. seq_len[b]-1 of its row.
 *  R6 extend: request r's chunk has c_r = qo_indptr[r+1] - qo_indptr[r]
 *     queries and prefix length p_r = seq_len[r] - c_r; chunk query j sees
 *     keys 0 .. p_r + j (full prefix, causal within the chunk).
 *  R7 zero keys give o = 0 and lse = -inf; merging with a -inf state returns
 *     the other state, and two -inf states give o = 0, lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Error codes returned by the oracle entry points. */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

typedef struct {
  int64_t L;   /* num_layers */
  int64_t NP;  /* num_pages */
  int64_t P;   /* page_size */
  int64_t Hkv; /* kv heads */
  int64_t D;   /* head_dim */
} pool_dims;

/* bf16 -> double: a bf16 value is the top half of an IEEE binary32. */
static double widen(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Row-major position of pool[c, layer, page, off, h, d]. */
static int64_t pool_pos(pool_dims g, int64_t c, int64_t layer, int64_t page,
                        int64_t off, int64_t h, int64_t d) {
  return (((((c * g.L + layer) * g.NP + page) * g.P + off) * g.Hkv + h) * g.D) + d;
}

/* R2: logical key i of a page_table row -> (physical page, offset). */
static void locate(const int32_t *row, int64_t P, int64_t i, int64_t *page,
                   int64_t *off) {
  *page = (int64_t)row[i / P];
  *off = i % P;
}

static int dims_ok(pool_dims g, int64_t layer) {
  return g.L > 0 && g.NP > 0 && g.P > 0 && g.Hkv > 0 && g.D > 0 && layer >= 0 &&
         layer < g.L;
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * store_kv: for every new token i, copy k[i] and v[i] (Hkv x D bf16 each,
 * token rows row_stride elements apart) into pool[0|1, layer, slot] where
 * slot = out_loc[i] (R1). Bits are copied unchanged.
 */
int oracle_kv_store(uint16_t *pool, int64_t L, int64_t NP, int64_t P, int64_t Hkv,
                    int64_t D, int64_t layer, const uint16_t *k, const uint16_t *v,
                    int64_t row_stride, const int32_t *out_loc, int64_t n) {
  pool_dims g = {L, NP, P, Hkv, D};
  if (!dims_ok(g, layer) || n < 0 || row_stride < Hkv * D) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    int64_t slot = (int64_t)out_loc[i];
    if (slot < 0 || slot >= NP * P) return ORACLE_BAD_ARG;
    int64_t page = slot / P, off = slot % P;
    for (int64_t h = 0; h < Hkv; ++h) {
      for (int64_t d = 0; d < D; ++d) {
        pool[pool_pos(g, 0, layer, page, off, h, d)] = k[i * row_stride + h * D + d];
        pool[pool_pos(g, 1, layer, page, off, h, d)] = v[i * row_stride + h * D + d];
      }
    }
  }
  return ORACLE_OK;
}

/*
 * One query vector q (D bf16) against the first n keys of a page_table row,
 * on kv head kvh. s is scratch for n scores. Writes o[D] and *lse (R4, R7).
 *   s_i = scale * sum_d q[d] K[i][d]
 *   m = max_i s_i,  Z = sum_i exp(s_i - m)
 *   o[d] = sum_i exp(s_i - m) / Z * V[i][d],   lse = m + log Z
 */
static void attend(const uint16_t *pool, pool_dims g, int64_t layer, int64_t kvh,
                   const uint16_t *q, const int32_t *row, int64_t n, double scale,
                   double *s, double *o, double *lse) {
  if (n <= 0) {
    for (int64_t d = 0; d < g.D; ++d) o[d] = 0.0;
    *lse = -INFINITY;
    return;
  }
  for (int64_t i = 0; i < n; ++i) {
    int64_t page, off;
    locate(row, g.P, i, &page, &off);
    double acc = 0.0;
    for (int64_t d = 0; d < g.D; ++d)
      acc += widen(q[d]) * widen(pool[pool_pos(g, 0, layer, page, off, kvh, d)]);
    s[i] = scale * acc;
  }
  double m = s[0];
  for (int64_t i = 1; i < n; ++i)
    if (s[i] > m) m = s[i];
  double z = 0.0;
  for (int64_t i = 0; i < n; ++i) z += exp(s[i] - m);
  for (int64_t d = 0; d < g.D; ++d) o[d] = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t page, off;
    locate(row, g.P, i, &page, &off);
    double w = exp(s[i] - m) / z;
    for (int64_t d = 0; d < g.D; ++d)
      o[d] += w * widen(pool[pool_pos(g, 1, layer, page, off, kvh, d)]);
  }
  *lse = m + log(z);
}

/* Checks that keys 0..n-1 of a row resolve to slots inside the pool. */
static int row_ok(const int32_t *row, pool_dims g, int64_t n, int64_t table_stride) {
  if (n < 0) return 0;
  if (n == 0) return 1;
  if ((n - 1) / g.P >= table_stride) return 0;
  for (int64_t i = 0; i < n; i += g.P) {
    int64_t page = (int64_t)row[i / g.P];
    if (page < 0 || page >= g.NP) return 0;
  }
  return 1;
}

/*
 * Decode attention (R3, R5): for every request b and q head h,
 *   o[b,h,:], lse[b,h] = attend(q[b,h,:], row(b), seq_lens[b])
 * with row(b) = page_table + (table_idx ? table_idx[b] : b) * table_stride.
 * q is [B, Hq, D] bf16; o is [B, Hq, D] double; lse is [B, Hq] double.
 */
int oracle_decode_attn(const uint16_t *pool, int64_t L, int64_t NP, int64_t P,
                       int64_t Hkv, int64_t D, int64_t layer, const uint16_t *q,
                       const int32_t *page_table, int64_t table_stride,
                       const int32_t *table_idx, const int32_t *seq_lens, int64_t B,
                       int64_t Hq, double scale, double *o, double *lse) {
  pool_dims g = {L, NP, P, Hkv, D};
  if (!dims_ok(g, layer) || B < 0 || Hq <= 0 || Hq % Hkv != 0 || table_stride <= 0)
    return ORACLE_BAD_ARG;
  int64_t group = Hq / Hkv;
  int64_t max_n = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int32_t *row = page_table + (table_idx ? (int64_t)table_idx[b] : b) * table_stride;
    if (!row_ok(row, g, seq_lens[b], table_stride)) return ORACLE_BAD_ARG;
    if (seq_lens[b] > max_n) max_n = seq_lens[b];
  }
  int failed = 0;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * Hq; ++bh) {
      if (!s) continue;
      int64_t b = bh / Hq, h = bh % Hq;
      const int32_t *row =
          page_table + (table_idx ? (int64_t)table_idx[b] : b) * table_stride;
      attend(pool, g, layer, h / group, q + bh * D, row, seq_lens[b], scale, s,
             o + bh * D, lse + bh);
    }
    free(s);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Extend attention (R3, R6): request r owns queries qo_indptr[r] ..
 * qo_indptr[r+1]-1 (q is [T, Hq, D] bf16, T = qo_indptr[B]); query j of the
 * chunk, q head h, gives
 *   o[t,h,:], lse[t,h] = attend(q[t,h,:], row(r), p_r + j + 1).
 * o is [T, Hq, D] double; lse is [T, Hq] double.
 */
int oracle_extend_attn(const uint16_t *pool, int64_t L, int64_t NP, int64_t P,
                       int64_t Hkv, int64_t D, int64_t layer, const uint16_t *q,
                       const int32_t *qo_indptr, const int32_t *page_table,
                       int64_t table_stride, const int32_t *table_idx,
                       const int32_t *seq_lens, int64_t B, int64_t Hq, double scale,
                       double *o, double *lse) {
  pool_dims g = {L, NP, P, Hkv, D};
  if (!dims_ok(g, layer) || B < 0 || Hq <= 0 || Hq % Hkv != 0 || table_stride <= 0)
    return ORACLE_BAD_ARG;
  if (B > 0 && qo_indptr[0] != 0) return ORACLE_BAD_ARG;
  int64_t group = Hq / Hkv;
  int64_t max_n = 0;
  for (int64_t r = 0; r < B; ++r) {
    int64_t c = (int64_t)qo_indptr[r + 1] - qo_indptr[r];
    int64_t p = (int64_t)seq_lens[r] - c;
    if (c < 0 || p < 0) return ORACLE_BAD_ARG;
    const int32_t *row = page_table + (table_idx ? (int64_t)table_idx[r] : r) * table_stride;
    if (!row_ok(row, g, seq_lens[r], table_stride)) return ORACLE_BAD_ARG;
    if (seq_lens[r] > max_n) max_n = seq_lens[r];
  }
  int64_t T = B > 0 ? (int64_t)qo_indptr[B] : 0;
  int failed = 0;
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t th = 0; th < T * Hq; ++th) {
      if (!s) continue;
      int64_t t = th / Hq, h = th % Hq;
      int64_t r = 0;
      while ((int64_t)qo_indptr[r + 1] <= t) ++r; /* request owning query t */
      int64_t c = (int64_t)qo_indptr[r + 1] - qo_indptr[r];
      int64_t p = (int64_t)seq_lens[r] - c;
      int64_t j = t - qo_indptr[r];
      const int32_t *row =
          page_table + (table_idx ? (int64_t)table_idx[r] : r) * table_stride;
      attend(pool, g, layer, h / group, q + th * D, row, p + j + 1, scale, s,
             o + th * D, lse + th);
    }
    free(s);
  }
  return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Merge of two attention states over disjoint key sets (R7):
 *   lse = log(exp(lse_a) + exp(lse_b))
 *   o   = (exp(lse_a) o_a + exp(lse_b) o_b) / exp(lse)
 * evaluated relative to m = max(lse_a, lse_b). All arrays double;
 * o_* are [rows, H, D], lse_* are [rows, H].
 */
int oracle_merge_lse(const double *o_a, const double *lse_a, const double *o_b,
                     const double *lse_b, int64_t rows, int64_t H, int64_t D, double *o,
                     double *lse) {
  if (rows < 0 || H <= 0 || D <= 0) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < rows * H; ++i) {
    double la = lse_a[i], lb = lse_b[i];
    if (la == -INFINITY && lb == -INFINITY) {
      for (int64_t d = 0; d < D; ++d) o[i * D + d] = 0.0;
      lse[i] = -INFINITY;
      continue;
    }
    if (la == -INFINITY || lb == -INFINITY) { /* an empty state adds nothing */
      const double *src = la == -INFINITY ? o_b : o_a;
      for (int64_t d = 0; d < D; ++d) o[i * D + d] = src[i * D + d];
      lse[i] = la == -INFINITY ? lb : la;
      continue;
    }
    double m = la > lb ? la : lb;
    double wa = exp(la - m), wb = exp(lb - m);
    double z = wa + wb;
    for (int64_t d = 0; d < D; ++d)
      o[i * D + d] = (wa * o_a[i * D + d] + wb * o_b[i * D + d]) / z;
    lse[i] = m + log(z);
  }
  return ORACLE_OK;
}
