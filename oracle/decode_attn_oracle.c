/*
 * decode_attn_oracle.c -- plain, slow fp64 CPU oracle for split-KV decode
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library and includes nothing from it.
 *
 * What it computes is the plain definition of exact attention,
 *     out = softmax(q . K^T * scale) . V      ("Capstone FlashAttention", §1.1,
 *                                              standard attention formula)
 * for each request b, new token t < q_len and query head h, with the
 * key/value head kvh = h / G, G = Hq / Hkv (contiguous GQA groups: 32 query
 * heads in 8 groups, "Capstone FlashAttention", §4.2), written as the
 * three-pass safe softmax of the same page (§1.2: max, then exponent sum,
 * then division), in fp64 from the bf16 inputs:
 *     s_j  = scale * sum_d q[d] * k_j[d]
 *     m    = max_j s_j
 *     l    = sum_j exp(s_j - m)
 *     out  = sum_j exp(s_j - m) * v_j / l
 *     lse  = m + ln(l)                      (natural log, scaled scores)
 * Keys are gathered through the block table: logical token j of request b
 * lives in physical page block_table[b][j / page_size], slot j % page_size
 * (PagedAttention, "Capstone FlashAttention", §4.1).  Valid keys are
 * j < seq_lens[b]; with a causal mask among the q_len new tokens, token t
 * (which sits at position L - q_len + t) sees keys j <= L - q_len + t.  A row
 * with no valid key yields out = 0, lse = -inf.  An optional key window
 * [key_lo, key_hi) restricts every row further (used to state the partial
 * result of one KV chunk).
 *
 * oracle_merge_partials() is the cross-chunk combine written out from its
 * definition: given normalised partial outputs O_s and their log-sum-exps
 * lse_s, M = max_s lse_s, w_s = exp(lse_s - M), out = sum w_s O_s / sum w_s,
 * lse = M + ln(sum w_s) -- the two-block merge of running max / running sum
 * ("Capstone FlashAttention", §1.2 formal proof; §2.3 FlashDecoding reduce).
 *
 * FP8 caches (kv_fp8 != 0): K and V hold one byte per element in the OCP
 * FP8 E4M3 format and the keys / values are k_scale * K and v_scale * V
 * (quantisation with explicit scaling factors: "Capstone FlashAttention",
 * §2.2 FP8 with scaling; the CUTLASS split-KV post, §5.8).  The byte is
 * decoded from the format's definition (e4m3_to_double) and everything else
 * is the same definition in fp64.
 *
 * Threads split the independent (b, t, h) rows; each row is computed start to
 * finish by one thread with no reordering beyond the definition.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG -1
#define ORACLE_ERR_PAGE -2   /* block table entry outside [0, num_pages) */
#define ORACLE_ERR_RANGE -3  /* token outside the cache capacity */
#define ORACLE_ERR_NOMEM -4

static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 holds the subnormals (m/8) * 2^(1-7) = m * 2^-9; fields
 * 1..15 the normals (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10); there are no
 * infinities and S.1111.111 is NaN (so the largest value is 1.75 * 2^8 = 448). */
static double e4m3_to_double(uint8_t x) {
  const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return sign ? -v : v;
}

typedef struct {
  int batch, q_len, num_q_heads, num_kv_heads, head_dim;
  const uint16_t *q;              /* [B, q_len, Hq, D] contiguous */
  const void *k, *v;              /* caches (bf16 bits or E4M3 bytes), element strides below */
  int kv_fp8;                     /* caches hold E4M3 bytes scaled by k_scale / v_scale */
  double k_scale, v_scale;
  int64_t stride_page, stride_tok, stride_head;
  int page_size;                  /* paged: tokens per page */
  const int32_t *block_table;     /* NULL: contiguous, request b = "page" b */
  int64_t bt_stride;
  int max_pages_per_seq;
  int num_pages;
  int capacity;                   /* contiguous: tokens per request */
  const int32_t *seq_lens;
  double scale;
  int causal;
  int64_t key_lo, key_hi;         /* extra key window */
  const int32_t *rows;            /* optional list of flat row ids */
  int64_t nrows;
  double *out, *lse;              /* [nrows_total, D], [nrows_total] */
  int nthreads;
} oracle_job;

typedef struct {
  oracle_job *job;
  int tid;
  int error;
} oracle_worker;

/* Element offset of token j's key (or value) row for request b and head kvh,
 * or -1 with *err set when the block table / capacity does not cover it. */
static int64_t kv_row(const oracle_job *J, int b, int64_t j, int kvh, int *err) {
  int64_t page, slot;
  if (J->block_table) {
    int64_t col = j / J->page_size;
    if (col >= J->max_pages_per_seq) { *err = ORACLE_ERR_RANGE; return -1; }
    page = J->block_table[(int64_t)b * J->bt_stride + col];
    if (page < 0 || page >= J->num_pages) { *err = ORACLE_ERR_PAGE; return -1; }
    slot = j % J->page_size;
  } else {
    if (j >= J->capacity) { *err = ORACLE_ERR_RANGE; return -1; }
    page = b;
    slot = j;
  }
  return page * J->stride_page + slot * J->stride_tok + (int64_t)kvh * J->stride_head;
}

/* e4m3_to_double of every code, filled once (the same definition, looked up). */
static double g_e4m3[256];
static pthread_once_t g_e4m3_once = PTHREAD_ONCE_INIT;
static void fill_e4m3(void) {
  for (int c = 0; c < 256; ++c) g_e4m3[c] = e4m3_to_double((uint8_t)c);
}

/* Element `e` of a cache as a real number. */
static double kv_value(const oracle_job *J, const void *base, double scale, int64_t e) {
  if (J->kv_fp8) return scale * g_e4m3[((const uint8_t *)base)[e]];
  return bf16_to_double(((const uint16_t *)base)[e]);
}

static int one_row(const oracle_job *J, int64_t flat, double *o, double *lse_out) {
  const int D = J->head_dim;
  const int Hq = J->num_q_heads;
  const int G = J->num_q_heads / J->num_kv_heads;
  const int h = (int)(flat % Hq);
  const int t = (int)((flat / Hq) % J->q_len);
  const int b = (int)(flat / ((int64_t)Hq * J->q_len));
  const int kvh = h / G;
  const int64_t L = J->seq_lens[b];
  int64_t hi = L;
  if (J->causal) hi = L - J->q_len + 1 + t;  /* keys 0 .. L - q_len + t */
  if (hi > L) hi = L;
  if (hi > J->key_hi) hi = J->key_hi;
  int64_t lo = J->key_lo > 0 ? J->key_lo : 0;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (hi <= lo) { *lse_out = -INFINITY; return ORACLE_OK; }

  const uint16_t *qrow = J->q + (((int64_t)b * J->q_len + t) * Hq + h) * D;
  double *qd = (double *)malloc(sizeof(double) * D);
  double *s = (double *)malloc(sizeof(double) * (size_t)(hi - lo));
  if (!qd || !s) { free(qd); free(s); return ORACLE_ERR_NOMEM; }
  for (int d = 0; d < D; ++d) qd[d] = bf16_to_double(qrow[d]);

  int err = ORACLE_OK;
  /* pass 1: scores and their maximum */
  double m = -INFINITY;
  for (int64_t j = lo; j < hi; ++j) {
    const int64_t kr = kv_row(J, b, j, kvh, &err);
    if (kr < 0) { free(qd); free(s); return err; }
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qd[d] * kv_value(J, J->k, J->k_scale, kr + d);
    s[j - lo] = J->scale * acc;
    if (s[j - lo] > m) m = s[j - lo];
  }
  /* pass 2: exponent sum */
  double l = 0.0;
  for (int64_t j = lo; j < hi; ++j) l += exp(s[j - lo] - m);
  /* pass 3: normalised weights times values */
  for (int64_t j = lo; j < hi; ++j) {
    const double p = exp(s[j - lo] - m) / l;
    const int64_t vr = kv_row(J, b, j, kvh, &err);
    if (vr < 0) { free(qd); free(s); return err; }
    for (int d = 0; d < D; ++d) o[d] += p * kv_value(J, J->v, J->v_scale, vr + d);
  }
  *lse_out = m + log(l);
  free(qd);
  free(s);
  return ORACLE_OK;
}

static void *worker_main(void *arg) {
  oracle_worker *w = (oracle_worker *)arg;
  oracle_job *J = w->job;
  const int D = J->head_dim;
  for (int64_t i = w->tid; i < J->nrows; i += J->nthreads) {
    const int64_t flat = J->rows ? (int64_t)J->rows[i] : i;
    const int64_t dst = i;
    int rc = one_row(J, flat, J->out + dst * D, J->lse + dst);
    if (rc != ORACLE_OK) w->error = rc;  /* any nonzero code is reported */
  }
  return NULL;
}

/*
 * Exact decode attention in fp64.
 *   q                 bf16 bits [B, q_len, Hq, D], contiguous
 *   k, v              bf16 bits (uint16), or E4M3 bytes when kv_fp8; element
 *                     (page, slot, head, d) at
 *                     page*stride_page + slot*stride_tok + head*stride_head + d
 *   kv_fp8, k_scale, v_scale
 *                     FP8 caches: keys = k_scale * K, values = v_scale * V
 *   block_table       int32 [B, bt_stride] (first max_pages_per_seq used), or
 *                     NULL for a contiguous cache where "page" = request and
 *                     capacity = tokens per request
 *   rows / nrows      optional subset of flat rows (b*q_len + t)*Hq + h;
 *                     rows == NULL computes all B*q_len*Hq rows in order
 *   out, lse          fp64 [nrows, D], [nrows]
 * Returns 0, or a negative code when an index leaves the cache.
 */
int oracle_decode_attn(int batch, int q_len, int num_q_heads, int num_kv_heads,
                       int head_dim, const uint16_t *q, const void *k,
                       const void *v, int64_t stride_page, int64_t stride_tok,
                       int64_t stride_head, int page_size,
                       const int32_t *block_table, int64_t bt_stride,
                       int max_pages_per_seq, int num_pages, int capacity,
                       const int32_t *seq_lens, double scale, int causal,
                       int64_t key_lo, int64_t key_hi, const int32_t *rows,
                       int64_t nrows, double *out, double *lse, int nthreads,
                       int kv_fp8, double k_scale, double v_scale) {
  if (batch < 0 || q_len < 1 || num_q_heads < 1 || num_kv_heads < 1 ||
      num_q_heads % num_kv_heads != 0 || head_dim < 1 || !q || !k || !v ||
      !seq_lens || !out || !lse)
    return ORACLE_ERR_ARG;
  if (block_table && page_size < 1) return ORACLE_ERR_ARG;
  oracle_job J;
  memset(&J, 0, sizeof J);
  J.batch = batch; J.q_len = q_len; J.num_q_heads = num_q_heads;
  J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
  J.q = q; J.k = k; J.v = v;
  J.kv_fp8 = kv_fp8; J.k_scale = k_scale; J.v_scale = v_scale;
  if (kv_fp8) pthread_once(&g_e4m3_once, fill_e4m3);
  J.stride_page = stride_page; J.stride_tok = stride_tok; J.stride_head = stride_head;
  J.page_size = page_size; J.block_table = block_table; J.bt_stride = bt_stride;
  J.max_pages_per_seq = max_pages_per_seq; J.num_pages = num_pages;
  J.capacity = capacity; J.seq_lens = seq_lens; J.scale = scale; J.causal = causal;
  J.key_lo = key_lo; J.key_hi = key_hi;
  J.rows = rows;
  J.nrows = rows ? nrows : (int64_t)batch * q_len * num_q_heads;
  J.out = out; J.lse = lse;
  J.nthreads = nthreads < 1 ? 1 : nthreads;
  if (J.nthreads > J.nrows && J.nrows > 0) J.nthreads = (int)J.nrows;
  if (J.nrows == 0) return ORACLE_OK;

  if (J.nthreads == 1) {
    oracle_worker w = {&J, 0, ORACLE_OK};
    worker_main(&w);
    return w.error;
  }
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * J.nthreads);
  oracle_worker *ws = (oracle_worker *)malloc(sizeof(oracle_worker) * J.nthreads);
  if (!th || !ws) { free(th); free(ws); return ORACLE_ERR_NOMEM; }
  int started = 0;
  for (int i = 0; i < J.nthreads; ++i) {
    ws[i].job = &J;
    ws[i].tid = i;
    ws[i].error = ORACLE_OK;
    if (pthread_create(&th[i], NULL, worker_main, &ws[i]) != 0) break;
    ++started;
  }
  /* rows of threads that failed to start are computed here */
  for (int i = started; i < J.nthreads; ++i) {
    ws[i].job = &J;
    ws[i].tid = i;
    ws[i].error = ORACLE_OK;
    worker_main(&ws[i]);
  }
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  int rc = ORACLE_OK;
  for (int i = 0; i < J.nthreads; ++i)
    if (ws[i].error != ORACLE_OK) rc = ws[i].error;
  free(th);
  free(ws);
  return rc;
}

/*
 * Combine of normalised partial results (fp64).
 *   part_out [nrows, nsplit, D], part_lse [nrows, nsplit]
 *   nvalid   optional per-row count of leading splits to use (NULL: all)
 * Splits whose lse is -inf carry no weight; a row with no finite lse gives
 * out = 0, lse = -inf.
 */
int oracle_merge_partials(int64_t nrows, int nsplit, int head_dim,
                          const double *part_out, const double *part_lse,
                          const int32_t *nvalid, double *out, double *lse) {
  if (nrows < 0 || nsplit < 0 || head_dim < 1 || !out || !lse) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < nrows; ++r) {
    const int n = nvalid ? nvalid[r] : nsplit;
    const double *pl = part_lse + r * nsplit;
    const double *po = part_out + r * (int64_t)nsplit * head_dim;
    double *o = out + r * head_dim;
    double M = -INFINITY;
    for (int s = 0; s < n; ++s)
      if (pl[s] > M) M = pl[s];
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
    double W = 0.0;
    for (int s = 0; s < n; ++s) W += exp(pl[s] - M);
    for (int s = 0; s < n; ++s) {
      const double w = exp(pl[s] - M) / W;
      for (int d = 0; d < head_dim; ++d) o[d] += w * po[(int64_t)s * head_dim + d];
    }
    lse[r] = M + log(W);
  }
  return ORACLE_OK;
}

/* The oracle's E4M3 decoding of every code, for its pins. */
void oracle_e4m3_table(double *out) {
  for (int c = 0; c < 256; ++c) out[c] = e4m3_to_double((uint8_t)c);
}
