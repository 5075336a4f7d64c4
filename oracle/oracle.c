/*
 * fp64 CPU oracle for batched paged MLA decode.  TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the bench's CPU-baseline leg call it; the
 * CUDA library never does.  It shares no code with the CUDA path.
 *
 * What it computes is the plain definition from the FlashInfer page
 * "prims_ts_batch_decode_with_kv_cache_mla" (parameter text):
 *
 *   for request b with L = seq_lens[b], q = q_len of b, page size ps:
 *     K_b[j] = kv_cache[block_tables[b][j / ps]][j % ps][0:576]   j in [0, L)
 *     V_b[j] = K_b[j][0:512]                (one-copy cache: V = latent part)
 *   for query row i in [0, q) and head h:
 *     visible j: 0 <= j <= L - q + i        (bottom-right causal)
 *                0 <= j <  L                (dense)
 *     under decode-context parallelism (the vLLM FlashInferMLAImpl page,
 *     forward_mqa, passes cp_world, cp_rank and causal_seqlens_kv_global to
 *     the kernel): this rank r of W holds the rows g of the global sequence
 *     (length Lg) with g mod W == r as its local rows j = g div W, and the
 *     causal bound applies to global positions: local row j is visible
 *     iff j * W + r <= Lg - q + i
 *     sparse top-k (the sparse_mla_top_k argument of the trtllm-gen MLA
 *     launcher in the FlashInfer issue "Support cum_seq_lens_q in
 *     trtllm_batch_decode_with_kv_cache_mla"; the pages name the argument
 *     only): query token t carries k logical KV positions of its request;
 *     the visible rows are exactly the listed ones that fall in [0, L), as
 *     listed (a repeated position counts each time it is listed)
 *     s_j   = bmm1_scale * sum_{d < 576} Q[b,i,h,d] * K_b[j][d]
 *     lse   = m + ln(sum_j exp(s_j - m)),  m = max_j s_j      (natural log,
 *             as the vLLM FlashInferMLAImpl page states for its LSE)
 *     O[:]  = bmm2_scale * sum_j exp(s_j - lse) * V_b[j][:]
 *
 * Everything is accumulated in double.  bf16 and e4m3 inputs (the cache,
 * and the query, which is e4m3 when the caller quantised it with a q_scale
 * folded into bmm1, as the FlashInfer pull request "dynamic scale factor
 * interface and one-copy kvcache on trtllm-gen mla" describes) are decoded
 * exactly from their bit patterns (both formats are subsets of double).
 * Work is split over (query token, head) pairs with POSIX threads; each pair
 * is computed independently, so the thread count never changes a result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK_DIM 576
#define V_DIM 512

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_E4M3 = 1 };  /* also the query's element type */

/* bf16 -> double: a bf16 is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* e4m3fn -> double: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, exponent 0 is subnormal. */
static double e4m3_to_double(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xF;
  int m = bits & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);            /* m/8 * 2^(1-7) */
  else
    v = ldexp(8.0 + (double)m, e - 10);  /* (1 + m/8) * 2^(e-7) */
  return sign ? -v : v;
}

double oracle_decode_bf16(uint16_t bits) { return bf16_to_double(bits); }
double oracle_decode_e4m3(uint8_t bits) { return e4m3_to_double(bits); }

typedef struct {
  int batch, num_heads, kv_dtype, q_dtype, page_size, max_pages_per_req, causal;
  int cp_world, cp_rank;               /* decode-context parallelism (cp_world 1: off) */
  const int32_t *seq_lens_global;      /* [B] global KV lengths when cp_world > 1 */
  int sparse_k;                        /* > 0: sparse top-k positions per token */
  const int32_t *sparse_idx;           /* [tokens, sparse_k] logical KV positions */
  const void *query;         /* [tokens, H, 576] bf16 bits or e4m3 codes (q_dtype) */
  const int64_t *q_start;    /* [B + 1] token offsets */
  const void *kv_cache;      /* [num_pages, ps, 576] */
  int64_t num_pages;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  double bmm1_scale, bmm2_scale;
  int64_t n_units;           /* work units = selected (token, head) pairs */
  const int64_t *sel;        /* [n_units, 2] (token, head), or NULL for all */
  double *out;               /* [n_units, 512] */
  double *lse;               /* [n_units] */
  int64_t next;              /* shared work counter */
  pthread_mutex_t lock;
  int status;                /* 0 ok, nonzero: a page id out of range */
} job_t;

static double kv_elem(const job_t *J, int64_t page, int row, int d) {
  int64_t off = (page * J->page_size + row) * QK_DIM + d;
  if (J->kv_dtype == ORACLE_KV_BF16)
    return bf16_to_double(((const uint16_t *)J->kv_cache)[off]);
  return e4m3_to_double(((const uint8_t *)J->kv_cache)[off]);
}

/* Which request owns query token t: the b with q_start[b] <= t < q_start[b+1]. */
static int owner(const job_t *J, int64_t t) {
  int lo = 0, hi = J->batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (J->q_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/* One (token, head) pair under sparse top-k: the listed positions of token t
 * that fall in [0, L), in list order; qv holds the decoded query row. */
static int sparse_unit(job_t *J, int64_t u, int64_t t, int b, int64_t L, double *s,
                       const double *qv) {
  const int32_t *list = J->sparse_idx + t * (int64_t)J->sparse_k;
  double *o = J->out + u * V_DIM;
  double m = -INFINITY;
  int64_t n = 0;
  for (int e = 0; e < J->sparse_k; ++e) {
    const int64_t j = list[e];
    if (j < 0 || j >= L) continue;
    int64_t page = J->block_tables[(int64_t)b * J->max_pages_per_req + j / J->page_size];
    if (page < 0 || page >= J->num_pages) return 1;
    int row = (int)(j % J->page_size);
    double acc = 0.0;
    for (int d = 0; d < QK_DIM; ++d) acc += qv[d] * kv_elem(J, page, row, d);
    s[n] = J->bmm1_scale * acc;
    if (s[n] > m) m = s[n];
    ++n;
  }
  for (int d = 0; d < V_DIM; ++d) o[d] = 0.0;
  if (n == 0) {
    J->lse[u] = -INFINITY;
    return 0;
  }
  double sum = 0.0;
  for (int64_t e = 0; e < n; ++e) sum += exp(s[e] - m);
  const double lse = m + log(sum);
  J->lse[u] = lse;
  n = 0;
  for (int e = 0; e < J->sparse_k; ++e) {
    const int64_t j = list[e];
    if (j < 0 || j >= L) continue;
    int64_t page = J->block_tables[(int64_t)b * J->max_pages_per_req + j / J->page_size];
    int row = (int)(j % J->page_size);
    const double pj = exp(s[n] - lse);
    for (int d = 0; d < V_DIM; ++d) o[d] += pj * kv_elem(J, page, row, d);
    ++n;
  }
  for (int d = 0; d < V_DIM; ++d) o[d] *= J->bmm2_scale;
  return 0;
}

static int one_unit(job_t *J, int64_t u, double *s, double *qv) {
  int64_t t = J->sel ? J->sel[2 * u] : u / J->num_heads;
  int h = J->sel ? (int)J->sel[2 * u + 1] : (int)(u % J->num_heads);
  int b = owner(J, t);
  int64_t i = t - J->q_start[b];
  int64_t q = J->q_start[b + 1] - J->q_start[b];
  int64_t L = J->seq_lens[b];
  int64_t last;   /* inclusive */
  if (!J->causal) {
    last = L - 1;
  } else if (J->cp_world > 1) {
    /* local row j holds global row j * W + r; the visible ones are those
       whose global position is at most Lg - q + i (a prefix of the rows) */
    const int64_t W = J->cp_world, r = J->cp_rank, Lg = J->seq_lens_global[b];
    int64_t n_vis = 0;
    while (n_vis < L && n_vis * W + r <= Lg - q + i) ++n_vis;
    last = n_vis - 1;
  } else {
    last = L - q + i;
  }
  if (last > L - 1) last = L - 1;
  int64_t n = last + 1;
  double *o = J->out + u * V_DIM;
  for (int d = 0; d < QK_DIM; ++d) {
    const int64_t off = (t * J->num_heads + h) * QK_DIM + d;
    qv[d] = J->q_dtype == ORACLE_KV_BF16 ? bf16_to_double(((const uint16_t *)J->query)[off])
                                         : e4m3_to_double(((const uint8_t *)J->query)[off]);
  }

  if (J->sparse_k > 0) return sparse_unit(J, u, t, b, L, s, qv);
  if (n <= 0) {  /* nothing visible: empty sum (a contract violation) */
    for (int d = 0; d < V_DIM; ++d) o[d] = 0.0;
    J->lse[u] = -INFINITY;
    return 0;
  }
  /* scores */
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    int64_t page = J->block_tables[(int64_t)b * J->max_pages_per_req + j / J->page_size];
    if (page < 0 || page >= J->num_pages) return 1;
    int row = (int)(j % J->page_size);
    double acc = 0.0;
    for (int d = 0; d < QK_DIM; ++d) acc += qv[d] * kv_elem(J, page, row, d);
    s[j] = J->bmm1_scale * acc;
    if (s[j] > m) m = s[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j < n; ++j) sum += exp(s[j] - m);
  double lse = m + log(sum);
  J->lse[u] = lse;
  for (int d = 0; d < V_DIM; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    int64_t page = J->block_tables[(int64_t)b * J->max_pages_per_req + j / J->page_size];
    int row = (int)(j % J->page_size);
    double p = exp(s[j] - lse);
    for (int d = 0; d < V_DIM; ++d) o[d] += p * kv_elem(J, page, row, d);
  }
  for (int d = 0; d < V_DIM; ++d) o[d] *= J->bmm2_scale;
  return 0;
}

static void *worker(void *arg) {
  job_t *J = (job_t *)arg;
  int64_t max_L = J->sparse_k > 1 ? J->sparse_k : 1;
  for (int b = 0; b < J->batch; ++b)
    if (J->seq_lens[b] > max_L) max_L = J->seq_lens[b];
  double *s = (double *)malloc(sizeof(double) * (size_t)max_L);
  double qv[QK_DIM];
  if (!s) {
    pthread_mutex_lock(&J->lock);
    J->status = 2;
    pthread_mutex_unlock(&J->lock);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int64_t u = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (u >= J->n_units) break;
    if (one_unit(J, u, s, qv)) {
      pthread_mutex_lock(&J->lock);
      J->status = 1;
      pthread_mutex_unlock(&J->lock);
    }
  }
  free(s);
  return NULL;
}

/*
 * Compute O and LSE for the selected (token, head) pairs (all pairs when
 * sel == NULL, in [token][head] order) on rank cp_rank of cp_world
 * decode-context-parallel ranks (cp_world 1: the whole sequence is local and
 * seq_lens_global is not read).  Returns 0 on success, 1 if a page id read
 * for a visible row was out of range, 2 on allocation failure, 3 on a bad
 * rank description.
 */
int oracle_mla_decode_full(int batch, int num_heads, int kv_dtype, int q_dtype,
                           const void *query, const int64_t *q_start,
                           const void *kv_cache, int64_t num_pages, int page_size,
                           const int32_t *block_tables, int max_pages_per_req,
                           const int32_t *seq_lens, int causal,
                           double bmm1_scale, double bmm2_scale,
                           int64_t n_sel, const int64_t *sel,
                           double *out, double *lse, int n_threads,
                           int cp_world, int cp_rank, const int32_t *seq_lens_global,
                           int sparse_k, const int32_t *sparse_idx) {
  job_t J;
  if (cp_world < 1 || cp_rank < 0 || cp_rank >= cp_world ||
      (cp_world > 1 && causal && !seq_lens_global) || sparse_k < 0 ||
      (sparse_k > 0 && (!sparse_idx || cp_world > 1)))
    return 3;
  memset(&J, 0, sizeof J);
  J.batch = batch; J.num_heads = num_heads; J.kv_dtype = kv_dtype; J.q_dtype = q_dtype;
  J.page_size = page_size; J.max_pages_per_req = max_pages_per_req; J.causal = causal;
  J.cp_world = cp_world; J.cp_rank = cp_rank; J.seq_lens_global = seq_lens_global;
  J.sparse_k = sparse_k; J.sparse_idx = sparse_idx;
  J.query = query; J.q_start = q_start; J.kv_cache = kv_cache; J.num_pages = num_pages;
  J.block_tables = block_tables; J.seq_lens = seq_lens;
  J.bmm1_scale = bmm1_scale; J.bmm2_scale = bmm2_scale;
  J.sel = sel;
  J.n_units = sel ? n_sel : q_start[batch] * (int64_t)num_heads;
  J.out = out; J.lse = lse;
  pthread_mutex_init(&J.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  pthread_t th[256];
  int started = 0;
  for (int k = 0; k < n_threads; ++k)
    if (pthread_create(&th[k], NULL, worker, &J) == 0) ++started;
  if (started == 0) worker(&J);
  for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.status;
}

/* Decode-context parallelism, no sparse selection. */
int oracle_mla_decode_dcp(int batch, int num_heads, int kv_dtype, int q_dtype,
                          const void *query, const int64_t *q_start,
                          const void *kv_cache, int64_t num_pages, int page_size,
                          const int32_t *block_tables, int max_pages_per_req,
                          const int32_t *seq_lens, int causal,
                          double bmm1_scale, double bmm2_scale,
                          int64_t n_sel, const int64_t *sel,
                          double *out, double *lse, int n_threads,
                          int cp_world, int cp_rank, const int32_t *seq_lens_global) {
  return oracle_mla_decode_full(batch, num_heads, kv_dtype, q_dtype, query, q_start, kv_cache,
                                num_pages, page_size, block_tables, max_pages_per_req, seq_lens,
                                causal, bmm1_scale, bmm2_scale, n_sel, sel, out, lse, n_threads,
                                cp_world, cp_rank, seq_lens_global, 0, NULL);
}

/* The whole sequence on one rank. */
int oracle_mla_decode_q(int batch, int num_heads, int kv_dtype, int q_dtype,
                        const void *query, const int64_t *q_start,
                        const void *kv_cache, int64_t num_pages, int page_size,
                        const int32_t *block_tables, int max_pages_per_req,
                        const int32_t *seq_lens, int causal,
                        double bmm1_scale, double bmm2_scale,
                        int64_t n_sel, const int64_t *sel,
                        double *out, double *lse, int n_threads) {
  return oracle_mla_decode_dcp(batch, num_heads, kv_dtype, q_dtype, query, q_start, kv_cache,
                               num_pages, page_size, block_tables, max_pages_per_req, seq_lens,
                               causal, bmm1_scale, bmm2_scale, n_sel, sel, out, lse, n_threads,
                               1, 0, NULL);
}

/* The same with a bf16 query. */
int oracle_mla_decode(int batch, int num_heads, int kv_dtype,
                      const uint16_t *query, const int64_t *q_start,
                      const void *kv_cache, int64_t num_pages, int page_size,
                      const int32_t *block_tables, int max_pages_per_req,
                      const int32_t *seq_lens, int causal,
                      double bmm1_scale, double bmm2_scale,
                      int64_t n_sel, const int64_t *sel,
                      double *out, double *lse, int n_threads) {
  return oracle_mla_decode_q(batch, num_heads, kv_dtype, ORACLE_KV_BF16, query, q_start, kv_cache,
                             num_pages, page_size, block_tables, max_pages_per_req, seq_lens,
                             causal, bmm1_scale, bmm2_scale, n_sel, sel, out, lse, n_threads);
}
