/*
 * Exact-attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load this file's
 * library. The product path never calls it and must not fall back to it.
 *
 * What it computes is the naive pipeline of "I/O-Aware Kernels" (datasystem.school, Module 5),
 * section "Naive attention: materializing the k x k score matrix": for one query row the full
 * row of scores s_j = scale * (q . k_j) is materialised, the softmax is taken in two passes
 * (row max, then exponentials and their sum), and the normalised row multiplies V. Section
 * "FlashAttention: tiling + online softmax" of the same page states that the tiled, fused method
 * yields exactly these numbers, which is why this definition is the oracle.
 *
 * Every value is carried in fp64. Inputs arrive as bf16 bit patterns (uint16) and are widened
 * here, by this file's own conversion. Outputs are fp64: O and the natural-log LSE of the
 * scaled scores over the keys each row may attend to, and optionally, per element of O, the
 * softmax-weighted mean magnitude of V, sum_j p_j |v_jc|. That quantity is not part of the
 * method: the tests use it to bound, element by element, how far rounding the softmax weights to
 * bf16 before P.V may move O (each weight moves by at most a relative 2^-8, so O_c moves by at
 * most 2^-8 sum_j p_j |v_jc|).
 *
 * Readings where the pages are silent (each one is listed with its reason in the design notes):
 *  - causal masking is bottom-right aligned: query row i of a sequence with q_len rows and
 *    kv_len keys may attend to key j iff j <= i + (kv_len - q_len);
 *  - grouped-query heads form contiguous groups: query head h reads key/value head
 *    h / (Hq / Hkv);
 *  - a row with no key it may attend to has O = 0 and LSE = -inf;
 *  - the paged layout ("FlashInfer: I/O-aware attention for serving", same page) is first
 *    gathered into contiguous keys and values per sequence through the page table, then fed to
 *    the same row routine as the dense layout.
 *
 * Work is split over independent query rows with POSIX threads; each row is computed by the
 * same single-threaded routine, so the thread count never changes a result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> fp64 (bf16 is the top half of an IEEE binary32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * One query row against n_allowed keys (rows of K and V in fp64, row-major [n][d]).
 * s is caller scratch of at least n_allowed doubles. vabs (d doubles) may be NULL.
 */
static void attend_row(const double* q, const double* K, const double* V, long n_allowed, int d,
                       double scale, double* s, double* o, double* lse, double* vabs) {
  if (n_allowed <= 0) {
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (vabs)
      for (int c = 0; c < d; ++c) vabs[c] = 0.0;
    *lse = -INFINITY;
    return;
  }
  /* the score row S_i. = scale * q K^T, materialised in full */
  for (long j = 0; j < n_allowed; ++j) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += q[c] * K[j * d + c];
    s[j] = scale * acc;
  }
  /* softmax, pass 1: row maximum */
  double m = s[0];
  for (long j = 1; j < n_allowed; ++j)
    if (s[j] > m) m = s[j];
  /* softmax, pass 2: exponentials and their sum */
  double sum = 0.0;
  for (long j = 0; j < n_allowed; ++j) {
    s[j] = exp(s[j] - m);
    sum += s[j];
  }
  /* P V with P = exp(s - m) / sum */
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (long j = 0; j < n_allowed; ++j) {
    double p = s[j] / sum;
    for (int c = 0; c < d; ++c) o[c] += p * V[j * d + c];
  }
  *lse = m + log(sum);
  /* mean magnitude of V under the same weights */
  if (vabs) {
    for (int c = 0; c < d; ++c) vabs[c] = 0.0;
    for (long j = 0; j < n_allowed; ++j) {
      double p = s[j] / sum;
      for (int c = 0; c < d; ++c) vabs[c] += p * fabs(V[j * d + c]);
    }
  }
}

/* Number of keys query row i may attend to (bottom-right causal alignment). */
static long allowed_keys(long i, long q_len, long kv_len, int causal) {
  if (!causal) return kv_len;
  long n = i + (kv_len - q_len) + 1;
  if (n < 0) n = 0;
  if (n > kv_len) n = kv_len;
  return n;
}

/* ------------------------------ dense layout ------------------------------------------ */

typedef struct {
  const uint16_t *q, *k, *v;
  int B, Sq, Skv, Hq, Hkv, d, causal;
  double scale;
  const int64_t* rows; /* n_rows triples (b, i, h) */
  int64_t n_rows;
  double *o, *lse, *vabs;
  int64_t begin, end;
  int status;
} DenseJob;

static void* dense_worker(void* arg) {
  DenseJob* J = (DenseJob*)arg;
  const int d = J->d;
  double* qd = (double*)malloc(sizeof(double) * d);
  double* K = (double*)malloc(sizeof(double) * (size_t)J->Skv * d);
  double* V = (double*)malloc(sizeof(double) * (size_t)J->Skv * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)(J->Skv > 0 ? J->Skv : 1));
  if (!qd || !K || !V || !s) {
    J->status = 1;
    free(qd); free(K); free(V); free(s);
    return NULL;
  }
  const int group = J->Hq / J->Hkv;
  for (int64_t r = J->begin; r < J->end; ++r) {
    const int64_t b = J->rows[3 * r + 0], i = J->rows[3 * r + 1], h = J->rows[3 * r + 2];
    const int64_t hk = h / group;
    for (int c = 0; c < d; ++c) qd[c] = bf16_to_double(J->q[((b * J->Sq + i) * J->Hq + h) * d + c]);
    const long n = allowed_keys(i, J->Sq, J->Skv, J->causal);
    for (long j = 0; j < n; ++j)
      for (int c = 0; c < d; ++c) {
        const int64_t at = ((b * J->Skv + j) * J->Hkv + hk) * d + c;
        K[j * d + c] = bf16_to_double(J->k[at]);
        V[j * d + c] = bf16_to_double(J->v[at]);
      }
    attend_row(qd, K, V, n, d, J->scale, s, J->o + r * d, J->lse + r, J->vabs ? J->vabs + r * d : NULL);
  }
  free(qd); free(K); free(V); free(s);
  return NULL;
}

static int run_jobs(void* jobs, size_t job_size, int n_threads, void* (*fn)(void*)) {
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  char* joinable = (char*)calloc((size_t)n_threads, 1);
  if (!th || !joinable) {
    free(th);
    free(joinable);
    return 1;
  }
  for (int t = 0; t < n_threads; ++t) {
    void* job = (char*)jobs + job_size * (size_t)t;
    if (pthread_create(&th[t], NULL, fn, job) == 0)
      joinable[t] = 1;
    else
      fn(job); /* run inline when a thread cannot be started */
  }
  for (int t = 0; t < n_threads; ++t)
    if (joinable[t]) pthread_join(th[t], NULL);
  free(th);
  free(joinable);
  return 0;
}

/*
 * Dense attention for selected query rows.
 *   q [B, Sq, Hq, d], k and v [B, Skv, Hkv, d]: bf16 bit patterns, contiguous.
 *   rows: n_rows triples (b, i, h); o [n_rows, d] and lse [n_rows]: fp64 outputs;
 *   vabs [n_rows, d] or NULL.
 * Returns 0 on success, nonzero on bad arguments or allocation failure.
 */
int oracle_dense_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int Sq, int Skv,
                      int Hq, int Hkv, int d, int causal, double scale, const int64_t* rows,
                      int64_t n_rows, double* o, double* lse, double* vabs, int n_threads) {
  if (B <= 0 || Sq < 0 || Skv < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return 2;
  for (int64_t r = 0; r < n_rows; ++r) {
    if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= Sq ||
        rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Hq)
      return 3;
  }
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_rows) n_threads = n_rows > 0 ? (int)n_rows : 1;
  DenseJob* jobs = (DenseJob*)calloc((size_t)n_threads, sizeof(DenseJob));
  if (!jobs) return 1;
  for (int t = 0; t < n_threads; ++t) {
    DenseJob* J = &jobs[t];
    J->q = q; J->k = k; J->v = v;
    J->B = B; J->Sq = Sq; J->Skv = Skv; J->Hq = Hq; J->Hkv = Hkv; J->d = d; J->causal = causal;
    J->scale = scale; J->rows = rows; J->n_rows = n_rows; J->o = o; J->lse = lse; J->vabs = vabs;
    J->begin = n_rows * t / n_threads;
    J->end = n_rows * (t + 1) / n_threads;
  }
  int rc = run_jobs(jobs, sizeof(DenseJob), n_threads, dense_worker);
  for (int t = 0; t < n_threads; ++t) rc |= jobs[t].status;
  free(jobs);
  return rc;
}

/* ------------------------------ paged layout ------------------------------------------ */

typedef struct {
  const uint16_t *q, *k_pages, *v_pages;
  const int32_t *page_table, *cu_seqlens_q, *kv_lens;
  int page_size, num_seqs, max_pages_per_seq, num_pages, Hq, Hkv, d, causal;
  double scale;
  const int64_t* rows; /* n_rows pairs (token t, head h) */
  int64_t n_rows;
  double *o, *lse, *vabs;
  int64_t begin, end;
  int status;
} PagedJob;

/* Sequence holding packed query token t: the s with cu[s] <= t < cu[s+1]. */
static int seq_of_token(const int32_t* cu, int num_seqs, int64_t t) {
  for (int s = 0; s < num_seqs; ++s)
    if (t >= cu[s] && t < cu[s + 1]) return s;
  return -1;
}

static void* paged_worker(void* arg) {
  PagedJob* J = (PagedJob*)arg;
  const int d = J->d;
  long max_kv = 0;
  for (int s = 0; s < J->num_seqs; ++s)
    if (J->kv_lens[s] > max_kv) max_kv = J->kv_lens[s];
  double* qd = (double*)malloc(sizeof(double) * d);
  double* K = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1) * d);
  double* V = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1) * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)(max_kv > 0 ? max_kv : 1));
  if (!qd || !K || !V || !s) {
    J->status = 1;
    free(qd); free(K); free(V); free(s);
    return NULL;
  }
  const int group = J->Hq / J->Hkv;
  for (int64_t r = J->begin; r < J->end; ++r) {
    const int64_t t = J->rows[2 * r + 0], h = J->rows[2 * r + 1];
    const int sq = seq_of_token(J->cu_seqlens_q, J->num_seqs, t);
    if (sq < 0) { J->status = 3; continue; }
    const long q_len = J->cu_seqlens_q[sq + 1] - J->cu_seqlens_q[sq];
    const long kv_len = J->kv_lens[sq];
    const long i = (long)(t - J->cu_seqlens_q[sq]);
    const int64_t hk = h / group;
    for (int c = 0; c < d; ++c) qd[c] = bf16_to_double(J->q[(t * J->Hq + h) * d + c]);
    /* gather this sequence's keys and values for head hk into contiguous rows */
    const long n = allowed_keys(i, q_len, kv_len, J->causal);
    for (long j = 0; j < n; ++j) {
      const int32_t page = J->page_table[(int64_t)sq * J->max_pages_per_seq + j / J->page_size];
      const long slot = j % J->page_size;
      if (page < 0 || page >= J->num_pages) { J->status = 4; break; }
      for (int c = 0; c < d; ++c) {
        const int64_t at = (((int64_t)page * J->page_size + slot) * J->Hkv + hk) * d + c;
        K[j * d + c] = bf16_to_double(J->k_pages[at]);
        V[j * d + c] = bf16_to_double(J->v_pages[at]);
      }
    }
    attend_row(qd, K, V, n, d, J->scale, s, J->o + r * d, J->lse + r, J->vabs ? J->vabs + r * d : NULL);
  }
  free(qd); free(K); free(V); free(s);
  return NULL;
}

/*
 * Paged, ragged attention for selected (token, head) rows.
 *   q [total_q, Hq, d]; k_pages and v_pages [num_pages, page_size, Hkv, d] (bf16 bits);
 *   page_table [num_seqs, max_pages_per_seq] (int32, -1 = unused); cu_seqlens_q [num_seqs+1];
 *   kv_lens [num_seqs]; rows: n_rows pairs (t, h); o [n_rows, d], lse [n_rows] fp64;
 *   vabs [n_rows, d] or NULL.
 */
int oracle_paged_rows(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                      const int32_t* page_table, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                      int page_size, int num_seqs, int max_pages_per_seq, int num_pages, int Hq, int Hkv,
                      int d, int causal, double scale, const int64_t* rows, int64_t n_rows, double* o,
                      double* lse, double* vabs, int n_threads) {
  if (page_size <= 0 || num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0) return 2;
  for (int s = 0; s < num_seqs; ++s) {
    if (kv_lens[s] < 0 || kv_lens[s] > (int64_t)max_pages_per_seq * page_size) return 2;
    if (cu_seqlens_q[s + 1] < cu_seqlens_q[s]) return 2;
  }
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[2 * r] < 0 || rows[2 * r] >= cu_seqlens_q[num_seqs] || rows[2 * r + 1] < 0 ||
        rows[2 * r + 1] >= Hq)
      return 3;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_rows) n_threads = n_rows > 0 ? (int)n_rows : 1;
  PagedJob* jobs = (PagedJob*)calloc((size_t)n_threads, sizeof(PagedJob));
  if (!jobs) return 1;
  for (int t = 0; t < n_threads; ++t) {
    PagedJob* J = &jobs[t];
    J->q = q; J->k_pages = k_pages; J->v_pages = v_pages;
    J->page_table = page_table; J->cu_seqlens_q = cu_seqlens_q; J->kv_lens = kv_lens;
    J->page_size = page_size; J->num_seqs = num_seqs; J->max_pages_per_seq = max_pages_per_seq;
    J->num_pages = num_pages; J->Hq = Hq; J->Hkv = Hkv; J->d = d; J->causal = causal;
    J->scale = scale; J->rows = rows; J->n_rows = n_rows; J->o = o; J->lse = lse; J->vabs = vabs;
    J->begin = n_rows * t / n_threads;
    J->end = n_rows * (t + 1) / n_threads;
  }
  int rc = run_jobs(jobs, sizeof(PagedJob), n_threads, paged_worker);
  for (int t = 0; t < n_threads; ++t) rc |= jobs[t].status;
  free(jobs);
  return rc;
}
