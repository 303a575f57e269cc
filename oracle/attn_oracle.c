/*
 * CPU oracle of the attention that consumes the projection's q, k, v —
 * TEST INFRASTRUCTURE ONLY (same rules as fp_oracle.c: only the test-suite,
 * the smoke check and the benchmark's CPU-baseline leg load it; the product
 * library neither links nor calls it, and the two share no code).
 *
 * Source: memory-efficient-attention issue #7, "Improve performance via
 * batched-matmul and fused multiplies". The opening comment computes attention
 * with one scaled batched matmul of queries against keys (baddbmm, the scale
 * fused into the multiply), a softmax over the keys, and a second batched
 * matmul with the values (bmm), on tensors laid out [batch*heads, tokens,
 * channels_per_head]; it chunks the queries, and the keys/values, and lists
 * fast paths for when one chunk covers all queries or all keys. The later
 * comments on that page transpose the key once, up front, so k may arrive as
 * [batch*heads, channels_per_head, tokens].
 *
 * The operation, per batch*head index z, query i, channel j:
 *     out[z, i, j] = sum_t softmax_t(scale * q[z, i, :] . k[z, t, :]) v[z, t, j]
 * Readings taken where the page is silent: scale = head_dim^(-1/2) unless the
 * caller passes another (the page's baddbmm takes it as its alpha argument
 * without printing its value); the softmax runs over the keys, with no mask.
 *
 * Steps, in the page's chunked form, all in float64 on the exactly widened
 * stored inputs (bf16 or f32):
 *  1. queries in chunks of q_chunk rows (the q-chunking; one chunk when
 *     q_chunk >= the query count — the page's first fast path);
 *  2. per query chunk, keys and values in chunks of kv_chunk (one chunk when
 *     kv_chunk >= the key count — "attention slicing", the second fast path).
 *     For each kv chunk c, the scaled scores s = scale * q k_c^T, their row
 *     maximum m_c, the weights e = exp(s - m_c), the weighted values
 *     e v_c and the weight sums sum(e);
 *  3. the kv chunks are combined per query row with the largest of their
 *     maxima, M = max_c m_c: out = sum_c exp(m_c - M) (e v_c) /
 *     sum_c exp(m_c - M) sum(e). With one kv chunk this is the plain softmax.
 * The result does not depend on the chunk sizes beyond rounding: that is the
 * property the chunking relies on, and the tests pin it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const void *q, *k, *v;
  int bf16;
  int64_t BH, Tq, Tk;
  int hd, k_transposed;
  double scale;
  int64_t q_chunk, kv_chunk;
  double* out;  /* [BH, Tq, hd] */
  int mutate;
  int64_t next_job;  /* (z, query chunk) work items, taken under the lock */
  pthread_mutex_t mu;
} ajob_t;

/* planted mistakes, for the tests that check the pins catch them */
enum { AM_NONE = 0, AM_NO_MERGE_RESCALE = 1, AM_NO_SCALE = 2, AM_K_INDEX_SWAP = 3,
       AM_SOFTMAX_OVER_QUERIES = 4, AM_SUM_NOT_RESCALED = 5 };

static double aload(const void* p, int bf16, int64_t i) {
  if (bf16) {
    uint32_t b = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
  }
  return (double)((const float*)p)[i];
}

static double q_at(const ajob_t* a, int64_t z, int64_t i, int j) {
  return aload(a->q, a->bf16, (z * a->Tq + i) * a->hd + j);
}

static double k_at(const ajob_t* a, int64_t z, int64_t t, int j) {
  int transposed = a->k_transposed;
  if (a->mutate == AM_K_INDEX_SWAP) transposed = !transposed;
  if (transposed) return aload(a->k, a->bf16, (z * a->hd + j) * a->Tk + t);
  return aload(a->k, a->bf16, (z * a->Tk + t) * a->hd + j);
}

static double v_at(const ajob_t* a, int64_t z, int64_t t, int j) {
  return aload(a->v, a->bf16, (z * a->Tk + t) * a->hd + j);
}

/* One query chunk [i0, i1) of one z: steps 2 and 3. */
static void query_chunk(const ajob_t* a, int64_t z, int64_t i0, int64_t i1) {
  const int hd = a->hd;
  const double scale = a->mutate == AM_NO_SCALE ? 1.0 : a->scale;
  const int64_t nq = i1 - i0;
  const int64_t kc = a->kv_chunk;
  double* s = (double*)malloc(sizeof(double) * (size_t)(nq * kc));
  double* mx = (double*)malloc(sizeof(double) * (size_t)nq);       /* running M */
  double* den = (double*)malloc(sizeof(double) * (size_t)nq);      /* running sum */
  double* num = (double*)calloc((size_t)(nq * hd), sizeof(double)); /* running e v */
  for (int64_t r = 0; r < nq; ++r) {
    mx[r] = -INFINITY;
    den[r] = 0.0;
  }
  for (int64_t t0 = 0; t0 < a->Tk; t0 += kc) {
    const int64_t t1 = t0 + kc < a->Tk ? t0 + kc : a->Tk;
    const int64_t nk = t1 - t0;
    /* scores of this kv chunk: s = scale * q k_c^T */
    for (int64_t r = 0; r < nq; ++r)
      for (int64_t c = 0; c < nk; ++c) {
        double acc = 0.0;
        for (int j = 0; j < hd; ++j) acc += q_at(a, z, i0 + r, j) * k_at(a, z, t0 + c, j);
        s[r * kc + c] = scale * acc;
      }
    for (int64_t r = 0; r < nq; ++r) {
      /* chunk maximum m_c, weights e = exp(s - m_c), their sum and e v_c */
      double m_c = -INFINITY;
      for (int64_t c = 0; c < nk; ++c) m_c = s[r * kc + c] > m_c ? s[r * kc + c] : m_c;
      double es = 0.0;
      double ev[512];
      for (int j = 0; j < hd; ++j) ev[j] = 0.0;
      for (int64_t c = 0; c < nk; ++c) {
        const double e = exp(s[r * kc + c] - m_c);
        es += e;
        for (int j = 0; j < hd; ++j) ev[j] += e * v_at(a, z, t0 + c, j);
      }
      /* combine with the chunks before it under the larger maximum */
      const double M = mx[r] > m_c ? mx[r] : m_c;
      const double old_w = mx[r] == -INFINITY ? 0.0 : exp(mx[r] - M);
      double new_w = exp(m_c - M);
      if (a->mutate == AM_NO_MERGE_RESCALE) new_w = 1.0;
      for (int j = 0; j < hd; ++j) num[r * hd + j] = num[r * hd + j] * old_w + ev[j] * new_w;
      den[r] = den[r] * (a->mutate == AM_SUM_NOT_RESCALED ? 1.0 : old_w) + es * new_w;
      mx[r] = M;
    }
  }
  for (int64_t r = 0; r < nq; ++r)
    for (int j = 0; j < hd; ++j)
      a->out[((z * a->Tq) + i0 + r) * hd + j] = num[r * hd + j] / den[r];
  free(s);
  free(mx);
  free(den);
  free(num);
}

/* The planted mistake "softmax over the queries": normalise each key's
 * column over the queries of the whole sequence instead of each query's row
 * over the keys. */
static void wrong_axis(const ajob_t* a, int64_t z) {
  const int hd = a->hd;
  for (int64_t i = 0; i < a->Tq; ++i)
    for (int j = 0; j < hd; ++j) a->out[(z * a->Tq + i) * hd + j] = 0.0;
  double* col = (double*)malloc(sizeof(double) * (size_t)a->Tq);
  for (int64_t t = 0; t < a->Tk; ++t) {
    double m = -INFINITY, sum = 0.0;
    for (int64_t i = 0; i < a->Tq; ++i) {
      double acc = 0.0;
      for (int j = 0; j < hd; ++j) acc += q_at(a, z, i, j) * k_at(a, z, t, j);
      col[i] = a->scale * acc;
      m = col[i] > m ? col[i] : m;
    }
    for (int64_t i = 0; i < a->Tq; ++i) sum += exp(col[i] - m);
    for (int64_t i = 0; i < a->Tq; ++i)
      for (int j = 0; j < hd; ++j)
        a->out[(z * a->Tq + i) * hd + j] += exp(col[i] - m) / sum * v_at(a, z, t, j);
  }
  free(col);
}

static void* attn_worker(void* arg) {
  ajob_t* a = (ajob_t*)arg;
  const int64_t nqc = (a->Tq + a->q_chunk - 1) / a->q_chunk;
  const int64_t jobs = a->mutate == AM_SOFTMAX_OVER_QUERIES ? a->BH : a->BH * nqc;
  for (;;) {
    pthread_mutex_lock(&a->mu);
    const int64_t job = a->next_job++;
    pthread_mutex_unlock(&a->mu);
    if (job >= jobs) break;
    if (a->mutate == AM_SOFTMAX_OVER_QUERIES) {
      wrong_axis(a, job);
      continue;
    }
    const int64_t z = job / nqc, c = job % nqc;
    const int64_t i0 = c * a->q_chunk;
    const int64_t i1 = i0 + a->q_chunk < a->Tq ? i0 + a->q_chunk : a->Tq;
    query_chunk(a, z, i0, i1);
  }
  return NULL;
}

/* Returns 0, or a negative code for arguments it cannot evaluate. */
int oracle_attention(const void* q, const void* k, const void* v, int bf16, int64_t BH,
                     int64_t Tq, int64_t Tk, int hd, int k_transposed, double scale,
                     int64_t q_chunk, int64_t kv_chunk, double* out, int threads, int mutate) {
  if (BH < 0 || Tq < 0 || Tk <= 0 || hd <= 0 || hd > 512 || q_chunk <= 0 || kv_chunk <= 0)
    return -1;
  ajob_t a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.bf16 = bf16;
  a.BH = BH;
  a.Tq = Tq;
  a.Tk = Tk;
  a.hd = hd;
  a.k_transposed = k_transposed;
  a.scale = scale;
  a.q_chunk = q_chunk;
  a.kv_chunk = kv_chunk;
  a.out = out;
  a.mutate = mutate;
  a.next_job = 0;
  pthread_mutex_init(&a.mu, NULL);
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t th[256];
  for (int i = 1; i < threads; ++i) pthread_create(&th[i], NULL, attn_worker, &a);
  attn_worker(&a);
  for (int i = 1; i < threads; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&a.mu);
  return 0;
}
