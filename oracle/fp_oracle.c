/*
 * CPU oracle of the fused input projection — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load this file's library. The product library neither links nor calls it,
 * and the two share no code.
 *
 * It is a plain, slow, fp64 statement of the operation, one token at a time:
 *
 *  1. Gather ("Make fused_ff_qkv contiguous", Walrus PR #12, opening comment:
 *     the channels-first activation b c h w d is rearranged to b h w d c and
 *     fed to the fused linear as [tokens, C]). Token m runs row-major over all
 *     non-channel axes; the first n_batch_dims of them form the batch index b,
 *     the others the in-sequence index t, so m = b*T + t. The row X[m, :] is
 *     read through the caller's strides, one element at a time.
 *  2. Fused linear (same page, second comment: one fused_ff_qkv linear yields
 *     ff, q, k, v): Y[m, n] = sum_c X[m, c] * W[c, n], W stored [C, N]
 *     row-major, N = F + 3*C, column blocks [ff | q | k | v], inside a block
 *     column = head*head_dim + j.
 *  3. Bias, then activation ("[perf] Fused linear", xformers PR #283, PR
 *     description: the op is w x + b followed by the activation). Bias applies
 *     to every column; the activation (exact erf GELU, tanh GELU, SiLU, or the
 *     squared ReLU the same PR's thread names among activations that are slow
 *     in eager PyTorch) only to the ff block.
 *  4. Rotary embedding of q and k ("Improve performance on RoPE", nvFuser
 *     issue #1597, the rope_one_entry listing): over the first rope_n_elem
 *     lanes of a head, x1/x2 are the two halves, rotated = cat(-x2, x1), and
 *     out = x*cos + rotated*sin; lanes past rope_n_elem pass through. The page
 *     leaves cos/sin as inputs; here cos/sin of lane i and lane i + half are
 *     both those of theta_i = pos[t] * base^(-2 i / rope_n_elem).
 *  5. Split into head-major buffers ("Improve performance via batched-matmul
 *     and fused multiplies", memory-efficient-attention issue #7: the
 *     [batch*heads, tokens, head_dim] layout): ff -> [M, F] token-major,
 *     q/k/v element (b, t, head, j) -> ((b*heads + head)*T + t)*head_dim + j.
 *     Optionally k is emitted pre-transposed, [batch*heads, head_dim, tokens]
 *     (same issue, the comments on transposing the key once up front).
 *
 * Grouped-query layout (nvFuser issue #1597, split_qkv listing), selected by
 * n_query_groups > 0: the q|k|v part of a token row is [groups][q_per_kv + 2]
 * [head_dim] — q_per_kv query heads, then one key and one value head per
 * group. q is scattered to [B*heads, T, hd]; k and v stay one per group,
 * [B*groups, T, hd] (the listing's expand is a broadcast, not data).
 *
 * All arithmetic is float64 on the exactly-widened stored inputs (bf16 or
 * f32). cos/sin/erf/tanh/exp/pow come from the C library.
 *
 * Backward (oracle_backward, below): the gradients of the same operation
 * with respect to x, W and b, given upstream gradients in the output layouts.
 * The pages name the backward pass of the fused linear only as the part that
 * is left unfused and slow ("[perf] Fused linear", xformers PR #283); its
 * content is the chain rule through steps 5..1 taken in reverse:
 *  5'. gather the upstream gradient row of token m from the split buffers;
 *  4'. rotary embedding: the transpose of the rotation, per pair (i, i+half):
 *      du_i = g_i cos_i + g_{i+half} sin_{i+half},
 *      du_{i+half} = g_{i+half} cos_{i+half} - g_i sin_i; other lanes copy;
 *  3'. activation: times act'(y) at the pre-activation y = x W + b of the ff
 *      block, recomputed from the inputs (nothing is saved by the forward);
 *      bias: db = sum over tokens of G;
 *  2'. fused linear: dx[m, c] = sum_n W[c, n] G[m, n], dW = X^T G;
 *  1'. dx is returned per token, [M, C] in token order m = b*T + t.
 *
 * `mutate` != 0 plants one deliberate mistake (see the MUT_* list). Only the
 * oracle's own pin tests use it, to show that each pin catches a real error.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ACT_NONE = 0, ACT_GELU_ERF = 1, ACT_GELU_TANH = 2, ACT_SILU = 3, ACT_RELU2 = 4 };

enum {
  MUT_NONE = 0,
  MUT_DROP_BIAS = 1,         /* bias forgotten */
  MUT_ROPE_SIGN = 2,         /* rotated = cat(x2, -x1) */
  MUT_W_TRANSPOSED = 3,      /* W read as [N, C] */
  MUT_TANH_CONST = 4,        /* cubic coefficient of tanh-GELU off */
  MUT_SCATTER_ORDER = 5,     /* (head*B + b) instead of (b*heads + head) */
  MUT_ROPE_INTERLEAVED = 6,  /* pairs (2i, 2i+1) instead of (i, i+half) */
  MUT_ROPE_FREQ = 7,         /* base^(-i/n) instead of base^(-2i/n) */
  MUT_VIEW_NOT_PERMUTE = 8,  /* x read as if it were contiguous [M, C] */
  MUT_ACT_ON_Q = 9,          /* activation also on the q block */
  MUT_POS_GLOBAL = 10,       /* positions do not restart per batch element */
  MUT_ROPE_ON_V = 11,        /* v rotated too */
  MUT_QK_SWAPPED = 12,       /* q and k column blocks exchanged */
  MUT_GELU_SCALE = 13,       /* erf(y/2) instead of erf(y/sqrt 2) */
  MUT_RELU2_UNSQUARED = 14,  /* squared ReLU returned as plain ReLU */
  /* backward */
  MUT_BWD_ROPE_FORWARD = 21, /* gradient rotated by R instead of its transpose */
  MUT_BWD_ACT_VALUE = 22,    /* act(y) used where act'(y) belongs */
  MUT_BWD_NO_RECOMPUTE_BIAS = 23, /* pre-activation recomputed without the bias */
  MUT_BWD_DW_SWAP = 24,      /* dW accumulated as G^T x (rows and columns crossed) */
  MUT_BWD_DX_NO_W = 25,      /* dx from W's row sums (missing the gradient weights) */
};

typedef struct {
  const void* x;
  int x_bf16;
  int ndim;
  const int64_t* sizes;
  const int64_t* strides;
  int channel_dim;
  int n_batch_dims;
  const void* W;
  const void* bias;
  const int32_t* pos;
  const double* rope_cos;  /* [T, n_elem] or NULL */
  const double* rope_sin;
  int C, F, heads, hd, groups, rope_n_elem, act, k_transposed;
  double rope_base;
  const int64_t* rows;
  int64_t n_rows;
  double *out_ff, *out_q, *out_k, *out_v;
  int mutate;
  int64_t M, T, Bb, N;
  int64_t row_begin, row_end;
} job_t;

static double widen(const void* p, int is_bf16, int64_t i) {
  if (is_bf16) {
    uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
  }
  return (double)((const float*)p)[i];
}

/* Offset of element (m, c=0), and (b, t), for token m. */
static void locate_token(const job_t* j, int64_t m, int64_t* off, int64_t* b, int64_t* t) {
  int64_t idx[16];
  int64_t rem = m, o = 0;
  for (int a = j->ndim - 1; a >= 0; --a) {
    if (a == j->channel_dim) continue;
    idx[a] = rem % j->sizes[a];
    rem /= j->sizes[a];
    o += idx[a] * j->strides[a];
  }
  int64_t bb = 0, tt = 0;
  int seen = 0;
  for (int a = 0; a < j->ndim; ++a) {
    if (a == j->channel_dim) continue;
    if (seen < j->n_batch_dims) bb = bb * j->sizes[a] + idx[a];
    else tt = tt * j->sizes[a] + idx[a];
    ++seen;
  }
  *off = o;
  *b = bb;
  *t = tt;
}

static double activation(int act, double y, int mutate) {
  switch (act) {
    case ACT_GELU_ERF:
      if (mutate == MUT_GELU_SCALE) return 0.5 * y * (1.0 + erf(y / 2.0));
      return 0.5 * y * (1.0 + erf(y / sqrt(2.0)));
    case ACT_GELU_TANH: {
      double k3 = (mutate == MUT_TANH_CONST) ? 0.0447 : 0.044715;
      return 0.5 * y * (1.0 + tanh(sqrt(2.0 / acos(-1.0)) * (y + k3 * y * y * y)));
    }
    case ACT_SILU:
      return y / (1.0 + exp(-y));
    case ACT_RELU2:
      if (mutate == MUT_RELU2_UNSQUARED) return y > 0.0 ? y : 0.0;
      return y > 0.0 ? y * y : 0.0;
    default:
      return y;
  }
}

/* rope_one_entry on one head vector u[hd] at position p (in place). With
 * tab_cos/tab_sin (the n_elem values of the token's row of caller-given
 * [T, n_elem] tables) those are the per-lane cos/sin; otherwise both halves
 * of pair i use cos/sin of theta_i = p * base^(-2i/n_elem). */
static void rotate_half(double* u, int hd, int n_elem, double p, double base, int mutate,
                        const double* tab_cos, const double* tab_sin) {
  double xr[1024], rotated[1024], cosv[1024], sinv[1024];
  int half = n_elem / 2;
  for (int i = 0; i < n_elem; ++i) xr[i] = u[i];
  if (tab_cos) {
    for (int i = 0; i < n_elem; ++i) {
      cosv[i] = tab_cos[i];
      sinv[i] = tab_sin[i];
    }
  } else {
    for (int i = 0; i < half; ++i) {
      double e = (mutate == MUT_ROPE_FREQ) ? (double)i / n_elem : 2.0 * i / n_elem;
      double theta = p * pow(base, -e);
      cosv[i] = cosv[i + half] = cos(theta);
      sinv[i] = sinv[i + half] = sin(theta);
    }
  }
  if (mutate == MUT_ROPE_INTERLEAVED) {
    /* a plausible mix-up with the interleaved (GPT-J) convention */
    for (int i = 0; i < half; ++i) {
      double c = cosv[i], s = sinv[i];
      double a = xr[2 * i], b = xr[2 * i + 1];
      u[2 * i] = a * c - b * s;
      u[2 * i + 1] = b * c + a * s;
    }
    return;
  }
  for (int i = 0; i < half; ++i) {
    if (mutate == MUT_ROPE_SIGN) {
      rotated[i] = xr[i + half];
      rotated[i + half] = -xr[i];
    } else {
      rotated[i] = -xr[i + half];
      rotated[i + half] = xr[i];
    }
  }
  for (int i = 0; i < n_elem; ++i) u[i] = xr[i] * cosv[i] + rotated[i] * sinv[i];
  (void)hd; /* lanes n_elem..hd-1 pass through untouched */
}

static void* run_rows(void* arg) {
  const job_t* j = (const job_t*)arg;
  const int C = j->C, F = j->F, hd = j->hd, H = j->heads;
  const int G = j->groups;
  const int64_t N = j->N;
  const int elem_bf16 = j->x_bf16;
  double* X = (double*)malloc(sizeof(double) * (size_t)C);
  double* Y = (double*)malloc(sizeof(double) * (size_t)N);
  for (int64_t r = j->row_begin; r < j->row_end; ++r) {
    int64_t m = j->rows ? j->rows[r] : r;
    int64_t off, b, t;
    locate_token(j, m, &off, &b, &t);
    /* 1. gather the token's channel vector */
    for (int c = 0; c < C; ++c) {
      int64_t e = (j->mutate == MUT_VIEW_NOT_PERMUTE) ? m * C + c
                                                       : off + (int64_t)c * j->strides[j->channel_dim];
      X[c] = widen(j->x, elem_bf16, e);
    }
    /* 2. fused linear */
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int c = 0; c < C; ++c) {
        int64_t wi = (j->mutate == MUT_W_TRANSPOSED) ? (n * C + c) % (N * C) : (int64_t)c * N + n;
        acc += X[c] * widen(j->W, elem_bf16, wi);
      }
      Y[n] = acc;
    }
    /* 3. bias, activation on the ff block */
    if (j->bias && j->mutate != MUT_DROP_BIAS)
      for (int64_t n = 0; n < N; ++n) Y[n] += widen(j->bias, elem_bf16, n);
    for (int n = 0; n < F; ++n) Y[n] = activation(j->act, Y[n], j->mutate);

    /* locate the q, k, v head vectors inside the row */
    int nq = H, nkv = G ? G : H;
    int q_per_kv = G ? H / G : 1;
    double* qh[1024];
    double* kh[1024];
    double* vh[1024];
    for (int h = 0; h < nq; ++h) {
      int grp = h / q_per_kv, within = h % q_per_kv;
      qh[h] = G ? &Y[F + ((int64_t)grp * (q_per_kv + 2) + within) * hd] : &Y[F + (int64_t)h * hd];
    }
    for (int g = 0; g < nkv; ++g) {
      kh[g] = G ? &Y[F + ((int64_t)g * (q_per_kv + 2) + q_per_kv) * hd] : &Y[F + (int64_t)C + (int64_t)g * hd];
      vh[g] = G ? &Y[F + ((int64_t)g * (q_per_kv + 2) + q_per_kv + 1) * hd]
                : &Y[F + 2 * (int64_t)C + (int64_t)g * hd];
    }
    if (j->mutate == MUT_QK_SWAPPED && !G)
      for (int h = 0; h < nq; ++h) {
        double* tmp = qh[h];
        qh[h] = kh[h];
        kh[h] = tmp;
      }
    if (j->mutate == MUT_ACT_ON_Q)
      for (int h = 0; h < nq; ++h)
        for (int i = 0; i < hd; ++i) qh[h][i] = activation(ACT_SILU, qh[h][i], 0);

    /* 4. rotary embedding of q and k */
    if (j->rope_base > 0.0 && H > 0) {
      int64_t tp = (j->mutate == MUT_POS_GLOBAL) ? m : t;
      double p = j->pos ? (double)j->pos[tp % j->T] : (double)tp;
      int ne = j->rope_n_elem > 0 ? j->rope_n_elem : hd;
      const double* tc = j->rope_cos ? j->rope_cos + (tp % j->T) * ne : NULL;
      const double* ts = j->rope_sin ? j->rope_sin + (tp % j->T) * ne : NULL;
      for (int h = 0; h < nq; ++h) rotate_half(qh[h], hd, ne, p, j->rope_base, j->mutate, tc, ts);
      for (int g = 0; g < nkv; ++g) rotate_half(kh[g], hd, ne, p, j->rope_base, j->mutate, tc, ts);
      if (j->mutate == MUT_ROPE_ON_V)
        for (int g = 0; g < nkv; ++g) rotate_half(vh[g], hd, ne, p, j->rope_base, 0, tc, ts);
    }

    /* 5. split / scatter */
    if (j->rows) {
      /* sampled rows: ff [n_rows, F]; q [n_rows, heads*hd]; k, v [n_rows, nkv*hd] */
      if (F) memcpy(&j->out_ff[r * F], Y, sizeof(double) * (size_t)F);
      for (int h = 0; h < nq; ++h) memcpy(&j->out_q[(r * nq + h) * hd], qh[h], sizeof(double) * (size_t)hd);
      for (int g = 0; g < nkv; ++g) {
        memcpy(&j->out_k[(r * nkv + g) * hd], kh[g], sizeof(double) * (size_t)hd);
        memcpy(&j->out_v[(r * nkv + g) * hd], vh[g], sizeof(double) * (size_t)hd);
      }
    } else {
      if (F) memcpy(&j->out_ff[m * F], Y, sizeof(double) * (size_t)F);
      for (int h = 0; h < nq; ++h) {
        int64_t row = (j->mutate == MUT_SCATTER_ORDER) ? ((int64_t)h * j->Bb + b) : (b * nq + h);
        memcpy(&j->out_q[(row * j->T + t) * hd], qh[h], sizeof(double) * (size_t)hd);
      }
      for (int g = 0; g < nkv; ++g) {
        int64_t row = (j->mutate == MUT_SCATTER_ORDER) ? ((int64_t)g * j->Bb + b) : (b * nkv + g);
        if (j->k_transposed) /* [B*kv, hd, T]: lane-major, tokens contiguous */
          for (int i = 0; i < hd; ++i) j->out_k[(row * hd + i) * j->T + t] = kh[g][i];
        else
          memcpy(&j->out_k[(row * j->T + t) * hd], kh[g], sizeof(double) * (size_t)hd);
        memcpy(&j->out_v[(row * j->T + t) * hd], vh[g], sizeof(double) * (size_t)hd);
      }
    }
  }
  free(X);
  free(Y);
  return NULL;
}

/*
 * Entry point. Returns 0 on success, a negative number on a rejected argument.
 *
 *  x, W, bias: stored values; bf16 as uint16 bits when x_bf16, else float32.
 *    x is addressed through sizes/strides (elements). W is [C, N] row-major,
 *    N = F + 3*heads*hd (or F + (heads + 2*groups)*hd when groups > 0).
 *    bias is [N] or NULL. pos is [T] int32 or NULL (positions 0..T-1).
 *  rope_cos/rope_sin: NULL, or caller-given [T, n_rot] tables (row t is the
 *    token's cos/sin per rotated lane; pos is then unused).
 *  rows/n_rows: NULL for every token (outputs scattered to the head-major
 *    layout), else the token indices to evaluate (outputs per sampled row).
 *  n_threads: worker threads (>= 1).
 */
int oracle_forward(const void* x, int x_bf16, int ndim, const int64_t* sizes, const int64_t* strides,
                   int channel_dim, int n_batch_dims, const void* W, const void* bias, const int32_t* pos,
                   const double* rope_cos, const double* rope_sin,
                   int C, int F, int heads, int head_dim, int groups, int rope_n_elem, int act,
                   int k_transposed, double rope_base, const int64_t* rows, int64_t n_rows,
                   double* out_ff, double* out_q, double* out_k, double* out_v, int n_threads,
                   int mutate) {
  if (ndim < 1 || ndim > 16 || channel_dim < 0 || channel_dim >= ndim) return -1;
  if (sizes[channel_dim] != C || C <= 0 || F < 0 || heads < 0) return -2;
  if (heads > 0 && (head_dim <= 0 || head_dim % 2 || head_dim > 1024 || heads > 1024)) return -3;
  if (groups > 0 && (heads % groups)) return -4;
  if (!groups && heads > 0 && heads * head_dim != C) return -5;
  if (rope_n_elem < 0 || rope_n_elem > head_dim || rope_n_elem % 2) return -6;
  job_t j;
  memset(&j, 0, sizeof j);
  j.x = x;
  j.x_bf16 = x_bf16;
  j.ndim = ndim;
  j.sizes = sizes;
  j.strides = strides;
  j.channel_dim = channel_dim;
  j.n_batch_dims = n_batch_dims;
  j.W = W;
  j.bias = bias;
  j.pos = pos;
  j.rope_cos = rope_cos;
  j.rope_sin = rope_sin;
  j.C = C;
  j.F = F;
  j.heads = heads;
  j.hd = head_dim;
  j.groups = groups;
  j.rope_n_elem = rope_n_elem;
  j.act = act;
  j.k_transposed = k_transposed;
  j.rope_base = rope_base;
  j.rows = rows;
  j.out_ff = out_ff;
  j.out_q = out_q;
  j.out_k = out_k;
  j.out_v = out_v;
  j.mutate = mutate;
  int64_t Bb = 1, T = 1;
  int seen = 0;
  for (int a = 0; a < ndim; ++a) {
    if (a == channel_dim) continue;
    if (seen < n_batch_dims) Bb *= sizes[a];
    else T *= sizes[a];
    ++seen;
  }
  if (n_batch_dims < 0 || n_batch_dims > seen) return -7;
  j.Bb = Bb;
  j.T = T;
  j.M = Bb * T;
  j.N = (int64_t)F + (groups ? (int64_t)(heads + 2 * groups) * head_dim : 3 * (int64_t)heads * head_dim);
  int64_t total = rows ? n_rows : j.M;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > total) n_threads = total > 0 ? (int)total : 1;
  pthread_t th[256];
  job_t jobs[256];
  for (int i = 0; i < n_threads; ++i) {
    jobs[i] = j;
    jobs[i].row_begin = total * i / n_threads;
    jobs[i].row_end = total * (i + 1) / n_threads;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, run_rows, &jobs[i]);
  run_rows(&jobs[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
  return 0;
}


/* ------------------------------------------------------------------ backward */

/* Derivative of the ff activation at pre-activation y, in fp64. */
static double activation_deriv(int act, double y, int mutate) {
  if (mutate == MUT_BWD_ACT_VALUE) return activation(act, y, 0);
  const double pi = acos(-1.0);
  switch (act) {
    case ACT_GELU_ERF: /* d/dy [y Phi(y)] = Phi(y) + y phi(y) */
      return 0.5 * (1.0 + erf(y / sqrt(2.0))) + y * exp(-0.5 * y * y) / sqrt(2.0 * pi);
    case ACT_GELU_TANH: {
      const double k0 = sqrt(2.0 / pi), k3 = 0.044715;
      const double th = tanh(k0 * (y + k3 * y * y * y));
      return 0.5 * (1.0 + th) + 0.5 * y * (1.0 - th * th) * k0 * (1.0 + 3.0 * k3 * y * y);
    }
    case ACT_SILU: {
      const double sg = 1.0 / (1.0 + exp(-y));
      return sg * (1.0 + y * (1.0 - sg));
    }
    case ACT_RELU2:
      return y > 0.0 ? 2.0 * y : 0.0;
    default:
      return 1.0;
  }
}

typedef struct {
  job_t f;  /* the forward description (x, W, bias, pos, tables, shape) */
  const void *g_ff, *g_q, *g_k, *g_v;
  int mode; /* 0: dx of every token, dW, db; 1: dx of the sampled rows; 2: dW, db of sampled columns */
  const int64_t* cols;
  int64_t n_cols;
  double *dx, *dW, *db; /* thread-private dW/db partials in modes 0 and 2 */
} bjob_t;

/* Column n of the fused output -> block (0 ff, 1 q, 2 k, 3 v), head, lane. */
static void decode_column(const job_t* j, int64_t n, int* seg, int* head, int* lane) {
  if (n < j->F) {
    *seg = 0;
    *head = 0;
    *lane = (int)n;
    return;
  }
  int64_t w = n - j->F;
  if (j->groups) {
    int qpk = j->heads / j->groups;
    int64_t per = (int64_t)(qpk + 2) * j->hd;
    int g = (int)(w / per);
    int r = (int)(w % per), slot = r / j->hd;
    *lane = r % j->hd;
    if (slot < qpk) {
      *seg = 1;
      *head = g * qpk + slot;
    } else {
      *seg = slot == qpk ? 2 : 3;
      *head = g;
    }
    return;
  }
  *seg = 1 + (int)(w / j->C);
  int r = (int)(w % j->C);
  *head = r / j->hd;
  *lane = r % j->hd;
}

/* Upstream gradient of (block, head, lane) at token m = (b, t), widened. */
static double upstream(const bjob_t* bj, int seg, int head, int lane, int64_t m, int64_t b,
                       int64_t t) {
  const job_t* j = &bj->f;
  const int nkv = j->groups ? j->groups : j->heads;
  switch (seg) {
    case 0:
      return widen(bj->g_ff, j->x_bf16, m * j->F + lane);
    case 1:
      return widen(bj->g_q, j->x_bf16, ((b * j->heads + head) * j->T + t) * j->hd + lane);
    case 2:
      if (j->k_transposed)
        return widen(bj->g_k, j->x_bf16, ((b * nkv + head) * j->hd + lane) * j->T + t);
      return widen(bj->g_k, j->x_bf16, ((b * nkv + head) * j->T + t) * j->hd + lane);
    default:
      return widen(bj->g_v, j->x_bf16, ((b * nkv + head) * j->T + t) * j->hd + lane);
  }
}

/* cos and sin used by rotated lane `lane` at token t (forward's convention). */
static void lane_angle(const job_t* j, int lane, int64_t t, double* c, double* s) {
  int ne = j->rope_n_elem > 0 ? j->rope_n_elem : j->hd;
  int half = ne / 2;
  if (j->rope_cos) {
    *c = j->rope_cos[(t % j->T) * ne + lane];
    *s = j->rope_sin[(t % j->T) * ne + lane];
    return;
  }
  double p = j->pos ? (double)j->pos[t % j->T] : (double)t;
  double theta = p * pow(j->rope_base, -2.0 * (lane % half) / ne);
  *c = cos(theta);
  *s = sin(theta);
}

/* G[m, n]: gradient of the loss with respect to the pre-activation, pre-rotation
 * value of fused column n at token m. X is the token's gathered channel row. */
static double grad_at(const bjob_t* bj, int64_t m, int64_t b, int64_t t, int64_t n,
                      const double* X) {
  const job_t* j = &bj->f;
  int seg, head, lane;
  decode_column(j, n, &seg, &head, &lane);
  if (seg == 0) {
    double y = 0.0;
    for (int c = 0; c < j->C; ++c) y += X[c] * widen(j->W, j->x_bf16, (int64_t)c * j->N + n);
    if (j->bias && bj->f.mutate != MUT_BWD_NO_RECOMPUTE_BIAS) y += widen(j->bias, j->x_bf16, n);
    return upstream(bj, 0, 0, lane, m, b, t) * activation_deriv(j->act, y, j->mutate);
  }
  const double g = upstream(bj, seg, head, lane, m, b, t);
  const int ne = j->rope_n_elem > 0 ? j->rope_n_elem : j->hd;
  if (seg == 3 || !(j->rope_base > 0.0) || lane >= ne) return g;
  const int half = ne / 2;
  const int partner = lane < half ? lane + half : lane - half;
  const double gp = upstream(bj, seg, head, partner, m, b, t);
  double c, s, cp, sp;
  lane_angle(j, lane, t, &c, &s);
  lane_angle(j, partner, t, &cp, &sp);
  if (j->mutate == MUT_BWD_ROPE_FORWARD) /* forward rotation: x c + rotated s */
    return lane < half ? g * c - gp * s : g * c + gp * s;
  /* transpose: lane < half: g c + g' s'; lane >= half: g c - g' s' */
  return lane < half ? g * c + gp * sp : g * c - gp * sp;
}

static void* run_backward(void* arg) {
  bjob_t* bj = (bjob_t*)arg;
  const job_t* j = &bj->f;
  const int C = j->C;
  const int64_t N = j->N;
  double* X = (double*)malloc(sizeof(double) * (size_t)C);
  double* G = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  for (int64_t r = j->row_begin; r < j->row_end; ++r) {
    int64_t m = (bj->mode == 1 && j->rows) ? j->rows[r] : r;
    int64_t off, b, t;
    locate_token(j, m, &off, &b, &t);
    for (int c = 0; c < C; ++c)
      X[c] = widen(j->x, j->x_bf16, off + (int64_t)c * j->strides[j->channel_dim]);
    if (bj->mode == 2) {
      for (int64_t k = 0; k < bj->n_cols; ++k) {
        const double gv = grad_at(bj, m, b, t, bj->cols[k], X);
        bj->db[k] += gv;
        for (int c = 0; c < C; ++c) bj->dW[(int64_t)c * bj->n_cols + k] += X[c] * gv;
      }
      continue;
    }
    for (int64_t n = 0; n < N; ++n) G[n] = grad_at(bj, m, b, t, n, X);
    double* dxr = bj->dx + (bj->mode == 1 ? r : m) * C;
    for (int c = 0; c < C; ++c) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n)
        acc += (j->mutate == MUT_BWD_DX_NO_W ? 1.0 : G[n]) * widen(j->W, j->x_bf16, (int64_t)c * N + n);
      dxr[c] = acc;
    }
    if (bj->mode == 0) {
      for (int64_t n = 0; n < N; ++n) {
        bj->db[n] += G[n];
        for (int c = 0; c < C; ++c) {
          if (j->mutate == MUT_BWD_DW_SWAP) /* crossed indices, same buffer size */
            bj->dW[(n * C + c) % (N * C)] += X[c] * G[n];
          else
            bj->dW[(int64_t)c * N + n] += X[c] * G[n];
        }
      }
    }
  }
  free(X);
  free(G);
  return NULL;
}

/*
 * Backward entry point. Same shape arguments as oracle_forward, plus:
 *  g_ff, g_q, g_k, g_v: upstream gradients in the forward's output layouts
 *    (dtype of x; g_k pre-transposed when k_transposed); NULL for an empty block.
 *  mode 0: dx [M, C] (token order), dW [C, N], db [N] (db, dW zero-filled here);
 *  mode 1: dx [n_rows, C] of the tokens in rows[];
 *  mode 2: dW [C, n_cols] and db [n_cols] of the fused columns in cols[].
 * Returns 0, or a negative number on a rejected argument.
 */
int oracle_backward(const void* x, int x_bf16, int ndim, const int64_t* sizes,
                    const int64_t* strides, int channel_dim, int n_batch_dims, const void* W,
                    const void* bias, const int32_t* pos, const double* rope_cos,
                    const double* rope_sin, int C, int F, int heads, int head_dim, int groups,
                    int rope_n_elem, int act, int k_transposed, double rope_base,
                    const void* g_ff, const void* g_q, const void* g_k, const void* g_v, int mode,
                    const int64_t* rows, int64_t n_rows, const int64_t* cols, int64_t n_cols,
                    double* dx, double* dW, double* db, int n_threads, int mutate) {
  if (ndim < 1 || ndim > 16 || channel_dim < 0 || channel_dim >= ndim) return -1;
  if (sizes[channel_dim] != C || C <= 0 || F < 0 || heads < 0) return -2;
  if (heads > 0 && (head_dim <= 0 || head_dim % 2 || head_dim > 1024 || heads > 1024)) return -3;
  if (groups > 0 && (heads % groups)) return -4;
  if (!groups && heads > 0 && heads * head_dim != C) return -5;
  if (rope_n_elem < 0 || rope_n_elem > head_dim || rope_n_elem % 2) return -6;
  if (mode < 0 || mode > 2) return -8;
  bjob_t bj;
  memset(&bj, 0, sizeof bj);
  job_t* j = &bj.f;
  j->x = x;
  j->x_bf16 = x_bf16;
  j->ndim = ndim;
  j->sizes = sizes;
  j->strides = strides;
  j->channel_dim = channel_dim;
  j->n_batch_dims = n_batch_dims;
  j->W = W;
  j->bias = bias;
  j->pos = pos;
  j->rope_cos = rope_cos;
  j->rope_sin = rope_sin;
  j->C = C;
  j->F = F;
  j->heads = heads;
  j->hd = head_dim;
  j->groups = groups;
  j->rope_n_elem = rope_n_elem;
  j->act = act;
  j->k_transposed = k_transposed;
  j->rope_base = rope_base;
  j->rows = rows;
  j->mutate = mutate;
  int64_t Bb = 1, T = 1;
  int seen = 0;
  for (int a = 0; a < ndim; ++a) {
    if (a == channel_dim) continue;
    if (seen < n_batch_dims) Bb *= sizes[a];
    else T *= sizes[a];
    ++seen;
  }
  if (n_batch_dims < 0 || n_batch_dims > seen) return -7;
  j->Bb = Bb;
  j->T = T;
  j->M = Bb * T;
  j->N = (int64_t)F + (groups ? (int64_t)(heads + 2 * groups) * head_dim : 3 * (int64_t)heads * head_dim);
  bj.g_ff = g_ff;
  bj.g_q = g_q;
  bj.g_k = g_k;
  bj.g_v = g_v;
  bj.mode = mode;
  bj.cols = cols;
  bj.n_cols = n_cols;
  if (mode == 1)
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= j->M) return -9;
  if (mode == 2)
    for (int64_t k = 0; k < n_cols; ++k)
      if (cols[k] < 0 || cols[k] >= j->N) return -9;
  if ((F > 0 && !g_ff) || (heads > 0 && (!g_q || !g_k || !g_v))) return -10;
  const int64_t total = mode == 1 ? n_rows : j->M;
  const int64_t wcols = mode == 2 ? n_cols : j->N;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > total) n_threads = total > 0 ? (int)total : 1;
  pthread_t th[256];
  bjob_t* jobs = (bjob_t*)calloc((size_t)n_threads, sizeof(bjob_t));
  const int partials = mode != 1;
  for (int i = 0; i < n_threads; ++i) {
    jobs[i] = bj;
    jobs[i].f.row_begin = total * i / n_threads;
    jobs[i].f.row_end = total * (i + 1) / n_threads;
    jobs[i].dx = dx;
    if (partials) {
      jobs[i].dW = (double*)calloc((size_t)(C * wcols), sizeof(double));
      jobs[i].db = (double*)calloc((size_t)(wcols > 0 ? wcols : 1), sizeof(double));
    }
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, run_backward, &jobs[i]);
  run_backward(&jobs[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
  if (partials) {
    /* fixed summation order: thread 0, 1, ... */
    memset(dW, 0, sizeof(double) * (size_t)(C * wcols));
    memset(db, 0, sizeof(double) * (size_t)wcols);
    for (int i = 0; i < n_threads; ++i) {
      for (int64_t e = 0; e < C * wcols; ++e) dW[e] += jobs[i].dW[e];
      for (int64_t e = 0; e < wcols; ++e) db[e] += jobs[i].db[e];
      free(jobs[i].dW);
      free(jobs[i].db);
    }
  }
  free(jobs);
  return 0;
}
