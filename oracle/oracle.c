/*
 * CPU oracle for scaled dot-product attention and multi-head attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes, written out as the plain definition (fp64 throughout;
 * inputs are float32 values, e.g. bf16 values widened exactly):
 *
 *   "Attention Is All You Need", section 3.2.1, Eq. (1):
 *       Attention(Q, K, V) = softmax(Q K^T / sqrt(d_k)) V
 *   For one query row i: score s_j = scale * (q_i . k_j) for every key j,
 *   a softmax over j (exponentials divided by their sum), and the output row
 *   is the sum over j of the weights times the value rows v_j.
 *
 *   Section 3.2.3 (decoder self-attention): illegal connections are masked by
 *   setting their input to the softmax to -infinity, so a query at position i
 *   sees keys j <= i (its own position included).  A key-padding mask is read
 *   the same way: keys j >= len_b of batch entry b get -infinity.
 *
 *   Section 4 (restricted self-attention): each output position considers
 *   only a neighbourhood of size r of the input sequence centred on it.  Read
 *   here as keys i - floor((r-1)/2) <= j <= i + floor(r/2): exactly r
 *   positions, symmetric for odd r; it combines with the other masks.
 *
 *   Autoregressive decoding (section 3.1: the decoder generates one symbol at
 *   a time, consuming the symbols generated so far): a decoding step attends
 *   n_q new queries to the cached keys and values.  Read here as: the new
 *   queries are the last n_q positions of each sequence's cache of length
 *   len_b, so query i sits at position len_b - n_q + i and, by the causal
 *   rule, sees keys j <= len_b - n_q + i.
 *
 *   Training (section 5) needs the gradients of Eq. (1).  With P = softmax(S),
 *   S = scale * Q K^T, O = P V and an upstream gradient dO of O, the chain rule
 *   gives, per head:
 *       dV = P^T dO,   dP = dO V^T,   D_i = sum_j P_ij dP_ij (= dO_i . O_i),
 *       dS = P o (dP - D),   dQ = scale * dS K,   dK = scale * dS^T Q,
 *   the softmax Jacobian written out row by row; masked entries have P = 0.
 *   A backward routine is handed the forward output O and forms D_i from it;
 *   the oracle takes that O as an optional input for the same term.
 *
 *   Section 3.2.2, multi-head attention:
 *       MultiHead(Q, K, V) = Concat(head_1, ..., head_h) W^O,
 *       head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V),
 *   with W_i^Q, W_i^K in R^{d_model x d_k}, W_i^V in R^{d_model x d_v} and
 *   W^O in R^{h d_v x d_model}.  The per-head matrices are the column blocks of
 *   the concatenated [d_model, h*d] weights (head i = columns [i*d, (i+1)*d)),
 *   and no bias is added (none is written in the definition).
 *
 * Readings where the definition is silent (also listed in the design notes):
 *   - the softmax subtracts the row maximum before exponentiating; the
 *     softmax is shift invariant, so the value is the same and it cannot
 *     overflow;
 *   - a row whose keys are all masked has output 0 (0/0 otherwise);
 *   - the causal mask requires n_q == n_k (decoder self-attention);
 *   - padding lengths are clamped into [0, n_k].
 *
 * Parallelism: the outer loop over independent output rows is split across
 * POSIX threads; each row is computed by the same plain loops.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_MASK_NONE = 0, ORACLE_MASK_CAUSAL = 1, ORACLE_MASK_PADDING = 2 };

/* ------------------------------------------------------------------------ */
/* A plain parallel-for over [0, n): contiguous chunks, one per thread.       */
typedef void (*range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct { range_fn fn; void* ctx; int64_t begin, end; } chunk_t;

static void* run_chunk(void* p) {
  chunk_t* c = (chunk_t*)p;
  c->fn(c->ctx, c->begin, c->end);
  return NULL;
}

static void parallel_for(int64_t n, int n_threads, range_fn fn, void* ctx) {
  if (n <= 0) return;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n) n_threads = (int)n;
  if (n_threads == 1) { fn(ctx, 0, n); return; }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)n_threads);
  chunk_t* ch = (chunk_t*)malloc(sizeof(chunk_t) * (size_t)n_threads);
  int started = 0;
  for (int t = 0; t < n_threads; ++t) {
    ch[t].fn = fn; ch[t].ctx = ctx;
    ch[t].begin = n * t / n_threads;
    ch[t].end = n * (t + 1) / n_threads;
    if (pthread_create(&th[t], NULL, run_chunk, &ch[t]) != 0) {
      run_chunk(&ch[t]);  /* could not start a thread: do the chunk here */
      th[t] = (pthread_t)0;
    } else {
      ++started;
    }
  }
  for (int t = 0; t < n_threads; ++t)
    if (th[t] != (pthread_t)0) pthread_join(th[t], NULL);
  (void)started;
  free(th);
  free(ch);
}

/* ------------------------------------------------------------------------ */
/* One output row of Eq. (1): q is the query (d_k), K rows at k + j*k_stride, */
/* V rows at v + j*v_stride; keys j < len are candidates, the causal rule     */
/* (j <= i) applies when causal != 0, and keys outside [i - left, i + right] */
/* are hidden (restricted attention).  scores: scratch [n_k].                */
static void attention_row(const float* q, const float* k, const float* v, double* out,
                          int64_t k_stride, int64_t v_stride, int n_k, int d_k, int d_v,
                          int i, int causal, int len, int64_t left, int64_t right,
                          double scale, double* scores) {
  double m = -INFINITY;
  int any = 0;
  for (int j = 0; j < n_k; ++j) {
    int visible = (j < len) && !(causal && j > i) && (j >= i - left) && (j <= i + right);
    if (!visible) { scores[j] = -INFINITY; continue; }
    double dot = 0.0;
    const float* kj = k + (int64_t)j * k_stride;
    for (int c = 0; c < d_k; ++c) dot += (double)q[c] * (double)kj[c];
    scores[j] = scale * dot;
    if (scores[j] > m) m = scores[j];
    any = 1;
  }
  for (int c = 0; c < d_v; ++c) out[c] = 0.0;
  if (!any) return;               /* every key masked: output row is 0 */
  double l = 0.0;
  for (int j = 0; j < n_k; ++j) {
    double p = (scores[j] == -INFINITY) ? 0.0 : exp(scores[j] - m);
    scores[j] = p;
    l += p;
  }
  for (int j = 0; j < n_k; ++j) {
    if (scores[j] == 0.0) continue;
    double w = scores[j] / l;
    const float* vj = v + (int64_t)j * v_stride;
    for (int c = 0; c < d_v; ++c) out[c] += w * (double)vj[c];
  }
}

static int clamp_len(const int32_t* kv_lengths, int mask_kind, int bi, int n_k) {
  if (!(mask_kind & ORACLE_MASK_PADDING) || kv_lengths == NULL) return n_k;
  int len = kv_lengths[bi];
  if (len < 0) len = 0;
  if (len > n_k) len = n_k;
  return len;
}

/* ------------------------------------------------------------------------ */
/* Scaled dot-product attention over BHSD tensors.                           */
typedef struct {
  const float *q, *k, *v;
  double* out;
  int b, h, n_q, n_k, d_k, d_v, mask_kind;
  const int32_t* kv_lengths;
  double scale;
  const int64_t* rows;   /* flat row ids ((bi*h + hi)*n_q + i), or NULL = all */
  int64_t left, right;    /* restricted-attention reach (unbounded by default) */
} sdpa_ctx;

static void sdpa_range(void* p, int64_t begin, int64_t end) {
  sdpa_ctx* c = (sdpa_ctx*)p;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  for (int64_t r = begin; r < end; ++r) {
    int64_t flat = c->rows ? c->rows[r] : r;
    int i = (int)(flat % c->n_q);
    int64_t bh = flat / c->n_q;
    int bi = (int)(bh / c->h);
    const float* q = c->q + flat * c->d_k;
    const float* k = c->k + bh * (int64_t)c->n_k * c->d_k;
    const float* v = c->v + bh * (int64_t)c->n_k * c->d_v;
    int len = clamp_len(c->kv_lengths, c->mask_kind, bi, c->n_k);
    attention_row(q, k, v, c->out + r * c->d_v, c->d_k, c->d_v, c->n_k, c->d_k, c->d_v, i,
                  (c->mask_kind & ORACLE_MASK_CAUSAL) != 0, len, c->left, c->right, c->scale,
                  scores);
  }
  free(scores);
}

static int sdpa_common(const float* q, const float* k, const float* v, double* out,
                       int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                       const int32_t* kv_lengths, double scale, int64_t left, int64_t right,
                       const int64_t* rows, int64_t n_rows, int n_threads) {
  if (b < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k < 1 || d_v < 1) return -1;
  if ((mask_kind & ORACLE_MASK_CAUSAL) && n_q != n_k) return -1;
  if ((mask_kind & ORACLE_MASK_PADDING) && kv_lengths == NULL) return -1;
  sdpa_ctx c = {q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths,
                scale > 0.0 ? scale : 1.0 / sqrt((double)d_k), rows, left, right};
  int64_t n = rows ? n_rows : (int64_t)b * h * n_q;
  parallel_for(n, n_threads, sdpa_range, &c);
  return 0;
}

/*
 * Eq. (1) with masks.  q [b,h,n_q,d_k], k [b,h,n_k,d_k], v [b,h,n_k,d_v]
 * contiguous float32; kv_lengths int32 [b] (read only with the padding bit).
 * rows == NULL: out is [b,h,n_q,d_v]; else out[r] is the row rows[r].
 * scale <= 0 selects 1/sqrt(d_k).  Returns 0, or -1 on bad arguments.
 */
int oracle_sdpa(const float* q, const float* k, const float* v, double* out,
                int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                const int32_t* kv_lengths, double scale,
                const int64_t* rows, int64_t n_rows, int n_threads) {
  return sdpa_common(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths, scale,
                     INT64_MAX / 4, INT64_MAX / 4, rows, n_rows, n_threads);
}

/*
 * Restricted self-attention (section 4): as oracle_sdpa, with each query i
 * limited to the r keys i - floor((r-1)/2) .. i + floor(r/2).  r >= 1.
 */
int oracle_sdpa_restricted(const float* q, const float* k, const float* v, double* out,
                           int b, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                           const int32_t* kv_lengths, int r, double scale,
                           const int64_t* rows, int64_t n_rows, int n_threads) {
  if (r < 1) return -1;
  return sdpa_common(q, k, v, out, b, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths, scale,
                     (int64_t)((r - 1) / 2), (int64_t)(r / 2), rows, n_rows, n_threads);
}

/* ------------------------------------------------------------------------ */
/* Log of the softmax denominator of Eq. (1) for every query row:             */
/*   lse_i = ln sum_{j visible} exp(scale q_i . k_j)                          */
/* (-inf when no key is visible), taken as m + ln sum exp(s_j - m) with m the */
/* row maximum.  The visibility rule is attention_row's.  This is the value a */
/* backward pass needs to rebuild the softmax weights exp(s_ij - lse_i).      */
typedef struct {
  const float *q, *k;
  double* lse;
  int h, n_q, n_k, d_k, mask_kind;
  const int32_t* kv_lengths;
  double scale;
  int64_t left, right;
} lse_ctx;

static void lse_range(void* p, int64_t begin, int64_t end) {
  lse_ctx* c = (lse_ctx*)p;
  double* s = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  for (int64_t r = begin; r < end; ++r) {
    int i = (int)(r % c->n_q);
    int64_t bh = r / c->n_q;
    int bi = (int)(bh / c->h);
    int len = clamp_len(c->kv_lengths, c->mask_kind, bi, c->n_k);
    int causal = (c->mask_kind & ORACLE_MASK_CAUSAL) != 0;
    const float* q = c->q + r * c->d_k;
    const float* k = c->k + bh * (int64_t)c->n_k * c->d_k;
    double m = -INFINITY;
    for (int j = 0; j < c->n_k; ++j) {
      int visible = (j < len) && !(causal && j > i) && (j >= i - c->left) && (j <= i + c->right);
      s[j] = -INFINITY;
      if (!visible) continue;
      double dot = 0.0;
      for (int e = 0; e < c->d_k; ++e) dot += (double)q[e] * (double)k[(int64_t)j * c->d_k + e];
      s[j] = c->scale * dot;
      if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) { c->lse[r] = -INFINITY; continue; }
    double l = 0.0;
    for (int j = 0; j < c->n_k; ++j)
      if (s[j] != -INFINITY) l += exp(s[j] - m);
    c->lse[r] = m + log(l);
  }
  free(s);
}

/*
 * lse [b,h,n_q] of the rows of oracle_sdpa (r == 0) or oracle_sdpa_restricted
 * (r >= 1) on the same arguments.  Returns 0, or -1 on bad arguments.
 */
int oracle_sdpa_lse(const float* q, const float* k, double* lse, int b, int h, int n_q, int n_k,
                    int d_k, int mask_kind, const int32_t* kv_lengths, int r, double scale,
                    int n_threads) {
  if (b < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k < 1 || r < 0) return -1;
  if ((mask_kind & ORACLE_MASK_CAUSAL) && n_q != n_k) return -1;
  if ((mask_kind & ORACLE_MASK_PADDING) && kv_lengths == NULL) return -1;
  lse_ctx c = {q, k, lse, h, n_q, n_k, d_k, mask_kind, kv_lengths,
               scale > 0.0 ? scale : 1.0 / sqrt((double)d_k),
               r > 0 ? (int64_t)((r - 1) / 2) : INT64_MAX / 4,
               r > 0 ? (int64_t)(r / 2) : INT64_MAX / 4};
  parallel_for((int64_t)b * h * n_q, n_threads, lse_range, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Gradients of Eq. (1) for one (batch, head): plain loops over rows.         */
typedef struct {
  const float *q, *k, *v, *dout, *out;
  double *dq, *dk, *dv;
  int h, n_q, n_k, d_k, d_v, mask_kind;
  const int32_t* kv_lengths;
  double scale;
  int64_t left, right;
} bwd_ctx;

static void bwd_range(void* p, int64_t begin, int64_t end) {
  bwd_ctx* c = (bwd_ctx*)p;
  double* prow = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  double* dprow = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  for (int64_t bh = begin; bh < end; ++bh) {
    int bi = (int)(bh / c->h);
    int len = clamp_len(c->kv_lengths, c->mask_kind, bi, c->n_k);
    int causal = (c->mask_kind & ORACLE_MASK_CAUSAL) != 0;
    const float* q = c->q + bh * (int64_t)c->n_q * c->d_k;
    const float* k = c->k + bh * (int64_t)c->n_k * c->d_k;
    const float* v = c->v + bh * (int64_t)c->n_k * c->d_v;
    const float* dout = c->dout + bh * (int64_t)c->n_q * c->d_v;
    double* dq = c->dq + bh * (int64_t)c->n_q * c->d_k;
    double* dk = c->dk + bh * (int64_t)c->n_k * c->d_k;
    double* dv = c->dv + bh * (int64_t)c->n_k * c->d_v;
    for (int64_t x = 0; x < (int64_t)c->n_k * c->d_k; ++x) dk[x] = 0.0;
    for (int64_t x = 0; x < (int64_t)c->n_k * c->d_v; ++x) dv[x] = 0.0;
    for (int i = 0; i < c->n_q; ++i) {
      const float* qi = q + (int64_t)i * c->d_k;
      const float* doi = dout + (int64_t)i * c->d_v;
      double* dqi = dq + (int64_t)i * c->d_k;
      for (int x = 0; x < c->d_k; ++x) dqi[x] = 0.0;
      /* P row (softmax with the max shift; masked entries 0) */
      double m = -INFINITY;
      int any = 0;
      for (int j = 0; j < c->n_k; ++j) {
        int visible = (j < len) && !(causal && j > i) && (j >= i - c->left) && (j <= i + c->right);
        if (!visible) { prow[j] = -INFINITY; continue; }
        double dot = 0.0;
        const float* kj = k + (int64_t)j * c->d_k;
        for (int x = 0; x < c->d_k; ++x) dot += (double)qi[x] * (double)kj[x];
        prow[j] = c->scale * dot;
        if (prow[j] > m) m = prow[j];
        any = 1;
      }
      if (!any) continue;            /* no visible key: output 0, gradients 0 */
      double l = 0.0;
      for (int j = 0; j < c->n_k; ++j) {
        prow[j] = (prow[j] == -INFINITY) ? 0.0 : exp(prow[j] - m);
        l += prow[j];
      }
      for (int j = 0; j < c->n_k; ++j) prow[j] /= l;
      /* dP row = dO_i . v_j, and D_i = sum_j P_ij dP_ij */
      double Di = 0.0;
      for (int j = 0; j < c->n_k; ++j) {
        if (prow[j] == 0.0) { dprow[j] = 0.0; continue; }
        double dot = 0.0;
        const float* vj = v + (int64_t)j * c->d_v;
        for (int x = 0; x < c->d_v; ++x) dot += (double)doi[x] * (double)vj[x];
        dprow[j] = dot;
        Di += prow[j] * dot;
      }
      /* With a forward output O handed in, D_i is dO_i . O_i of that O (what
         the backward routine is given); without one, sum_j P_ij dP_ij above is
         dO_i . O_i of the exact O. */
      if (c->out != NULL) {
        const float* oi = c->out + bh * (int64_t)c->n_q * c->d_v + (int64_t)i * c->d_v;
        Di = 0.0;
        for (int x = 0; x < c->d_v; ++x) Di += (double)doi[x] * (double)oi[x];
      }
      for (int j = 0; j < c->n_k; ++j) {
        if (prow[j] == 0.0) continue;
        double ds = prow[j] * (dprow[j] - Di);
        const float* kj = k + (int64_t)j * c->d_k;
        double* dkj = dk + (int64_t)j * c->d_k;
        double* dvj = dv + (int64_t)j * c->d_v;
        for (int x = 0; x < c->d_k; ++x) {
          dqi[x] += c->scale * ds * (double)kj[x];
          dkj[x] += c->scale * ds * (double)qi[x];
        }
        for (int x = 0; x < c->d_v; ++x) dvj[x] += prow[j] * (double)doi[x];
      }
    }
  }
  free(prow);
  free(dprow);
}

/*
 * Gradients of Eq. (1) with masks: given q, k, v (BHSD float32) and dout
 * [b,h,n_q,d_v], writes dq [b,h,n_q,d_k], dk [b,h,n_k,d_k], dv [b,h,n_k,d_v]
 * (fp64).  out [b,h,n_q,d_v] is the forward output the backward is handed, or
 * NULL for the exact one: it enters only through D_i = dO_i . O_i, the row
 * term of dS = P o (dP - D).  Parallel over (batch, head).  Returns 0, or -1
 * on bad arguments.
 */
int oracle_sdpa_backward(const float* q, const float* k, const float* v, const float* dout,
                         const float* out,
                         double* dq, double* dk, double* dv, int b, int h, int n_q, int n_k,
                         int d_k, int d_v, int mask_kind, const int32_t* kv_lengths,
                         double scale, int r, int n_threads) {
  if (b < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k < 1 || d_v < 1) return -1;
  if ((mask_kind & ORACLE_MASK_CAUSAL) && n_q != n_k) return -1;
  if ((mask_kind & ORACLE_MASK_PADDING) && kv_lengths == NULL) return -1;
  bwd_ctx c = {q, k, v, dout, out, dq, dk, dv, h, n_q, n_k, d_k, d_v, mask_kind, kv_lengths,
               scale > 0.0 ? scale : 1.0 / sqrt((double)d_k),
               r > 0 ? (int64_t)((r - 1) / 2) : INT64_MAX / 4,
               r > 0 ? (int64_t)(r / 2) : INT64_MAX / 4};
  parallel_for((int64_t)b * h, n_threads, bwd_range, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* One decoding step over a key/value cache.                                  */
typedef struct {
  const float *q, *k, *v;
  double* out;
  int h, n_q, n_k, d_k, d_v;
  const int32_t* kv_lengths;
  double scale;
  const int64_t* rows;
} decode_ctx;

static void decode_range(void* p, int64_t begin, int64_t end) {
  decode_ctx* c = (decode_ctx*)p;
  double* scores = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  for (int64_t r = begin; r < end; ++r) {
    int64_t flat = c->rows ? c->rows[r] : r;
    int i = (int)(flat % c->n_q);
    int64_t bh = flat / c->n_q;
    int bi = (int)(bh / c->h);
    int len = clamp_len(c->kv_lengths, ORACLE_MASK_PADDING, bi, c->n_k);
    int pos = len - c->n_q + i;   /* position of this query in its sequence */
    const float* q = c->q + flat * c->d_k;
    const float* k = c->k + bh * (int64_t)c->n_k * c->d_k;
    const float* v = c->v + bh * (int64_t)c->n_k * c->d_v;
    if (pos < 0) {                 /* the query lies before the cache: nothing visible */
      for (int cc = 0; cc < c->d_v; ++cc) c->out[r * c->d_v + cc] = 0.0;
      continue;
    }
    attention_row(q, k, v, c->out + r * c->d_v, c->d_k, c->d_v, c->n_k, c->d_k, c->d_v, pos,
                  1, len, INT64_MAX / 4, INT64_MAX / 4, c->scale, scores);
  }
  free(scores);
}

/*
 * Decoding step: q [b,h,n_q,d_k] new queries, k [b,h,n_k,d_k] and
 * v [b,h,n_k,d_v] caches, kv_lengths int32 [b] cache lengths (NULL: all
 * n_k).  Query i sees keys j <= len_b - n_q + i.  Output as oracle_sdpa.
 */
int oracle_sdpa_decode(const float* q, const float* k, const float* v, double* out,
                       int b, int h, int n_q, int n_k, int d_k, int d_v,
                       const int32_t* kv_lengths, double scale,
                       const int64_t* rows, int64_t n_rows, int n_threads) {
  if (b < 0 || h < 0 || n_q < 1 || n_k < 0 || d_k < 1 || d_v < 1) return -1;
  int32_t* lens = NULL;
  if (kv_lengths == NULL) {
    lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(b > 0 ? b : 1));
    for (int i = 0; i < b; ++i) lens[i] = n_k;
  }
  decode_ctx c = {q, k, v, out, h, n_q, n_k, d_k, d_v, kv_lengths ? kv_lengths : lens,
                  scale > 0.0 ? scale : 1.0 / sqrt((double)d_k), rows};
  int64_t n = rows ? n_rows : (int64_t)b * h * n_q;
  parallel_for(n, n_threads, decode_range, &c);
  free(lens);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Multi-head attention (section 3.2.2).                                     */
typedef struct {
  const float *x, *w;
  double* y;       /* [n_rows, n_out] */
  int d_in, n_out;
} proj_ctx;

/* y[r, :] = x[r, :] . W   (plain row-times-matrix, fp64 sums) */
static void proj_range(void* p, int64_t begin, int64_t end) {
  proj_ctx* c = (proj_ctx*)p;
  for (int64_t r = begin; r < end; ++r) {
    double* yr = c->y + r * c->n_out;
    for (int o = 0; o < c->n_out; ++o) yr[o] = 0.0;
    const float* xr = c->x + r * c->d_in;
    for (int t = 0; t < c->d_in; ++t) {
      double xv = (double)xr[t];
      const float* wt = c->w + (int64_t)t * c->n_out;
      for (int o = 0; o < c->n_out; ++o) yr[o] += xv * (double)wt[o];
    }
  }
}

typedef struct {
  const float *xq, *wq, *wo;
  const double *kp, *vp;   /* projected keys/values of one batch entry, fp64 */
  double* y;
  int n_q, n_k, d_model, h, d_k, d_v, mask_kind, len, bi;
  double scale;
  const int64_t* rows;     /* flat ids bi*n_q + i of this batch entry */
} mha_ctx;

/* attention_row over fp64 projected K/V (same arithmetic as attention_row). */
static void attention_row_f64(const double* q, const double* k, const double* v, double* out,
                              int64_t k_stride, int64_t v_stride, int n_k, int d_k, int d_v,
                              int i, int causal, int len, double scale, double* scores) {
  double m = -INFINITY;
  int any = 0;
  for (int j = 0; j < n_k; ++j) {
    int visible = (j < len) && !(causal && j > i);
    if (!visible) { scores[j] = -INFINITY; continue; }
    double dot = 0.0;
    const double* kj = k + (int64_t)j * k_stride;
    for (int c = 0; c < d_k; ++c) dot += q[c] * kj[c];
    scores[j] = scale * dot;
    if (scores[j] > m) m = scores[j];
    any = 1;
  }
  for (int c = 0; c < d_v; ++c) out[c] = 0.0;
  if (!any) return;
  double l = 0.0;
  for (int j = 0; j < n_k; ++j) {
    double p = (scores[j] == -INFINITY) ? 0.0 : exp(scores[j] - m);
    scores[j] = p;
    l += p;
  }
  for (int j = 0; j < n_k; ++j) {
    if (scores[j] == 0.0) continue;
    double w = scores[j] / l;
    const double* vj = v + (int64_t)j * v_stride;
    for (int c = 0; c < d_v; ++c) out[c] += w * vj[c];
  }
}

static void mha_rows_range(void* p, int64_t begin, int64_t end) {
  mha_ctx* c = (mha_ctx*)p;
  int hdk = c->h * c->d_k, hdv = c->h * c->d_v;
  double* qp = (double*)malloc(sizeof(double) * (size_t)hdk);
  double* concat = (double*)malloc(sizeof(double) * (size_t)hdv);
  double* scores = (double*)malloc(sizeof(double) * (size_t)(c->n_k > 0 ? c->n_k : 1));
  for (int64_t r = begin; r < end; ++r) {
    int64_t flat = c->rows[r];
    int i = (int)(flat % c->n_q);
    /* Q row = X_q[b, i, :] W^Q (all heads) */
    const float* xr = c->xq + flat * c->d_model;
    for (int o = 0; o < hdk; ++o) qp[o] = 0.0;
    for (int t = 0; t < c->d_model; ++t) {
      double xv = (double)xr[t];
      const float* wt = c->wq + (int64_t)t * hdk;
      for (int o = 0; o < hdk; ++o) qp[o] += xv * (double)wt[o];
    }
    /* head_i = Attention on column block i; Concat in head order */
    for (int hi = 0; hi < c->h; ++hi)
      attention_row_f64(qp + hi * c->d_k, c->kp + hi * c->d_k, c->vp + hi * c->d_v,
                        concat + hi * c->d_v, hdk, hdv, c->n_k, c->d_k, c->d_v, i,
                        (c->mask_kind & ORACLE_MASK_CAUSAL) != 0, c->len, c->scale, scores);
    /* Y row = Concat W^O */
    double* yr = c->y + r * c->d_model;
    for (int o = 0; o < c->d_model; ++o) yr[o] = 0.0;
    for (int t = 0; t < hdv; ++t) {
      const float* wt = c->wo + (int64_t)t * c->d_model;
      for (int o = 0; o < c->d_model; ++o) yr[o] += concat[t] * (double)wt[o];
    }
  }
  free(qp);
  free(concat);
  free(scores);
}

/*
 * MultiHead(X_q, X_kv, X_kv) = Concat(head_1..head_h) W^O.
 * xq [b,n_q,d_model], xkv [b,n_k,d_model], wq/wk [d_model,h*d_k],
 * wv [d_model,h*d_v], wo [h*d_v,d_model], all float32 row-major.
 * rows: flat ids (bi*n_q + i) in any order, or NULL for all b*n_q rows;
 * y[r, :] receives row rows[r] (or row r).  Returns 0, or -1 on bad args.
 */
int oracle_mha(const float* xq, const float* xkv, const float* wq, const float* wk,
               const float* wv, const float* wo, double* y,
               int b, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
               int mask_kind, const int32_t* kv_lengths, double scale,
               const int64_t* rows, int64_t n_rows, int n_threads) {
  if (b < 0 || n_q < 0 || n_k < 0 || d_model < 1 || h < 1 || d_k < 1 || d_v < 1) return -1;
  if ((mask_kind & ORACLE_MASK_CAUSAL) && n_q != n_k) return -1;
  if ((mask_kind & ORACLE_MASK_PADDING) && kv_lengths == NULL) return -1;
  int64_t total = rows ? n_rows : (int64_t)b * n_q;
  int64_t* all = NULL;
  if (!rows) {
    all = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    for (int64_t r = 0; r < total; ++r) all[r] = r;
    rows = all;
  }
  int hdk = h * d_k, hdv = h * d_v;
  double* kp = (double*)malloc(sizeof(double) * (size_t)n_k * hdk + 8);
  double* vp = (double*)malloc(sizeof(double) * (size_t)n_k * hdv + 8);
  int64_t* sel = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
  int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
  double* ybuf = (double*)malloc(sizeof(double) * (size_t)(total > 0 ? total : 1) * d_model);
  double sc = scale > 0.0 ? scale : 1.0 / sqrt((double)d_k);
  for (int bi = 0; bi < b; ++bi) {
    /* rows of this batch entry */
    int64_t cnt = 0;
    for (int64_t r = 0; r < total; ++r)
      if (rows[r] / n_q == bi) { sel[cnt] = rows[r]; pos[cnt] = r; ++cnt; }
    if (cnt == 0) continue;
    /* K = X_kv W^K, V = X_kv W^V for this batch entry (fp64, no rounding) */
    proj_ctx pk = {xkv + (int64_t)bi * n_k * d_model, wk, kp, d_model, hdk};
    parallel_for(n_k, n_threads, proj_range, &pk);
    proj_ctx pv = {xkv + (int64_t)bi * n_k * d_model, wv, vp, d_model, hdv};
    parallel_for(n_k, n_threads, proj_range, &pv);
    mha_ctx c = {xq, wq, wo, kp, vp, ybuf, n_q, n_k, d_model, h, d_k, d_v, mask_kind,
                 clamp_len(kv_lengths, mask_kind, bi, n_k), bi, sc, sel};
    parallel_for(cnt, n_threads, mha_rows_range, &c);
    for (int64_t r = 0; r < cnt; ++r)
      memcpy(y + pos[r] * d_model, ybuf + r * d_model, sizeof(double) * (size_t)d_model);
  }
  free(kp); free(vp); free(sel); free(pos); free(ybuf); free(all);
  return 0;
}
