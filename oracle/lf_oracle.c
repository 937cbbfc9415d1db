/*
 * lf_oracle.c -- plain, slow fp64 CPU oracle for Longformer-style attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link or call
 * this file; only the tests, the package's smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or constant with
 * the CUDA library.
 *
 * What it computes (velog.io/@lainshower/Longformer, section 3-1 "Attention
 * Pattern"):
 *   - Sliding window: a token attends w/2 neighbours on each side of itself.
 *     Read here as |i - j| <= w/2 with the token itself included, so an
 *     interior row attends w + 1 keys.
 *   - Dilated sliding window: the window keeps its number of cells and
 *     leaves gaps between them.  Read here as offsets that are multiples of
 *     the head's dilation delta, up to delta * w/2 on each side.
 *   - Global attention: the chosen tokens attend to every token and every
 *     token attends to them; a global key that already lies in a row's band
 *     is counted once (the attended set is a set union).
 *   - Linear projections for global attention: the global computation uses
 *     its own Q/K/V projections.  Read here as: rows of global tokens score
 *     qg against kg of all valid keys and average vg; every other row uses
 *     q, k and v for both its band and the global columns.
 * The autoregressive variant (section 4.1) is read as the same window with
 * its forward half removed: keys i - delta*t for t = 0..w/2.  Causality also
 * restricts global rows (keys j <= g) and global columns (g <= i).
 * Padding: pad_len[b] trailing tokens of batch row b are padding; they are
 * never attended and their output rows are exact zeros.
 * Scale 1/sqrt(d); no dropout.  An optional relative position bias is added
 * to the band keys' scores (band_bias below).
 *
 * Everything is evaluated in double: for each row the attended set is
 * enumerated, scores are computed with a plain dot product, the row maximum
 * is subtracted, exp() from libm is applied and the weighted values are
 * summed and divided by the weight total.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type of the input tensors */
enum { ORC_F64 = 0, ORC_F32 = 1, ORC_BF16 = 2 };

static double load_elem(int dtype, const void* base, int64_t idx) {
  if (dtype == ORC_F64) return ((const double*)base)[idx];
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  /* bf16: the upper 16 bits of an IEEE binary32 */
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

typedef struct {
  int dtype;
  const void *q, *k, *v, *qg, *kg, *vg;
  const int32_t* global_idx;
  int32_t G, B, H, n, d, w, causal;
  const int32_t* dilation;
  const int32_t* pad_len;
  const int32_t* w_heads; /* window of each head, or NULL: w for every head */
  const float* rel_bias;  /* [H, w + 1] relative position bias of the band keys, or NULL */
} problem;

/* The window of head h (section 4.1 "Attention Pattern": window sizes differ
 * between layers, and heads within a layer differ in their pattern). */
static int64_t window_of(const problem* p, int32_t h) {
  return p->w_heads ? p->w_heads[h] : p->w;
}

/* rank of position i in the sorted global list, or -1 if i is not global */
static int global_rank(const problem* p, int32_t i) {
  for (int32_t r = 0; r < p->G; ++r)
    if (p->global_idx[r] == i) return r;
  return -1;
}

/* Is key j inside row i's (dilated, possibly causal) window? */
static int in_window(const problem* p, int32_t h, int32_t i, int32_t j) {
  int64_t delta = p->dilation[h];
  int64_t half = window_of(p, h) / 2;
  int64_t off = (int64_t)j - (int64_t)i;           /* key offset from the row */
  if (off % delta != 0) return 0;                  /* dilation gaps */
  int64_t steps = off / delta;
  int64_t left = half;                             /* look-back reach in steps */
  int64_t right = p->causal ? 0 : half;            /* look-ahead reach in steps */
  return steps >= -left && steps <= right;
}

/*
 * The relative position bias of key j in row i's band (Memorizing
 * Transformer notes, "Position bias": a T5-style bias added to the attention
 * scores, a learned scalar per head and relative position).  Read here as
 * rel_bias[h][t + w/2] added to the scaled score of the band key at window
 * step t = (j - i) / delta, t in [-w/2, w/2]; the caller expands any bucketing
 * of relative positions into that table.  Global columns outside the band
 * and the global tokens' own rows get no bias.
 */
static double band_bias(const problem* p, int32_t h, int32_t i, int32_t j) {
  if (!p->rel_bias || !in_window(p, h, i, j)) return 0.0;
  int64_t t = ((int64_t)j - (int64_t)i) / p->dilation[h];
  return (double)p->rel_bias[(int64_t)h * (p->w + 1) + t + p->w / 2];
}

/*
 * Enumerate the attended key set of row (b, h, i).  Writes the key indices
 * to keys[] (capacity n) and returns their count.  *is_global_row is set when
 * the row belongs to a global token (its keys then index kg/vg).
 * Returns 0 for padding rows.
 */
static int32_t attended_set(const problem* p, int32_t b, int32_t h, int32_t i,
                            int32_t* keys, int* is_global_row) {
  int32_t L = p->n - (p->pad_len ? p->pad_len[b] : 0);
  int32_t cnt = 0;
  *is_global_row = 0;
  if (i >= L) return 0;
  if (global_rank(p, i) >= 0) {
    /* a global token attends every valid token (only earlier ones if causal) */
    *is_global_row = 1;
    for (int32_t j = 0; j < L; ++j)
      if (!p->causal || j <= i) keys[cnt++] = j;
    return cnt;
  }
  /* the window: offsets delta*t for t in [-half, +half] (t <= 0 if causal) */
  int64_t delta = p->dilation[h];
  int64_t half = window_of(p, h) / 2;
  if (half > p->n) half = p->n;                  /* wider reaches nothing new */
  int64_t right = p->causal ? 0 : half;
  for (int64_t t = -half; t <= right; ++t) {
    int64_t j = (int64_t)i + delta * t;
    if (j >= 0 && j < L) keys[cnt++] = (int32_t)j;
  }
  /* the global columns, each counted once */
  for (int32_t r = 0; r < p->G; ++r) {
    int32_t g = p->global_idx[r];
    if (g >= L || (p->causal && g > i)) continue;
    if (in_window(p, h, i, g)) continue;         /* already in the band */
    keys[cnt++] = g;
  }
  return cnt;
}

/* one output row: softmax(scale * <q_row, k_j> + bias) weighted sum of v_j over keys */
static void one_row(const problem* p, int32_t b, int32_t h, int32_t i,
                    int32_t* keys, double* scores, double* out_row) {
  const int32_t n = p->n, d = p->d;
  const int64_t bh = (int64_t)b * p->H + h;
  int is_g = 0;
  int32_t cnt = attended_set(p, b, h, i, keys, &is_g);
  for (int32_t c = 0; c < d; ++c) out_row[c] = 0.0;
  if (cnt == 0) return;

  const void *qs, *ks, *vs;
  int64_t qrow;
  if (is_g) {
    qs = p->qg; ks = p->kg; vs = p->vg;
    qrow = bh * p->G + global_rank(p, i);
  } else {
    qs = p->q; ks = p->k; vs = p->v;
    qrow = bh * n + i;
  }
  const double scale = 1.0 / sqrt((double)d);
  double mx = -INFINITY;
  for (int32_t t = 0; t < cnt; ++t) {
    int64_t krow = bh * n + keys[t];
    double s = 0.0;
    for (int32_t c = 0; c < d; ++c)
      s += load_elem(p->dtype, qs, qrow * d + c) * load_elem(p->dtype, ks, krow * d + c);
    s *= scale;
    if (!is_g) s += band_bias(p, h, i, keys[t]);
    scores[t] = s;
    if (s > mx) mx = s;
  }
  double total = 0.0;
  for (int32_t t = 0; t < cnt; ++t) {
    double e = exp(scores[t] - mx);
    total += e;
    int64_t vrow = bh * n + keys[t];
    for (int32_t c = 0; c < d; ++c) out_row[c] += e * load_elem(p->dtype, vs, vrow * d + c);
  }
  for (int32_t c = 0; c < d; ++c) out_row[c] /= total;
}

static int check_problem(const problem* p) {
  if (p->B < 0 || p->H < 0 || p->n < 0 || p->d <= 0) return 1;
  if (p->rel_bias && p->w_heads) return 1; /* the bias table is sized by the one w */
  for (int32_t h = 0; h < (p->w_heads ? p->H : 1); ++h) {
    int64_t w = p->w_heads ? p->w_heads[h] : p->w;
    if (w < 0 || (w & 1)) return 1;
  }
  if (p->G < 0 || (p->G > 0 && !p->global_idx)) return 1;
  for (int32_t h = 0; h < p->H; ++h)
    if (p->dilation[h] < 1) return 1;
  for (int32_t r = 0; r < p->G; ++r) {
    if (p->global_idx[r] < 0 || p->global_idx[r] >= p->n) return 1;
    if (r > 0 && p->global_idx[r] <= p->global_idx[r - 1]) return 1;
  }
  if (p->pad_len)
    for (int32_t b = 0; b < p->B; ++b)
      if (p->pad_len[b] < 0 || p->pad_len[b] > p->n) return 1;
  return 0;
}

/*
 * Full or sampled forward.  rows == NULL: every row, out is [B, H, n, d].
 * Otherwise rows[0..nrows) are flat row ids ((b*H + h)*n + i) and out is
 * [nrows, d].  Returns 0 on success, 1 on an invalid problem.
 */
int lf_oracle_fwd(int dtype, const void* q, const void* k, const void* v,
                  const void* qg, const void* kg, const void* vg,
                  const int32_t* global_idx, int32_t G,
                  int32_t B, int32_t H, int32_t n, int32_t d, int32_t w, const int32_t* w_heads,
                  const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                  const float* rel_bias,
                  const int64_t* rows, int64_t nrows, double* out, int32_t nthreads) {
  problem p = {dtype, q, k, v, qg, kg, vg, global_idx, G, B, H, n, d, w, causal, dilation, pad_len, w_heads,
               rel_bias};
  if (check_problem(&p)) return 1;
  int64_t total = rows ? nrows : (int64_t)B * H * n;
  if (total == 0) return 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int err = 0;
#pragma omp parallel
  {
    int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!keys || !scores) {
#pragma omp atomic write
      err = 2;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t t = 0; t < total; ++t) {
        int64_t flat = rows ? rows[t] : t;
        int32_t i = (int32_t)(flat % n);
        int64_t bh = flat / n;
        int32_t h = (int32_t)(bh % H), b = (int32_t)(bh / H);
        one_row(&p, b, h, i, keys, scores, out + t * d);
      }
    }
    free(keys);
    free(scores);
  }
  return err;
}

/*
 * Backward of one row: with L = sum(dout * out), adds this row's share of
 * dL/dq (or dL/dqg for a global row), dL/dk, dL/dv (or dL/dkg, dL/dvg) into
 * the float64 gradient arrays.  The chain rule through the row's softmax,
 * written out: p_t = softmax(s)_t with s_t = scale * <q_row, k_t>;
 *   dv_t   += p_t * dout_row
 *   dp_t    = <dout_row, v_t>
 *   ds_t    = p_t * (dp_t - sum_u p_u dp_u)
 *   dq_row += scale * sum_t ds_t k_t
 *   dk_t   += scale * ds_t q_row
 *   drb[t]  += ds_t for a band key at window step t (relative bias)
 */
static void one_row_bwd(const problem* p, const void* dout, int32_t b, int32_t h, int32_t i,
                        int32_t* keys, double* scores, double* dp, double* dq, double* dk,
                        double* dv, double* dqg, double* dkg, double* dvg, double* drb) {
  const int32_t n = p->n, d = p->d;
  const int64_t bh = (int64_t)b * p->H + h;
  int is_g = 0;
  int32_t cnt = attended_set(p, b, h, i, keys, &is_g);
  if (cnt == 0) return;
  const void *qs, *ks, *vs;
  double *dq_row, *dks, *dvs;
  int64_t qrow;
  if (is_g) {
    qs = p->qg; ks = p->kg; vs = p->vg;
    qrow = bh * p->G + global_rank(p, i);
    dq_row = dqg + qrow * d; dks = dkg; dvs = dvg;
  } else {
    qs = p->q; ks = p->k; vs = p->v;
    qrow = bh * n + i;
    dq_row = dq + qrow * d; dks = dk; dvs = dv;
  }
  const int64_t orow = bh * n + i;  /* the row's output (and dout) position */
  const double scale = 1.0 / sqrt((double)d);
  /* softmax weights, exactly as the forward computes them */
  double mx = -INFINITY;
  for (int32_t t = 0; t < cnt; ++t) {
    int64_t krow = bh * n + keys[t];
    double s = 0.0;
    for (int32_t c = 0; c < d; ++c)
      s += load_elem(p->dtype, qs, qrow * d + c) * load_elem(p->dtype, ks, krow * d + c);
    scores[t] = s * scale + (is_g ? 0.0 : band_bias(p, h, i, keys[t]));
    if (scores[t] > mx) mx = scores[t];
  }
  double total = 0.0;
  for (int32_t t = 0; t < cnt; ++t) {
    scores[t] = exp(scores[t] - mx);
    total += scores[t];
  }
  for (int32_t t = 0; t < cnt; ++t) scores[t] /= total;  /* scores[] now holds p */
  /* dp_t and their p-weighted sum */
  double dsum = 0.0;
  for (int32_t t = 0; t < cnt; ++t) {
    int64_t vrow = bh * n + keys[t];
    double x = 0.0;
    for (int32_t c = 0; c < d; ++c)
      x += load_elem(p->dtype, dout, orow * d + c) * load_elem(p->dtype, vs, vrow * d + c);
    dp[t] = x;
    dsum += scores[t] * x;
  }
  for (int32_t t = 0; t < cnt; ++t) {
    int64_t kvrow = bh * n + keys[t];
    double ds = scores[t] * (dp[t] - dsum);
    /* the bias enters the score with weight 1: its gradient is ds */
    if (drb && !is_g && in_window(p, h, i, keys[t]))
      drb[((int64_t)keys[t] - i) / p->dilation[h] + p->w / 2] += ds;
    for (int32_t c = 0; c < d; ++c) {
      dvs[kvrow * d + c] += scores[t] * load_elem(p->dtype, dout, orow * d + c);
      dq_row[c] += scale * ds * load_elem(p->dtype, ks, kvrow * d + c);
      dks[kvrow * d + c] += scale * ds * load_elem(p->dtype, qs, qrow * d + c);
    }
  }
}

/*
 * Gradients of L = sum(dout * out) with respect to q, k, v (float64 arrays
 * [B, H, n, d]) and, when G > 0, qg ([B, H, G, d]), kg and vg ([B, H, n, d]).
 * dout has the inputs' dtype and out's shape.  The arrays are zeroed here.
 * Each (b, h) slice is independent (its rows only touch its own slices).
 * Returns 0, 1 for an invalid problem, 2 if memory ran out.
 */
int lf_oracle_bwd(int dtype, const void* q, const void* k, const void* v,
                  const void* qg, const void* kg, const void* vg, const void* dout,
                  const int32_t* global_idx, int32_t G,
                  int32_t B, int32_t H, int32_t n, int32_t d, int32_t w, const int32_t* w_heads,
                  const int32_t* dilation, int32_t causal, const int32_t* pad_len,
                  const float* rel_bias,
                  double* dq, double* dk, double* dv, double* dqg, double* dkg, double* dvg,
                  double* d_rel_bias, int32_t nthreads) {
  problem p = {dtype, q, k, v, qg, kg, vg, global_idx, G, B, H, n, d, w, causal, dilation, pad_len, w_heads,
               rel_bias};
  if (check_problem(&p)) return 1;
  if (d_rel_bias && !rel_bias) return 1;
  /* the bias gradient: one [w + 1] row per (b, h) (each (b, h) runs on one
   * thread), summed over b in order at the end */
  double* drb_bh = NULL;
  if (d_rel_bias) {
    drb_bh = (double*)calloc((size_t)B * H * (w + 1) + 1, sizeof(double));
    if (!drb_bh) return 2;
  }
  if (!dq || !dk || !dv || (G > 0 && (!dqg || !dkg || !dvg))) return 1;
  const size_t full = (size_t)B * H * n * d;
  memset(dq, 0, full * sizeof(double));
  memset(dk, 0, full * sizeof(double));
  memset(dv, 0, full * sizeof(double));
  if (G > 0) {
    memset(dqg, 0, (size_t)B * H * G * d * sizeof(double));
    memset(dkg, 0, full * sizeof(double));
    memset(dvg, 0, full * sizeof(double));
  }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int err = 0;
#pragma omp parallel
  {
    int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!keys || !scores || !dp) {
#pragma omp atomic write
      err = 2;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t bh = 0; bh < (int64_t)B * H; ++bh)
        for (int32_t i = 0; i < n; ++i)
          one_row_bwd(&p, dout, (int32_t)(bh / H), (int32_t)(bh % H), i, keys, scores, dp, dq, dk,
                      dv, dqg, dkg, dvg, drb_bh ? drb_bh + bh * (w + 1) : NULL);
    }
    free(keys);
    free(scores);
    free(dp);
  }
  if (drb_bh) {
    memset(d_rel_bias, 0, (size_t)H * (w + 1) * sizeof(double));
    for (int32_t b = 0; b < B; ++b)
      for (int32_t h = 0; h < H; ++h)
        for (int32_t t = 0; t <= w; ++t)
          d_rel_bias[(int64_t)h * (w + 1) + t] += drb_bh[((int64_t)b * H + h) * (w + 1) + t];
    free(drb_bh);
  }
  return err;
}

/*
 * Linear projections of hidden states into per-head tensors (section 3-1,
 * "Linear Projections for Global Attention": the band and the global
 * attention each have their own W_q, W_k, W_v).  x: [B, n, K] hidden states;
 * w: [N, K] with N = n_out * H * d, the weights of n_out projections stacked
 * along N (row t*H*d + h*d + c gives output t, head h, column c); bias: [N]
 * float32 or NULL.  y: float64 [n_out, B, H, n, d],
 *   y[t, b, h, i, c] = sum_k x[b, i, k] * w[t*H*d + h*d + c, k] + bias[...].
 * x and w share dtype.  Returns 0, or 1 for invalid sizes.
 */
int lf_oracle_proj(int dtype, const void* x, const void* w, const float* bias, int32_t B, int32_t n,
                   int32_t K, int32_t n_out, int32_t H, int32_t d, double* y, int32_t nthreads) {
  if (B < 0 || n < 0 || K < 1 || n_out < 1 || H < 1 || d < 1) return 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const int64_t N = (int64_t)n_out * H * d;
#pragma omp parallel for schedule(static)
  for (int64_t row = 0; row < (int64_t)B * n; ++row) {
    const int64_t b = row / n, i = row % n;
    for (int64_t col = 0; col < N; ++col) {
      double acc = bias ? (double)bias[col] : 0.0;
      for (int32_t kk = 0; kk < K; ++kk)
        acc += load_elem(dtype, x, row * K + kk) * load_elem(dtype, w, col * K + kk);
      const int64_t t = col / ((int64_t)H * d), h = (col / d) % H, c = col % d;
      y[((((t * B + b) * H + h) * n) + i) * d + c] = acc;
    }
  }
  return 0;
}

/*
 * Memory attention combined with the local output (Memorizing Transformer
 * notes, section "Memorizing Transformer": each query also attends the k
 * (key, value) pairs a kNN lookup retrieved from a memory of earlier
 * segments, and the two results are mixed per head by a scalar weight).
 * q, local: [B, H, n, d]; mem_k, mem_v: [B, H, M, d] (the memory of each
 * (b, h)); idx: [B, H, n, km] int32 positions in that memory, -1 for an empty
 * slot; gate: [H] weights in [0, 1].  out: float64 [B, H, n, d],
 *   o_mem = sum_j softmax_j(<q, mem_k[idx_j]> / sqrt(d)) mem_v[idx_j] over the
 *           non-empty slots (zero if every slot is empty),
 *   out = gate[h] * o_mem + (1 - gate[h]) * local.
 * q, local, mem_k, mem_v share dtype.  Returns 0, or 1 for invalid sizes or
 * an index outside [-1, M).
 */
int lf_oracle_mem_combine(int dtype, const void* q, const void* local, const void* mem_k, const void* mem_v,
                          const int32_t* idx, const double* gate, int32_t B, int32_t H, int32_t n, int32_t d,
                          int32_t M, int32_t km, double* out, int32_t nthreads) {
  if (B < 0 || H < 1 || n < 0 || d < 1 || M < 0 || km < 1) return 1;
  for (int64_t t = 0; t < (int64_t)B * H * n * km; ++t)
    if (idx[t] < -1 || idx[t] >= M) return 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)km);
#pragma omp for schedule(static)
    for (int64_t row = 0; row < (int64_t)B * H * n; ++row) {
      const int64_t bh = row / n;
      const int32_t h = (int32_t)(bh % H);
      const int32_t* ix = idx + row * km;
      double mx = -INFINITY;
      for (int32_t j = 0; j < km; ++j) {
        s[j] = -INFINITY;
        if (ix[j] < 0) continue;
        double acc = 0.0;
        for (int32_t c = 0; c < d; ++c)
          acc += load_elem(dtype, q, row * d + c) * load_elem(dtype, mem_k, (bh * M + ix[j]) * d + c);
        s[j] = acc * scale;
        if (s[j] > mx) mx = s[j];
      }
      double total = 0.0;
      for (int32_t j = 0; j < km; ++j) {
        s[j] = (ix[j] < 0) ? 0.0 : exp(s[j] - mx);
        total += s[j];
      }
      for (int32_t c = 0; c < d; ++c) {
        double om = 0.0;
        for (int32_t j = 0; j < km; ++j)
          if (ix[j] >= 0) om += s[j] * load_elem(dtype, mem_v, (bh * M + ix[j]) * d + c);
        if (total > 0.0) om /= total;
        out[row * d + c] = gate[h] * om + (1.0 - gate[h]) * load_elem(dtype, local, row * d + c);
      }
    }
    free(s);
  }
  return 0;
}

/* The attended key set of one row (for pattern tests).  keys must hold n ints. */
int32_t lf_oracle_attended(const int32_t* global_idx, int32_t G, int32_t B, int32_t H,
                           int32_t n, int32_t w, const int32_t* w_heads, const int32_t* dilation,
                           int32_t causal, const int32_t* pad_len, int32_t b, int32_t h, int32_t i,
                           int32_t* keys, int32_t* is_global_row) {
  problem p = {ORC_F64, 0, 0, 0, 0, 0, 0, global_idx, G, B, H, n, 1, w, causal, dilation, pad_len, w_heads, NULL};
  if (check_problem(&p)) return -1;
  int g = 0;
  int32_t cnt = attended_set(&p, b, h, i, keys, &g);
  *is_global_row = g;
  return cnt;
}

/*
 * Attended (row, key) pairs of a whole pattern, by enumerating every row's
 * attended set: *pairs over all rows, *global_pairs over the global tokens'
 * own rows.  Returns 0, or -1 for a rejected pattern.
 */
int32_t lf_oracle_count_pairs(const int32_t* global_idx, int32_t G, int32_t B, int32_t H,
                              int32_t n, int32_t w, const int32_t* w_heads, const int32_t* dilation,
                              int32_t causal, const int32_t* pad_len, int64_t* pairs,
                              int64_t* global_pairs) {
  problem p = {ORC_F64, 0, 0, 0, 0, 0, 0, global_idx, G, B, H, n, 1, w, causal, dilation, pad_len, w_heads, NULL};
  if (check_problem(&p)) return -1;
  int64_t tot = 0, gtot = 0;
  int err = 0;
#pragma omp parallel reduction(+ : tot, gtot) reduction(| : err)
  {
    int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    if (!keys) {
      err = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        for (int32_t i = 0; i < n; ++i) {
          int g = 0;
          int32_t cnt = attended_set(&p, (int32_t)(bh / H), (int32_t)(bh % H), i, keys, &g);
          tot += cnt;
          if (g) gtot += cnt;
        }
      }
      free(keys);
    }
  }
  if (err) return -1;
  *pairs = tot;
  *global_pairs = gtot;
  return 0;
}

/* Number of threads an OpenMP region of this library would use. */
int32_t lf_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
