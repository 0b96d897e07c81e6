/*
 * oracle.c -- plain, slow, fp64 CPU oracle for masked scaled-dot-product attention
 * under structured sparse masks.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file: only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header or table with the CUDA library.
 *
 * What it computes (all indices 0-based):
 *
 *   Allowed sets.  A mask is a union of simple rules ("Attention variants",
 *   sreshtalluri.github.io, §4 Implementation: "Sparse patterns are unions of simple
 *   rules"), intersected with causality when the mask is causal:
 *     - causal local window of width w, counting the query itself: 0 <= i-j < w
 *       ("Sparse attention" glossary, selfmadequant, §Choose the available reads,
 *       the set S_i = {max(1,i-w+1),...,i} in 1-based form; "Attention variants"
 *       §4 sliding_window).  w = 0 means no window: the full causal triangle
 *       (octlm "Sparse attention", §One mask function for every pattern).
 *     - bidirectional local radius r: |i-j| <= r ("Attention variants" §3 worked
 *       example, "local radius 2": query 12 reads 10..14).  r = -1: no limit.
 *     - dilation d >= 1 of the local window: only keys whose distance is a multiple
 *       of d, and w (or r) counts those keys, so the causal window reads i, i-d, ...,
 *       i-(w-1)d: 0 <= i-j < w d with (i-j) % d == 0 ("Attention variants" §6,
 *       the dilated(n, w, d) exercise).  d = 1 is the contiguous window.
 *     - strided columns: key j with j % s == o is readable by every query (causal:
 *       every later query).  o = 0 is the octlm convention (columns % stride == 0),
 *       o = s-1 the "Attention variants" local_strided convention.
 *     - global tokens G: rows in G read every key, columns in G are read by every
 *       query ("Attention variants" §4 with_global; ai360xpert "Sparse Attention",
 *       §Global tokens).  In a causal mask both stay causal ("Attention variants",
 *       the look-ahead warning after with_global).
 *     - random blocks (BigBird, getnybble "Sparse and sliding-window attention",
 *       §Block-sparse attention: BigBird): with block size b, a list of (query block,
 *       key block) pairs; query i reads every key j with (i / b, j / b) in the list
 *       (causal: j <= i).  Which blocks are random is an input (drawn by a seeded
 *       generator outside), so the rule itself is deterministic.
 *
 *   Attention.  For each query i with allowed set S_i (never empty: j = i is always
 *   allowed),
 *       s_ij = scale * q_i . k_j               (j in S_i)
 *       y_i  = sum_{j in S_i} softmax_j(s_ij) v_j,  softmax over S_i only
 *       LSE_i = ln sum_{j in S_i} exp(s_ij)
 *   ("Sparse attention" glossary, §Choose the available reads, the displayed
 *   equation for y_i and alpha_ij; softmax normalises over allowed keys only.)
 *   Evaluated in fp64 with the usual max subtraction, which leaves the value
 *   unchanged.
 *
 *   Gradients.  oracle_attention_bwd_head: dQ, dK, dV of the same y given dO, by the
 *   chain rule through the softmax over S_i (see the function);
 *   oracle_attention_bwd_dq_rows and oracle_attention_bwd_dkdv_keys: the same
 *   gradients for listed query rows or listed keys only.
 *
 *   Decode.  oracle_decode: one new token against a ring-buffer KV cache that keeps
 *   the last cap tokens (see the function).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int causal;      /* 1: j <= i only */
  int64_t window;  /* causal local width, 0 = unbounded */
  int64_t radius;  /* bidirectional radius, -1 = unbounded */
  int64_t dilation; /* local keys every dilation-th position, >= 1 */
  int64_t stride;  /* 0 = none */
  int64_t offset;  /* strided columns: j % stride == offset */
  int64_t n_global;
  const int32_t* global_pos; /* sorted ascending, distinct */
  int64_t T;
  int64_t rand_block;        /* random-block size b (0 = no random blocks) */
  int64_t n_rand;
  const int32_t* rand_pairs; /* [n_rand][2] (query block, key block), sorted, distinct */
} omask;

/* ---- spec checks: the readings every valid mask obeys ------------------------- */

/* Returns 0 for a valid mask, a negative code naming the first violated rule. */
int oracle_validate(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                    int64_t offset, int64_t n_global, const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs) {
  if (T <= 0) return -1;
  if (causal != 0 && causal != 1) return -2;
  if (causal == 1 && (window < 0 || radius != -1)) return -3;
  if (causal == 0 && (radius < -1 || window != 0)) return -4;
  /* products of a width and the dilation must stay far inside int64 */
  if (dilation < 1 || dilation > ((int64_t)1 << 31) || window > ((int64_t)1 << 31) ||
      radius > ((int64_t)1 << 31))
    return -10;
  if (stride < 0) return -5;
  if (stride == 0 && offset != 0) return -6;
  if (stride > 0 && (offset < 0 || offset >= stride)) return -6;
  if (n_global < 0 || n_global > T) return -7;
  for (int64_t a = 0; a < n_global; a++) {
    if (gpos[a] < 0 || gpos[a] >= T) return -8;
    if (a > 0 && gpos[a] <= gpos[a - 1]) return -9; /* sorted, distinct */
  }
  if (n_rand < 0) return -11;
  if (n_rand > 0) {
    if (rand_block != 16 && rand_block != 32 && rand_block != 64 && rand_block != 128)
      return -11;
    const int64_t nb = (T + rand_block - 1) / rand_block;
    for (int64_t a = 0; a < n_rand; a++) {
      const int64_t q = rand_pairs[2 * a], k = rand_pairs[2 * a + 1];
      if (q < 0 || q >= nb || k < 0 || k >= nb) return -12;
      if (a > 0) { /* sorted by (query block, key block), distinct */
        const int64_t pq = rand_pairs[2 * a - 2], pk = rand_pairs[2 * a - 1];
        if (q < pq || (q == pq && k <= pk)) return -13;
      }
    }
  }
  return 0;
}

/* Index of the first random pair whose query block is >= qb (pairs are sorted). */
static int64_t rand_lower(const omask* m, int64_t qb) {
  int64_t lo = 0, hi = m->n_rand;
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (m->rand_pairs[2 * mid] < qb) lo = mid + 1; else hi = mid;
  }
  return lo;
}

/* Is (i, j) inside one of the random blocks of i's query block? */
static int in_random(const omask* m, int64_t i, int64_t j) {
  if (m->n_rand == 0) return 0;
  const int64_t qb = i / m->rand_block, kb = j / m->rand_block;
  for (int64_t a = rand_lower(m, qb); a < m->n_rand && m->rand_pairs[2 * a] == qb; a++)
    if (m->rand_pairs[2 * a + 1] == kb) return 1;
  return 0;
}

static int in_global(const omask* m, int64_t x) {
  for (int64_t a = 0; a < m->n_global; a++)
    if (m->global_pos[a] == x) return 1;
  return 0;
}

/* ---- the rule itself, one (i, j) pair at a time --------------------------------- */

static int allowed(const omask* m, int64_t i, int64_t j) {
  if (m->causal && j > i) return 0;             /* causality prohibits future reads */
  if (in_global(m, i)) return 1;                /* a global row reads every key */
  if (in_global(m, j)) return 1;                /* every query reads a global column */
  if (m->stride > 0 && j % m->stride == m->offset) return 1; /* strided column */
  if (in_random(m, i, j)) return 1;             /* a random block of i's query block */
  const int64_t gap = i - j;
  if (llabs(gap) % m->dilation != 0) return 0;                  /* every d-th key only */
  if (m->causal) return m->window == 0 || gap < m->window * m->dilation; /* 0 <= i-j < w d */
  return m->radius < 0 || llabs(gap) <= m->radius * m->dilation;         /* |i-j| <= r d */
}

int oracle_allowed(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                   int64_t offset, int64_t n_global, const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs,
                   int64_t i, int64_t j) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  return allowed(&m, i, j);
}

/* S_i by scanning every key and asking the rule: the plainest form. */
static int64_t row_set_scan(const omask* m, int64_t i, int32_t* out) {
  int64_t n = 0;
  for (int64_t j = 0; j < m->T; j++)
    if (allowed(m, i, j)) {
      if (out) out[n] = (int32_t)j;
      n++;
    }
  return n;
}

/* S_i as the literal union of the rule sets (window interval, strided progression,
 * global columns, or everything for a global row), each enumerated directly, then
 * merged in ascending order without repeats.  Same set as row_set_scan (a test
 * checks this); it exists because it costs O(|S_i| + |G|) instead of O(T). */
static int64_t row_set_union(const omask* m, int64_t i, int32_t* out) {
  const int64_t T = m->T;
  const int64_t jmax = m->causal ? i : T - 1; /* causal cut */
  int64_t n = 0;
  if (in_global(m, i)) { /* global row: every key causality permits */
    for (int64_t j = 0; j <= jmax; j++) out[n++] = (int32_t)j;
    return n;
  }
  int64_t lo, hi; /* local span; the local keys are its j with (i - j) % dilation == 0 */
  if (m->causal) {
    lo = (m->window == 0) ? 0 : i - (m->window - 1) * m->dilation;
    hi = i;
  } else {
    lo = (m->radius < 0) ? 0 : i - m->radius * m->dilation;
    hi = (m->radius < 0) ? T - 1 : i + m->radius * m->dilation;
  }
  if (lo < 0) lo = 0;
  if (hi > jmax) hi = jmax;
  /* four ascending streams: strided progression, global columns, local interval,
   * the columns of the random key blocks of i's query block (in key-block order) */
  int64_t js = (m->stride > 0) ? m->offset : T; /* next strided column */
  int64_t ag = 0;                                /* next global index */
  int64_t jl = lo + (i - lo) % m->dilation;       /* next local column (lo <= i) */
  const int64_t qb = m->n_rand ? i / m->rand_block : -1;
  int64_t ar = m->n_rand ? rand_lower(m, qb) : 0; /* current random pair */
  int64_t jr = (ar < m->n_rand && m->rand_pairs[2 * ar] == qb)
                   ? m->rand_pairs[2 * ar + 1] * m->rand_block : INT64_MAX;
  int64_t last = -1;
  for (;;) {
    int64_t cs = (js <= jmax) ? js : INT64_MAX;
    int64_t cg = (ag < m->n_global && m->global_pos[ag] <= jmax) ? m->global_pos[ag]
                                                                  : INT64_MAX;
    int64_t cl = (jl <= hi) ? jl : INT64_MAX;
    int64_t cr = (jr <= jmax && jr < T) ? jr : INT64_MAX;
    int64_t c = cs < cg ? cs : cg;
    if (cl < c) c = cl;
    if (cr < c) c = cr;
    if (c == INT64_MAX) break;
    if (c != last) out[n++] = (int32_t)c;
    last = c;
    if (c == cs) js += m->stride;
    if (c == cg) ag++;
    if (c == cl) jl += m->dilation;
    if (c == cr) { /* next column of this block, or the first of the next block */
      jr++;
      if (jr % m->rand_block == 0 || jr >= T) {
        ar++;
        jr = (ar < m->n_rand && m->rand_pairs[2 * ar] == qb)
                 ? m->rand_pairs[2 * ar + 1] * m->rand_block : INT64_MAX;
      }
    }
  }
  return n;
}

/* Allowed set of one query, ascending.  method 0: union of rule sets, 1: full scan.
 * `out` must hold T entries.  Returns |S_i|. */
int64_t oracle_row_set(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                       int64_t offset, int64_t n_global, const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs,
                       int64_t i, int method, int32_t* out) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  return method ? row_set_scan(&m, i, out) : row_set_union(&m, i, out);
}

/* Number of allowed (i, j) pairs: the sum of |S_i| (the glossary's edge count E). */
int64_t oracle_count_pairs(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                           int64_t offset, int64_t n_global, const int32_t* gpos,
                           int64_t T, int64_t rand_block, int64_t n_rand,
                           const int32_t* rand_pairs) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  int64_t total = 0;
#pragma omp parallel
  {
    int32_t* buf = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
#pragma omp for schedule(dynamic, 64) reduction(+ : total)
    for (int64_t i = 0; i < T; i++) total += row_set_union(&m, i, buf);
    free(buf);
  }
  return total;
}

/* Histogram of allowed pairs into BM x BN tiles: cnt[(i/BM) * nkb + (j/BN)].
 * `cnt` has ceil(T/BM) * ceil(T/BN) int32 entries and is overwritten. */
void oracle_tile_counts(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                        int64_t offset, int64_t n_global, const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs,
                        int64_t BM, int64_t BN, int32_t* cnt) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  const int64_t nqb = (T + BM - 1) / BM, nkb = (T + BN - 1) / BN;
  memset(cnt, 0, sizeof(int32_t) * (size_t)(nqb * nkb));
#pragma omp parallel
  {
    int32_t* buf = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
    /* one query block per iteration: its rows only touch its own row of tiles */
#pragma omp for schedule(dynamic, 1)
    for (int64_t qb = 0; qb < nqb; qb++) {
      for (int64_t i = qb * BM; i < (qb + 1) * BM && i < T; i++) {
        int64_t n = row_set_union(&m, i, buf);
        for (int64_t a = 0; a < n; a++) cnt[qb * nkb + buf[a] / BN] += 1;
      }
    }
    free(buf);
  }
}

/* ---- attention over the allowed sets ------------------------------------------- */

static double load_elem(const void* p, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)p)[idx];
  /* dtype 1: bf16 bit patterns; a bf16 value is the top half of an fp32 */
  uint32_t bits = (uint32_t)((const uint16_t*)p)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* One head.  Q, K, V: [T][d] row-major, dtype 0 = fp32, 1 = bf16 bits.
 * rows: the query indices to evaluate (n_rows of them).
 * O: [n_rows][d] fp64, LSE: [n_rows] fp64 (natural log).  Returns total |S_i|. */
int64_t oracle_attention_head(int causal, int64_t window, int64_t radius, int64_t dilation, int64_t stride,
                              int64_t offset, int64_t n_global, const int32_t* gpos,
                              int64_t T, int64_t rand_block, int64_t n_rand,
                              const int32_t* rand_pairs, int64_t d, int dtype, const void* Q,
                              const void* K, const void* V, double scale,
                              const int64_t* rows, int64_t n_rows, double* O,
                              double* LSE) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  int64_t total = 0;
#pragma omp parallel
  {
    int32_t* set = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
    double* s = (double*)malloc(sizeof(double) * (size_t)T);
    double* q = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4) reduction(+ : total)
    for (int64_t r = 0; r < n_rows; r++) {
      const int64_t i = rows[r];
      const int64_t n = row_set_union(&m, i, set);
      total += n;
      for (int64_t k = 0; k < d; k++) q[k] = load_elem(Q, dtype, i * d + k);
      /* logits over the allowed keys only */
      double mx = -INFINITY;
      for (int64_t a = 0; a < n; a++) {
        const int64_t j = set[a];
        double acc = 0.0;
        for (int64_t k = 0; k < d; k++) acc += q[k] * load_elem(K, dtype, j * d + k);
        s[a] = scale * acc;
        if (s[a] > mx) mx = s[a];
      }
      /* normaliser over S_i */
      double l = 0.0;
      for (int64_t a = 0; a < n; a++) l += exp(s[a] - mx);
      /* weighted values */
      double* y = O + r * d;
      for (int64_t k = 0; k < d; k++) y[k] = 0.0;
      for (int64_t a = 0; a < n; a++) {
        const double alpha = exp(s[a] - mx) / l;
        const int64_t j = set[a];
        for (int64_t k = 0; k < d; k++) y[k] += alpha * load_elem(V, dtype, j * d + k);
      }
      LSE[r] = mx + log(l);
    }
    free(set);
    free(s);
    free(q);
  }
  return total;
}

/* ---- gradients of the attention over the allowed sets ------------------------- */

/* One row i of the gradient: recomputes alpha_ij over S_i, adds row i's share to
 * dK and dV (when they are not NULL) and writes dQ_i to dq_row.  set, a, da: [T]. */
static void bwd_row(const omask* m, int64_t i, int64_t d, int dtype, const void* Q,
                    const void* K, const void* V, const void* dO, double scale, double* dq_row,
                    double* dK, double* dV, int32_t* set, double* a, double* da) {
  const int64_t n = row_set_union(m, i, set);
  double mx = -INFINITY;
  for (int64_t t = 0; t < n; t++) {
    double acc = 0.0;
    for (int64_t k = 0; k < d; k++)
      acc += load_elem(Q, dtype, i * d + k) * load_elem(K, dtype, set[t] * d + k);
    a[t] = scale * acc;
    if (a[t] > mx) mx = a[t];
  }
  double l = 0.0;
  for (int64_t t = 0; t < n; t++) l += exp(a[t] - mx);
  double D = 0.0;
  for (int64_t t = 0; t < n; t++) {
    a[t] = exp(a[t] - mx) / l; /* alpha_ij */
    double acc = 0.0;
    for (int64_t k = 0; k < d; k++)
      acc += load_elem(dO, dtype, i * d + k) * load_elem(V, dtype, set[t] * d + k);
    da[t] = acc;
    D += a[t] * acc;
  }
  for (int64_t k = 0; k < d; k++) dq_row[k] = 0.0;
  for (int64_t t = 0; t < n; t++) {
    const int64_t j = set[t];
    const double ds = a[t] * (da[t] - D);
    for (int64_t k = 0; k < d; k++) {
      dq_row[k] += scale * ds * load_elem(K, dtype, j * d + k);
      if (dV) dV[j * d + k] += a[t] * load_elem(dO, dtype, i * d + k);
      if (dK) dK[j * d + k] += scale * ds * load_elem(Q, dtype, i * d + k);
    }
  }
}

/* One head: given dO (the gradient of a loss with respect to y), the gradients with
 * respect to Q, K and V of y_i = sum_{j in S_i} alpha_ij v_j, alpha_ij =
 * softmax_{j in S_i}(scale q_i . k_j).  By the chain rule through the softmax over S_i:
 *   dV_j = sum_{i : j in S_i} alpha_ij dO_i
 *   dalpha_ij = dO_i . v_j,   D_i = sum_{j in S_i} alpha_ij dalpha_ij  (= dO_i . y_i)
 *   ds_ij = alpha_ij (dalpha_ij - D_i)            (softmax Jacobian over S_i)
 *   dQ_i = scale sum_{j in S_i} ds_ij k_j,   dK_j = scale sum_{i : j in S_i} ds_ij q_i
 * Every row is recomputed from its definition in fp64 (no saved forward state).
 * Q, K, V, dO: [T][d], dtype 0 = fp32, 1 = bf16 bits.  dQ, dK, dV: [T][d] fp64,
 * overwritten.  Sequential over rows (dK and dV gather from every row). */
void oracle_attention_bwd_head(int causal, int64_t window, int64_t radius, int64_t dilation,
                               int64_t stride, int64_t offset, int64_t n_global,
                               const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs, int64_t d, int dtype,
                               const void* Q, const void* K, const void* V, const void* dO,
                               double scale, double* dQ, double* dK, double* dV) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  int32_t* set = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
  double* a = (double*)malloc(sizeof(double) * (size_t)T);
  double* da = (double*)malloc(sizeof(double) * (size_t)T);
  memset(dK, 0, sizeof(double) * (size_t)(T * d));
  memset(dV, 0, sizeof(double) * (size_t)(T * d));
  for (int64_t i = 0; i < T; i++)
    bwd_row(&m, i, d, dtype, Q, K, V, dO, scale, dQ + i * d, dK, dV, set, a, da);
  free(set);
  free(a);
  free(da);
}

/* dQ alone for the listed rows (each row's dQ needs only its own set):
 * dQ_rows[r][d] = dQ of row rows[r].  Rows are independent, so they run in
 * parallel. */
void oracle_attention_bwd_dq_rows(int causal, int64_t window, int64_t radius, int64_t dilation,
                                  int64_t stride, int64_t offset, int64_t n_global,
                                  const int32_t* gpos, int64_t T, int64_t rand_block, int64_t n_rand, const int32_t* rand_pairs, int64_t d, int dtype,
                                  const void* Q, const void* K, const void* V, const void* dO,
                                  double scale, const int64_t* rows, int64_t n_rows,
                                  double* dQ_rows) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
#pragma omp parallel
  {
    int32_t* set = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
    double* a = (double*)malloc(sizeof(double) * (size_t)T);
    double* da = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; r++)
      bwd_row(&m, rows[r], d, dtype, Q, K, V, dO, scale, dQ_rows + r * d, NULL, NULL, set, a,
              da);
    free(set);
    free(a);
    free(da);
  }
}

/* dK and dV of the listed keys only.  Key j takes a share from every row i whose
 * allowed set holds it (the transposed set {i : j in S_i}), and each share needs row
 * i's whole softmax: its logit maximum, its normaliser and D_i, all over S_i.  So:
 * (1) mark the rows that read at least one listed key; (2) compute those rows'
 * softmax statistics over their allowed sets, as bwd_row does; (3) for each listed
 * key, visit the rows in ascending order and add
 *   dV_j += alpha_ij dO_i,   dK_j += scale alpha_ij (dO_i . v_j - D_i) q_i
 * (the same chain rule as oracle_attention_bwd_head, read key by key).
 * keys: n_keys distinct indices in [0, T).  dK_keys, dV_keys: [n_keys][d] fp64. */
void oracle_attention_bwd_dkdv_keys(int causal, int64_t window, int64_t radius,
                                    int64_t dilation, int64_t stride, int64_t offset,
                                    int64_t n_global, const int32_t* gpos, int64_t T,
                                    int64_t rand_block, int64_t n_rand,
                                    const int32_t* rand_pairs, int64_t d, int dtype,
                                    const void* Q, const void* K, const void* V,
                                    const void* dO, double scale, const int64_t* keys,
                                    int64_t n_keys, double* dK_keys, double* dV_keys) {
  omask m = {causal,     window,  radius, dilation, stride, offset,
               n_global,   gpos,    T,      rand_block, n_rand, rand_pairs};
  unsigned char* need = (unsigned char*)calloc((size_t)T, 1);
  double* rmax = (double*)malloc(sizeof(double) * (size_t)T);
  double* rsum = (double*)malloc(sizeof(double) * (size_t)T);
  double* rD = (double*)malloc(sizeof(double) * (size_t)T);
  /* (1) rows that read a listed key */
#pragma omp parallel for schedule(dynamic, 256)
  for (int64_t i = 0; i < T; i++)
    for (int64_t a = 0; a < n_keys; a++)
      if (allowed(&m, i, keys[a])) {
        need[i] = 1;
        break;
      }
  /* (2) their softmax statistics over S_i */
#pragma omp parallel
  {
    int32_t* set = (int32_t*)malloc(sizeof(int32_t) * (size_t)T);
    double* s = (double*)malloc(sizeof(double) * (size_t)T);
#pragma omp for schedule(dynamic, 8)
    for (int64_t i = 0; i < T; i++) {
      if (!need[i]) continue;
      const int64_t n = row_set_union(&m, i, set);
      double mx = -INFINITY;
      for (int64_t t = 0; t < n; t++) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; k++)
          acc += load_elem(Q, dtype, i * d + k) * load_elem(K, dtype, set[t] * d + k);
        s[t] = scale * acc;
        if (s[t] > mx) mx = s[t];
      }
      double l = 0.0;
      for (int64_t t = 0; t < n; t++) l += exp(s[t] - mx);
      double D = 0.0;
      for (int64_t t = 0; t < n; t++) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; k++)
          acc += load_elem(dO, dtype, i * d + k) * load_elem(V, dtype, set[t] * d + k);
        D += exp(s[t] - mx) / l * acc;
      }
      rmax[i] = mx;
      rsum[i] = l;
      rD[i] = D;
    }
    free(set);
    free(s);
  }
  /* (3) each listed key gathers the shares of the rows that read it */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t a = 0; a < n_keys; a++) {
    const int64_t j = keys[a];
    double* dk = dK_keys + a * d;
    double* dv = dV_keys + a * d;
    for (int64_t k = 0; k < d; k++) dk[k] = dv[k] = 0.0;
    for (int64_t i = 0; i < T; i++) {
      if (!allowed(&m, i, j)) continue;
      double qk = 0.0, gv = 0.0;
      for (int64_t k = 0; k < d; k++) {
        qk += load_elem(Q, dtype, i * d + k) * load_elem(K, dtype, j * d + k);
        gv += load_elem(dO, dtype, i * d + k) * load_elem(V, dtype, j * d + k);
      }
      const double alpha = exp(scale * qk - rmax[i]) / rsum[i];
      const double ds = alpha * (gv - rD[i]);
      for (int64_t k = 0; k < d; k++) {
        dv[k] += alpha * load_elem(dO, dtype, i * d + k);
        dk[k] += scale * ds * load_elem(Q, dtype, i * d + k);
      }
    }
  }
  free(need);
  free(rmax);
  free(rsum);
  free(rD);
}

/* ---- decode with a capped KV cache ------------------------------------------------ */

/* One decode step of one query head: the token at position t attends to positions
 * max(0, t-w+1) .. t, the w most recent tokens including itself ("Sparse and
 * sliding-window attention", getnybble, §Sliding window attention).  The cache keeps
 * only the last cap >= w tokens ("Attention variants" §1, a sliding-window layer keeps
 * the last w keys and values): position p lives in slot p % cap, so K/V of position
 * p are Kc[p % cap], Vc[p % cap].  q: [d], Kc, Vc: [cap][d] (dtype 0 fp32, 1 bf16
 * bits).  Writes out[d] (fp64) and *lse = ln sum exp(scale q.k).  t < 0: no keys,
 * out = 0, *lse = -inf. */
void oracle_decode(int64_t cap, int64_t w, int64_t t, int64_t d, int dtype, const void* q,
                   const void* Kc, const void* Vc, double scale, double* out, double* lse) {
  for (int64_t k = 0; k < d; k++) out[k] = 0.0;
  if (t < 0) {
    *lse = -INFINITY;
    return;
  }
  const int64_t p0 = t - w + 1 > 0 ? t - w + 1 : 0;
  const int64_t n = t - p0 + 1;
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double mx = -INFINITY;
  for (int64_t a = 0; a < n; a++) {
    const int64_t slot = (p0 + a) % cap;
    double acc = 0.0;
    for (int64_t k = 0; k < d; k++)
      acc += load_elem(q, dtype, k) * load_elem(Kc, dtype, slot * d + k);
    s[a] = scale * acc;
    if (s[a] > mx) mx = s[a];
  }
  double l = 0.0;
  for (int64_t a = 0; a < n; a++) l += exp(s[a] - mx);
  for (int64_t a = 0; a < n; a++) {
    const int64_t slot = (p0 + a) % cap;
    const double wgt = exp(s[a] - mx) / l;
    for (int64_t k = 0; k < d; k++) out[k] += wgt * load_elem(Vc, dtype, slot * d + k);
  }
  *lse = mx + log(l);
  free(s);
}

/* Number of OpenMP threads the oracle uses (1 when built without OpenMP). */
int oracle_num_threads(void) {
  int n = 1;
#ifdef _OPENMP
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
#endif
  return n;
}
