/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact scaled-dot-product
 * attention over packed ragged batches.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into a separate shared
 * library that only the test suite, the smoke check and the benchmark's CPU
 * baseline load.  The CUDA library never links, includes or calls it, and it
 * shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition, written out:
 *
 *   O_i = sum_{j in A_i} softmax_j(scale * q_i . k_j) v_j,
 *   lse_i = ln sum_{j in A_i} exp(scale * q_i . k_j)   (natural log of the
 *           scaled logits),
 *
 * with the allowed set A_i materialised explicitly as a boolean row over every
 * packed key, from per-token sequence ids and in-sequence positions
 * ("causal-mask-and-ragged-sequence-layouts", first paragraph).  The
 * "formal-correctness" page ("The FlashAttention Proof": online softmax
 * recurrence, and the invariant that it equals recomputed softmax) is why the
 * oracle is the two-pass stable softmax and not the online recurrence: the
 * recurrence computes the same function, so the oracle is that function.
 *
 * Conventions (each is a reading; they are listed with their reasons in the
 * design notes):
 *   - Layout: q [total_q, hq, d], k and v [total_k, hkv, d], o like q,
 *     lse [hq, total_q], all row-major, fp64.
 *   - GQA: query head h reads KV head h / (hq / hkv) (contiguous grouping).
 *   - mask_kind 0: no causal rule; 1: top-left, key position <= query
 *     position; 2: bottom-right, key position <= query position + Nk - Nq
 *     ("causal-mask-and-ragged-sequence-layouts", third paragraph).
 *   - window > 0 (causal kinds only) keeps, of the keys the causal rule
 *     allows, those at most window - 1 positions before the causal bound: a
 *     bounded window ("attention-algorithm-error-and-complexity-tests",
 *     fifth paragraph).
 *   - Pairs in different sequences are never allowed.
 *   - slopes != NULL adds a linear positional bias to every allowed logit:
 *     b_ij = -slopes[h] * |i + off - j|, the distance between key position j
 *     and the row's causal bound i + off (off = Nk - Nq for bottom-right, 0
 *     otherwise), so the key at the bound gets no bias ("attention-algorithm-
 *     error-and-complexity-tests", third paragraph, and "causal-mask-and-
 *     ragged-sequence-layouts", sixth paragraph: biases move with the
 *     positions and are rebuilt the same way in the backward).
 *   - btab != NULL adds an explicit bias tensor to every allowed logit:
 *     B[s][h][i][j] = btab[s * bss + h * bhs + i * brs + j] for sequence s,
 *     query head h, in-sequence row i and key j (a stride of 0 broadcasts),
 *     in the units of the scaled logits.  An entry of -inf removes the pair:
 *     exp(-inf) = 0, so it is an explicit mask ("attention-algorithm-error-
 *     and-complexity-tests", third paragraph: bias and mask terms enter the
 *     logits before the softmax; "causal-mask-and-ragged-sequence-layouts",
 *     sixth paragraph: the backward rebuilds them identically).
 *   - A row whose allowed set is empty, or whose allowed logits are all -inf,
 *     has O = 0 exactly and lse = -inf (same page, fourth paragraph).
 *
 * Backward (recompute form, at a given upstream gradient dO):
 *   P_ij = exp(s_ij - lse_i), dP_ij = dO_i . v_j, D_i = dO_i . O_i,
 *   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j, dK_j = scale sum_i dS_ij q_i,
 *   dV_j = sum_i P_ij dO_i,
 * computed on K and V repeated to hq heads and then summed over each group
 * ("attention-algorithm-error-and-complexity-tests", third paragraph).
 *
 * Parallelism: OpenMP over independent query heads or rows only; every sum is
 * taken in plain index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MASK_NONE 0
#define ORACLE_MASK_TOP_LEFT 1
#define ORACLE_MASK_BOTTOM_RIGHT 2

typedef struct {
  const double *q, *k, *v;
  const int32_t *cu_q, *cu_k;
  int batch, total_q, total_k, hq, hkv, d;
  double scale;
  int mask_kind;
  int window; /* > 0: at most `window` keys per row, the latest allowed ones */
  const double *slopes; /* [hq] linear positional bias slopes, or NULL */
  const double *btab;   /* explicit bias tensor, or NULL */
  int64_t bss, bhs, brs; /* its sequence, head and row strides */
  int32_t *seq_q, *pos_q, *seq_k, *pos_k; /* per-token metadata */
} problem_t;

/* Sequence id and in-sequence position of every packed token.  Returns 0, or
 * -1 when the cumulative lengths are not a valid partition of [0, total). */
int oracle_token_meta(const int32_t *cu, int batch, int total, int32_t *seq_id,
                      int32_t *pos) {
  if (batch < 0 || total < 0) return -1;
  if (cu[0] != 0 || cu[batch] != total) return -1;
  for (int s = 0; s < batch; s++)
    if (cu[s + 1] < cu[s]) return -1;
  for (int t = 0; t < total; t++) {
    seq_id[t] = -1;
    pos[t] = -1;
  }
  for (int s = 0; s < batch; s++)
    for (int t = cu[s]; t < cu[s + 1]; t++) {
      seq_id[t] = s;
      pos[t] = t - cu[s];
    }
  return 0;
}

/* The allowed-pair rule for one (query token, key token) pair. */
static int pair_allowed(const problem_t *p, int tq, int tk) {
  int s = p->seq_q[tq];
  if (s < 0 || p->seq_k[tk] != s) return 0;
  int i = p->pos_q[tq], j = p->pos_k[tk];
  int nq = p->cu_q[s + 1] - p->cu_q[s];
  int nk = p->cu_k[s + 1] - p->cu_k[s];
  int bound; /* the causal rule allows j <= bound */
  switch (p->mask_kind) {
    case ORACLE_MASK_NONE:
      return 1;
    case ORACLE_MASK_TOP_LEFT:
      bound = i;
      break;
    case ORACLE_MASK_BOTTOM_RIGHT:
      bound = i + nk - nq;
      break;
    default:
      return 0;
  }
  if (j > bound) return 0;
  /* bounded window: only the `window` positions up to the causal bound */
  if (p->window > 0 && bound - j >= p->window) return 0;
  return 1;
}

static double dot(const double *a, const double *b, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; c++) acc += a[c] * b[c];
  return acc;
}

/* The positional bias of query head h for an allowed (query token, key token)
 * pair: 0 without slopes. */
static double pos_bias(const problem_t *p, int tq, int tk, int h) {
  if (!p->slopes) return 0.0;
  int s = p->seq_q[tq];
  int nq = p->cu_q[s + 1] - p->cu_q[s];
  int nk = p->cu_k[s + 1] - p->cu_k[s];
  int off = p->mask_kind == ORACLE_MASK_BOTTOM_RIGHT ? nk - nq : 0;
  int dist = p->pos_q[tq] + off - p->pos_k[tk];
  return -p->slopes[h] * fabs((double)dist);
}

/* The explicit bias tensor's entry for an allowed (query token, key token)
 * pair of query head h: 0 without a tensor. */
static double tab_bias(const problem_t *p, int tq, int tk, int h) {
  if (!p->btab) return 0.0;
  int64_t s = p->seq_q[tq], i = p->pos_q[tq], j = p->pos_k[tk];
  return p->btab[s * p->bss + (int64_t)h * p->bhs + i * p->brs + j];
}

/* The logit of an allowed pair: scaled dot product plus both biases. */
static double logit(const problem_t *p, const double *qi, const double *kj,
                    int tq, int tk, int h) {
  return p->scale * dot(qi, kj, p->d) + pos_bias(p, tq, tk, h) + tab_bias(p, tq, tk, h);
}

static const double *q_row(const problem_t *p, int t, int h) {
  return p->q + ((size_t)t * p->hq + h) * p->d;
}
static const double *k_row(const problem_t *p, int t, int hk) {
  return p->k + ((size_t)t * p->hkv + hk) * p->d;
}
static const double *v_row(const problem_t *p, int t, int hk) {
  return p->v + ((size_t)t * p->hkv + hk) * p->d;
}

/* One query row: materialise its mask row over all packed keys, then the
 * two-pass stable softmax.  mrow (total_k bytes) and srow (total_k doubles)
 * are scratch. */
static void forward_row(const problem_t *p, int t, int h, unsigned char *mrow,
                        double *srow, double *o, double *lse) {
  int hk = h / (p->hq / p->hkv);
  int any = 0;
  for (int u = 0; u < p->total_k; u++) {
    mrow[u] = (unsigned char)pair_allowed(p, t, u);
    any |= mrow[u];
  }
  for (int c = 0; c < p->d; c++) o[c] = 0.0;
  if (!any) {
    *lse = -INFINITY;
    return;
  }
  const double *qi = q_row(p, t, h);
  double m = -INFINITY;
  for (int u = 0; u < p->total_k; u++) {
    if (!mrow[u]) continue;
    srow[u] = logit(p, qi, k_row(p, u, hk), t, u, h);
    if (srow[u] > m) m = srow[u];
  }
  if (m == -INFINITY) { /* every allowed logit masked by the bias tensor */
    *lse = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int u = 0; u < p->total_k; u++)
    if (mrow[u]) l += exp(srow[u] - m);
  double lse_i = m + log(l);
  for (int u = 0; u < p->total_k; u++) {
    if (!mrow[u]) continue;
    double pij = exp(srow[u] - lse_i);
    const double *vj = v_row(p, u, hk);
    for (int c = 0; c < p->d; c++) o[c] += pij * vj[c];
  }
  *lse = lse_i;
}

static int setup(problem_t *p, const double *q, const double *k,
                 const double *v, const int32_t *cu_q, const int32_t *cu_k,
                 int batch, int total_q, int total_k, int hq, int hkv, int d,
                 double scale, int mask_kind, int window, const double *slopes,
                 const double *btab, const int64_t *bstr) {
  p->seq_q = p->pos_q = p->seq_k = p->pos_k = NULL;
  if (btab && (!bstr || bstr[0] < 0 || bstr[1] < 0 || bstr[2] < 0)) return -1;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0 || d <= 0) return -1;
  if (mask_kind < 0 || mask_kind > 2) return -1;
  if (window > 0 && mask_kind == ORACLE_MASK_NONE) return -1;
  p->q = q;
  p->k = k;
  p->v = v;
  p->cu_q = cu_q;
  p->cu_k = cu_k;
  p->batch = batch;
  p->total_q = total_q;
  p->total_k = total_k;
  p->hq = hq;
  p->hkv = hkv;
  p->d = d;
  p->scale = scale;
  p->mask_kind = mask_kind;
  p->window = window;
  p->slopes = slopes;
  p->btab = btab;
  p->bss = btab ? bstr[0] : 0;
  p->bhs = btab ? bstr[1] : 0;
  p->brs = btab ? bstr[2] : 0;
  p->seq_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_q + 1));
  p->pos_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_q + 1));
  p->seq_k = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_k + 1));
  p->pos_k = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_k + 1));
  if (oracle_token_meta(cu_q, batch, total_q, p->seq_q, p->pos_q) != 0 ||
      oracle_token_meta(cu_k, batch, total_k, p->seq_k, p->pos_k) != 0)
    return -1;
  return 0;
}

static void teardown(problem_t *p) {
  free(p->seq_q);
  free(p->pos_q);
  free(p->seq_k);
  free(p->pos_k);
}

/* The packed boolean mask M[tq][tk] (total_q x total_k bytes) for a query head
 * (the rule does not depend on the head). */
int oracle_mask(const int32_t *cu_q, const int32_t *cu_k, int batch,
                int total_q, int total_k, int mask_kind, int window,
                unsigned char *m) {
  problem_t p;
  int rc = setup(&p, NULL, NULL, NULL, cu_q, cu_k, batch, total_q, total_k, 1,
                 1, 1, 1.0, mask_kind, window, NULL, NULL, NULL);
  if (rc == 0)
    for (int t = 0; t < total_q; t++)
      for (int u = 0; u < total_k; u++)
        m[(size_t)t * total_k + u] = (unsigned char)pair_allowed(&p, t, u);
  teardown(&p);
  return rc;
}

/* Forward.  rows == NULL: every (token, head) row, o [total_q, hq, d] and lse
 * [hq, total_q].  Otherwise rows holds nrows (token, head) pairs and o is
 * [nrows, d], lse [nrows]. */
int oracle_fwd(const double *q, const double *k, const double *v,
               const int32_t *cu_q, const int32_t *cu_k, int batch,
               int total_q, int total_k, int hq, int hkv, int d, double scale,
               int mask_kind, int window, const double *slopes,
               const double *btab, const int64_t *bstr,
               const int64_t *rows, int64_t nrows, double *o, double *lse) {
  problem_t p;
  int rc = setup(&p, q, k, v, cu_q, cu_k, batch, total_q, total_k, hq, hkv, d,
                 scale, mask_kind, window, slopes, btab, bstr);
  if (rc != 0) {
    teardown(&p);
    return rc;
  }
  int64_t n = rows ? nrows : (int64_t)total_q * hq;
#pragma omp parallel
  {
    unsigned char *mrow = (unsigned char *)malloc((size_t)total_k + 1);
    double *srow = (double *)malloc(sizeof(double) * ((size_t)total_k + 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; r++) {
      int t, h;
      double *orow, *lrow;
      if (rows) {
        t = (int)rows[2 * r];
        h = (int)rows[2 * r + 1];
        orow = o + (size_t)r * d;
        lrow = lse + r;
      } else {
        t = (int)(r / hq);
        h = (int)(r % hq);
        orow = o + ((size_t)t * hq + h) * d;
        lrow = lse + (size_t)h * total_q + t;
      }
      forward_row(&p, t, h, mrow, srow, orow, lrow);
    }
    free(mrow);
    free(srow);
  }
  teardown(&p);
  return 0;
}

/* The contribution of query row (t, h) to the gradients, given its lse and
 * D = dO . O.  dq_row gets scale sum_j dS_ij k_j; when dk_rep / dv_rep are
 * given ([total_k, hq, d], K and V repeated to hq heads), dS and P are added
 * into the rows of head h. */
static void backward_row(const problem_t *p, const double *dout, int t, int h,
                         double lse_i, double D_i, unsigned char *mrow,
                         double *dq_row, double *dk_rep, double *dv_rep) {
  int hk = h / (p->hq / p->hkv);
  const double *qi = q_row(p, t, h);
  const double *doi = dout + ((size_t)t * p->hq + h) * p->d;
  for (int c = 0; c < p->d; c++) dq_row[c] = 0.0;
  if (lse_i == -INFINITY) return; /* empty row: no contribution */
  for (int u = 0; u < p->total_k; u++) mrow[u] = (unsigned char)pair_allowed(p, t, u);
  for (int u = 0; u < p->total_k; u++) {
    if (!mrow[u]) continue;
    const double *kj = k_row(p, u, hk), *vj = v_row(p, u, hk);
    double s = logit(p, qi, kj, t, u, h);
    double pij = exp(s - lse_i);
    double dpij = dot(doi, vj, p->d);
    double ds = pij * (dpij - D_i);
    for (int c = 0; c < p->d; c++) dq_row[c] += p->scale * ds * kj[c];
    if (dk_rep) {
      double *dk = dk_rep + ((size_t)u * p->hq + h) * p->d;
      double *dv = dv_rep + ((size_t)u * p->hq + h) * p->d;
      for (int c = 0; c < p->d; c++) {
        dk[c] += p->scale * ds * qi[c];
        dv[c] += pij * doi[c];
      }
    }
  }
}

/* Full backward: dq [total_q, hq, d], dk and dv [total_k, hkv, d]; o and lse
 * (forward outputs, same layouts as oracle_fwd) are written as well. */
int oracle_bwd(const double *q, const double *k, const double *v,
               const double *dout, const int32_t *cu_q, const int32_t *cu_k,
               int batch, int total_q, int total_k, int hq, int hkv, int d,
               double scale, int mask_kind, int window, const double *slopes,
               const double *btab, const int64_t *bstr,
               double *dq, double *dk, double *dv, double *o, double *lse) {
  int rc = oracle_fwd(q, k, v, cu_q, cu_k, batch, total_q, total_k, hq, hkv, d,
                      scale, mask_kind, window, slopes, btab, bstr, NULL, 0, o, lse);
  if (rc != 0) return rc;
  problem_t p;
  rc = setup(&p, q, k, v, cu_q, cu_k, batch, total_q, total_k, hq, hkv, d,
             scale, mask_kind, window, slopes, btab, bstr);
  if (rc != 0) {
    teardown(&p);
    return rc;
  }
  size_t rep = (size_t)total_k * hq * d;
  double *dk_rep = (double *)calloc(rep + 1, sizeof(double));
  double *dv_rep = (double *)calloc(rep + 1, sizeof(double));
  /* Each query head writes only its own column of the repeated gradients. */
#pragma omp parallel
  {
    unsigned char *mrow = (unsigned char *)malloc((size_t)total_k + 1);
#pragma omp for schedule(dynamic, 1)
    for (int h = 0; h < hq; h++)
      for (int t = 0; t < total_q; t++) {
        const double *oi = o + ((size_t)t * hq + h) * d;
        const double *doi = dout + ((size_t)t * hq + h) * d;
        double D_i = dot(doi, oi, d);
        backward_row(&p, dout, t, h, lse[(size_t)h * total_q + t], D_i, mrow,
                     dq + ((size_t)t * hq + h) * d, dk_rep, dv_rep);
      }
    free(mrow);
  }
  /* Sum the repeated K/V gradients over each group of query heads. */
  int g = hq / hkv;
  for (int u = 0; u < total_k; u++)
    for (int hk = 0; hk < hkv; hk++)
      for (int c = 0; c < d; c++) {
        double sk = 0.0, sv = 0.0;
        for (int r = 0; r < g; r++) {
          sk += dk_rep[((size_t)u * hq + hk * g + r) * d + c];
          sv += dv_rep[((size_t)u * hq + hk * g + r) * d + c];
        }
        dk[((size_t)u * hkv + hk) * d + c] = sk;
        dv[((size_t)u * hkv + hk) * d + c] = sv;
      }
  free(dk_rep);
  free(dv_rep);
  teardown(&p);
  return 0;
}

/* Sampled backward for workloads too large for oracle_bwd: dQ of nq_rows query
 * rows (token, head) -> dq_out [nq_rows, d]; dK and dV of nk_rows key rows
 * (key token, kv head) -> dk_out, dv_out [nk_rows, d].  Every query row that
 * can reach a sampled key (same sequence, a head of its group) is run forward
 * first for its lse and D; nothing else is shared between rows. */
int oracle_bwd_sampled(const double *q, const double *k, const double *v,
                       const double *dout, const int32_t *cu_q,
                       const int32_t *cu_k, int batch, int total_q,
                       int total_k, int hq, int hkv, int d, double scale,
                       int mask_kind, int window, const double *slopes,
                       const double *btab, const int64_t *bstr,
                       const int64_t *q_rows, int64_t nq_rows,
                       double *dq_out, const int64_t *k_rows, int64_t nk_rows,
                       double *dk_out, double *dv_out) {
  problem_t p;
  int rc = setup(&p, q, k, v, cu_q, cu_k, batch, total_q, total_k, hq, hkv, d,
                 scale, mask_kind, window, slopes, btab, bstr);
  if (rc != 0) {
    teardown(&p);
    return rc;
  }
  int g = hq / hkv;
  size_t nrow = (size_t)total_q * hq;
  unsigned char *need = (unsigned char *)calloc(nrow + 1, 1);
  double *lse = (double *)malloc(sizeof(double) * (nrow + 1));
  double *D = (double *)malloc(sizeof(double) * (nrow + 1));
  for (int64_t r = 0; r < nq_rows; r++)
    need[(size_t)q_rows[2 * r] * hq + q_rows[2 * r + 1]] = 1;
  for (int64_t r = 0; r < nk_rows; r++) {
    int u = (int)k_rows[2 * r], hk = (int)k_rows[2 * r + 1];
    for (int t = 0; t < total_q; t++)
      if (pair_allowed(&p, t, u))
        for (int h = hk * g; h < hk * g + g; h++) need[(size_t)t * hq + h] = 1;
  }
#pragma omp parallel
  {
    unsigned char *mrow = (unsigned char *)malloc((size_t)total_k + 1);
    double *srow = (double *)malloc(sizeof(double) * ((size_t)total_k + 1));
    double *orow = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < (int64_t)nrow; r++) {
      if (!need[r]) continue;
      int t = (int)(r / hq), h = (int)(r % hq);
      forward_row(&p, t, h, mrow, srow, orow, &lse[r]);
      D[r] = dot(dout + (size_t)r * d, orow, d);
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < nq_rows; r++) {
      size_t row = (size_t)q_rows[2 * r] * hq + q_rows[2 * r + 1];
      backward_row(&p, dout, (int)q_rows[2 * r], (int)q_rows[2 * r + 1],
                   lse[row], D[row], mrow, dq_out + (size_t)r * d, NULL, NULL);
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < nk_rows; r++) {
      int u = (int)k_rows[2 * r], hk = (int)k_rows[2 * r + 1];
      const double *kj = k_row(&p, u, hk), *vj = v_row(&p, u, hk);
      double *dk = dk_out + (size_t)r * d, *dv = dv_out + (size_t)r * d;
      for (int c = 0; c < d; c++) dk[c] = dv[c] = 0.0;
      for (int h = hk * g; h < hk * g + g; h++)
        for (int t = 0; t < total_q; t++) {
          if (!pair_allowed(&p, t, u)) continue;
          size_t row = (size_t)t * hq + h;
          const double *qi = q_row(&p, t, h);
          const double *doi = dout + row * d;
          if (lse[row] == -INFINITY) continue; /* empty row */
          double s = logit(&p, qi, kj, t, u, h);
          double pij = exp(s - lse[row]);
          double ds = pij * (dot(doi, vj, d) - D[row]);
          for (int c = 0; c < d; c++) {
            dk[c] += scale * ds * qi[c];
            dv[c] += pij * doi[c];
          }
        }
    }
    free(mrow);
    free(srow);
    free(orow);
  }
  free(need);
  free(lse);
  free(D);
  teardown(&p);
  return 0;
}
