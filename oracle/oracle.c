/*
 * oracle.c -- fp64 CPU reference for block-diagonal-causal ("packed") attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do. It shares no code with the CUDA path.
 *
 * What it computes (the plain definition, fp64 throughout):
 *   mlx-train-perf 0.5.1 README, "Sequence packing": a token attends another
 *   only when both belong to the same original sequence, and attention is
 *   causal; the changelog entry adding `flash_attention(segments=...)` states
 *   the mask is driven by an O(N) per-token segment id. "Flash-attention
 *   training path" on the same README: the saved state is the attention output
 *   and its log-sum-exp; the backward recomputes from them.
 *
 *   Vis(i)   = { j <= i : seg[i] == seg[j] }            (seg == NULL: all equal)
 *   S_ij     = s * <q_i, k_j>                          (s = scale)
 *   lse_i    = ln sum_{j in Vis(i)} exp(S_ij)
 *   P_ij     = exp(S_ij - lse_i)
 *   o_i      = sum_{j in Vis(i)} P_ij v_j
 *   D_i      = <dO_i, o_i>
 *   dS_ij    = P_ij (<dO_i, v_j> - D_i)
 *   dq_i     = s sum_{j in Vis(i)} dS_ij k_j
 *   dk_j     = s sum_{h in group(g)} sum_{i : j in Vis(i)} dS_ij q_i
 *   dv_j     = sum_{h in group(g)} sum_{i : j in Vis(i)} P_ij dO_i
 *
 * Grouped-query heads are mapped contiguously (same README, "If you maintain
 * a trainer"): query head h reads kv head h / (Hq / Hkv).
 *
 * lse uses the max-shifted form ln sum exp(S - m) + m, an identity of real
 * arithmetic. Every output row is produced by its own sequential loop, so the
 * result does not depend on the thread count.
 *
 * Layouts: q, dO, o, dq are (B, Hq, N, D); k, v, dk, dv are (B, Hkv, N, D);
 * lse and D are (B, Hq, N); seg is (B, N) int32. All contiguous, row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t B, Hq, Hkv, N, D;
  double scale;
} orc_dims;

static inline int orc_visible(const int32_t* seg_row, int64_t i, int64_t j) {
  if (j > i) return 0;
  if (seg_row == NULL) return 1;
  return seg_row[i] == seg_row[j];
}

static inline double orc_dot(const double* a, const double* b, int64_t n) {
  double acc = 0.0;
  for (int64_t c = 0; c < n; ++c) acc += a[c] * b[c];
  return acc;
}

/* Pointers to the row of head h / kv head g at token i. */
static inline const double* qrow(const orc_dims* m, const double* base, int64_t b, int64_t h, int64_t i) {
  return base + ((b * m->Hq + h) * m->N + i) * m->D;
}
static inline const double* kvrow(const orc_dims* m, const double* base, int64_t b, int64_t g, int64_t i) {
  return base + ((b * m->Hkv + g) * m->N + i) * m->D;
}

/*
 * Forward for one query row (b, h, i): writes o_i (D values), lse_i, and, when
 * dout != NULL, D_i = <dO_i, o_i>. `sbuf` holds N doubles of scratch.
 */
static void orc_fwd_row(const orc_dims* m, const double* q, const double* k, const double* v,
                        const int32_t* seg, const double* dout, int64_t b, int64_t h, int64_t i,
                        double* o_out, double* lse_out, double* delta_out, double* sbuf) {
  const int64_t G = m->Hq / m->Hkv, g = h / G, D = m->D;
  const int32_t* srow = seg ? seg + b * m->N : NULL;
  const double* qi = qrow(m, q, b, h, i);
  double mx = -INFINITY;
  for (int64_t j = 0; j <= i; ++j) {
    if (!orc_visible(srow, i, j)) continue;
    double s = m->scale * orc_dot(qi, kvrow(m, k, b, g, j), D);
    sbuf[j] = s;
    if (s > mx) mx = s;
  }
  double sum = 0.0;
  for (int64_t j = 0; j <= i; ++j)
    if (orc_visible(srow, i, j)) sum += exp(sbuf[j] - mx);
  const double lse = mx + log(sum);
  for (int64_t c = 0; c < D; ++c) o_out[c] = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    if (!orc_visible(srow, i, j)) continue;
    const double p = exp(sbuf[j] - lse);
    const double* vj = kvrow(m, v, b, g, j);
    for (int64_t c = 0; c < D; ++c) o_out[c] += p * vj[c];
  }
  *lse_out = lse;
  if (dout && delta_out) *delta_out = orc_dot(qrow(m, dout, b, h, i), o_out, D);
}

/* dq_i for one query row; lse and delta are full (B, Hq, N) arrays. */
static void orc_dq_row(const orc_dims* m, const double* q, const double* k, const double* v,
                       const int32_t* seg, const double* dout, const double* lse,
                       const double* delta, int64_t b, int64_t h, int64_t i, double* dq_out) {
  const int64_t G = m->Hq / m->Hkv, g = h / G, D = m->D;
  const int32_t* srow = seg ? seg + b * m->N : NULL;
  const int64_t r = (b * m->Hq + h) * m->N + i;
  const double* qi = qrow(m, q, b, h, i);
  const double* doi = qrow(m, dout, b, h, i);
  for (int64_t c = 0; c < D; ++c) dq_out[c] = 0.0;
  for (int64_t j = 0; j <= i; ++j) {
    if (!orc_visible(srow, i, j)) continue;
    const double* kj = kvrow(m, k, b, g, j);
    const double p = exp(m->scale * orc_dot(qi, kj, D) - lse[r]);
    const double ds = p * (orc_dot(doi, kvrow(m, v, b, g, j), D) - delta[r]);
    for (int64_t c = 0; c < D; ++c) dq_out[c] += ds * kj[c];
  }
  for (int64_t c = 0; c < D; ++c) dq_out[c] *= m->scale;
}

/* dk_j, dv_j for one key row (b, g, j): sums over the group's query heads and
 * every query row i that sees j. */
static void orc_dkv_row(const orc_dims* m, const double* q, const double* k, const double* v,
                        const int32_t* seg, const double* dout, const double* lse,
                        const double* delta, int64_t b, int64_t g, int64_t j, double* dk_out,
                        double* dv_out) {
  const int64_t G = m->Hq / m->Hkv, D = m->D;
  const int32_t* srow = seg ? seg + b * m->N : NULL;
  const double* kj = kvrow(m, k, b, g, j);
  const double* vj = kvrow(m, v, b, g, j);
  for (int64_t c = 0; c < D; ++c) { dk_out[c] = 0.0; dv_out[c] = 0.0; }
  for (int64_t h = g * G; h < (g + 1) * G; ++h) {
    for (int64_t i = j; i < m->N; ++i) {
      if (!orc_visible(srow, i, j)) continue;
      const int64_t r = (b * m->Hq + h) * m->N + i;
      const double* qi = qrow(m, q, b, h, i);
      const double* doi = qrow(m, dout, b, h, i);
      const double p = exp(m->scale * orc_dot(qi, kj, D) - lse[r]);
      const double ds = p * (orc_dot(doi, vj, D) - delta[r]);
      for (int64_t c = 0; c < D; ++c) {
        dv_out[c] += p * doi[c];
        dk_out[c] += ds * qi[c];
      }
    }
  }
  for (int64_t c = 0; c < D; ++c) dk_out[c] *= m->scale;
}

/* ------------------------------------------------------------------------ */
/* exported: row lists (flat row index r = (b*H + h)*N + i)                 */
/* ------------------------------------------------------------------------ */

/* Forward for `nrows` query rows. out: nrows x D, lse/delta: nrows. */
void orc_fwd_rows(const orc_dims* m, const double* q, const double* k, const double* v,
                  const int32_t* seg, const double* dout, int64_t nrows, const int64_t* rows,
                  double* out, double* lse, double* delta) {
#pragma omp parallel
  {
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)m->N);
#pragma omp for schedule(dynamic, 8)
    for (int64_t t = 0; t < nrows; ++t) {
      const int64_t r = rows[t];
      const int64_t i = r % m->N, bh = r / m->N, h = bh % m->Hq, b = bh / m->Hq;
      orc_fwd_row(m, q, k, v, seg, dout, b, h, i, out + t * m->D, lse + t,
                  delta ? delta + t : NULL, sbuf);
    }
    free(sbuf);
  }
}

/* dq for `nrows` query rows (flat index over (B, Hq, N)); out: nrows x D. */
void orc_dq_rows(const orc_dims* m, const double* q, const double* k, const double* v,
                 const int32_t* seg, const double* dout, const double* lse, const double* delta,
                 int64_t nrows, const int64_t* rows, double* dq) {
#pragma omp parallel for schedule(dynamic, 8)
  for (int64_t t = 0; t < nrows; ++t) {
    const int64_t r = rows[t];
    const int64_t i = r % m->N, bh = r / m->N, h = bh % m->Hq, b = bh / m->Hq;
    orc_dq_row(m, q, k, v, seg, dout, lse, delta, b, h, i, dq + t * m->D);
  }
}

/* dk, dv for `nrows` key rows (flat index over (B, Hkv, N)); out: nrows x D each. */
void orc_dkv_rows(const orc_dims* m, const double* q, const double* k, const double* v,
                  const int32_t* seg, const double* dout, const double* lse, const double* delta,
                  int64_t nrows, const int64_t* rows, double* dk, double* dv) {
#pragma omp parallel for schedule(dynamic, 8)
  for (int64_t t = 0; t < nrows; ++t) {
    const int64_t r = rows[t];
    const int64_t j = r % m->N, bg = r / m->N, g = bg % m->Hkv, b = bg / m->Hkv;
    orc_dkv_row(m, q, k, v, seg, dout, lse, delta, b, g, j, dk + t * m->D, dv + t * m->D);
  }
}

int orc_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      extern int omp_get_num_threads(void);
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
