/*
 * mla_oracle.c -- plain fp64 CPU reference for replay attention over latent (MLA-style)
 * pages.
 *
 * TEST INFRASTRUCTURE ONLY (see longstraw_oracle.c): used by the tests, the smoke check
 * and the benchmark's CPU-baseline leg; the product library never links or calls it.
 *
 * The LongStraw explainer ("LongStraw: fitting million-token RL onto a fixed GPU
 * budget", section "Two incompatible architectures, same transaction", GLM bullet) keeps
 * the GLM model's multi-head latent attention state as CPU-resident latent pages and
 * replays each response over them; the pages give no equations for the layer.  The
 * attention is taken from the DeepSeek-V2 paper (Multi-head Latent Attention, "DeepSeek-V2:
 * A Strong, Economical, and Efficient Mixture-of-Experts Language Model", 2024) in the
 * form used when the key up-projection is absorbed into the query: every position j
 * keeps one row shared by all heads, its compressed latent c_j (d_c values) followed by
 * its decoupled rotary key r_j (d_r values); head h of token t brings an absorbed query
 * q_{t,h} of d_c + d_r values, and
 *   s_{t,h,j} = scale * <q_{t,h}, [c_j ; r_j]>,   j over the P prompt positions and the
 *               response positions j <= t
 *   lse_{t,h} = log sum_j exp(s_{t,h,j}),   o_{t,h} = sum_j exp(s_{t,h,j} - lse_{t,h}) c_j
 * (the value up-projection and output projection are weights, applied by the caller).
 * The prompt rows are stopgrad, as for the other attention layers.
 *
 * Written as the plain definition, one row at a time over all its keys: no splits, no
 * online rescaling.
 */
#include "longstraw_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double mla_bf16(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int mla_check(const lso_mla* a) {
  if (!a || a->R < 0 || a->H < 1 || a->d_c < 1 || a->d_r < 0 || a->P < 0) return 1;
  if (a->P > 0) {
    if (a->page_size < 1 || !a->page_table || !a->lat_pool) return 1;
    if (a->P > a->num_logical_pages * (int64_t)a->page_size) return 1;
  }
  if (a->R > 0 && (!a->q || !a->lat_resp)) return 1;
  return 0;
}

/* Latent row of key j of row (t): prompt position j < P through the page table, else
 * response position j - P.  NULL for a page id outside the pool. */
static const uint16_t* mla_key_row(const lso_mla* a, int64_t j) {
  const int64_t D = a->d_c + a->d_r;
  if (j < a->P) {
    const int32_t page = a->page_table[j / a->page_size];
    if (page < 0 || page >= a->num_pages) return NULL;
    return a->lat_pool + ((int64_t)page * a->page_size + j % a->page_size) * D;
  }
  return a->lat_resp + (j - a->P) * D;
}

/* One query row (t, h): o [d_c], lse.  Returns 0, or 1 for a bad page id. */
static int mla_row(const lso_mla* a, int32_t t, int32_t h, double* s, double* o, double* lse) {
  const int64_t D = a->d_c + a->d_r, nk = a->P + t + 1;
  const uint16_t* q = a->q + ((int64_t)t * a->H + h) * D;
  double m = -INFINITY;
  for (int64_t j = 0; j < nk; ++j) {
    const uint16_t* row = mla_key_row(a, j);
    if (!row) return 1;
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += mla_bf16(q[d]) * mla_bf16(row[d]);
    s[j] = a->scale * acc;
    if (s[j] > m) m = s[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j < nk; ++j) sum += exp(s[j] - m);
  for (int32_t d = 0; d < a->d_c; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < nk; ++j) {
    const double w = exp(s[j] - m) / sum;
    const uint16_t* row = mla_key_row(a, j);
    for (int32_t d = 0; d < a->d_c; ++d) o[d] += w * mla_bf16(row[d]);
  }
  *lse = m + log(sum);
  return 0;
}

static int mla_rows(const lso_mla* a, int32_t n, const int32_t* ts, const int32_t* hs,
                    double* o, double* lse) {
  int bad = 0, oom = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(a->P + a->R + 1));
    if (!s) {
#pragma omp atomic write
      oom = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int32_t i = 0; i < n; ++i) {
      const int32_t t = ts ? ts[i] : i / a->H, h = hs ? hs[i] : i % a->H;
      if (!s) continue;
      if (t < 0 || t >= a->R || h < 0 || h >= a->H ||
          mla_row(a, t, h, s, o + (int64_t)i * a->d_c, lse + i)) {
#pragma omp atomic write
        bad = 1;
      }
    }
    free(s);
  }
  return oom ? 2 : (bad ? 1 : 0);
}

int lso_mla_fwd(const lso_mla* a, double* o, double* lse) {
  if (mla_check(a) || !o || !lse) return 1;
  return mla_rows(a, a->R * a->H, NULL, NULL, o, lse);
}

int lso_mla_fwd_rows(const lso_mla* a, int32_t n, const int32_t* ts, const int32_t* hs,
                     double* o, double* lse) {
  if (mla_check(a) || n < 0 || !ts || !hs || (n > 0 && (!o || !lse))) return 1;
  return mla_rows(a, n, ts, hs, o, lse);
}

/*
 * Backward.  The prompt rows are stopgrad, so the gradients are dq for every query row
 * and d lat_j for the response's own rows j only.  With the row's exact forward (o, lse
 * as above) and its output gradient dO_{t,h} (d_c values):
 *   P_{t,h,j}  = exp(s_{t,h,j} - lse_{t,h})
 *   D_{t,h}    = <dO_{t,h}, o_{t,h}>
 *   dP_{t,h,j} = <dO_{t,h}, c_j>               (c_j: the row's first d_c values)
 *   dS_{t,h,j} = P_{t,h,j} (dP_{t,h,j} - D_{t,h})
 *   dq_{t,h}   = scale sum_j dS_{t,h,j} [c_j ; r_j]          over every visible j
 *   d lat_j    = sum_{t >= j} sum_h ( P_{t,h,j} [dO_{t,h} ; 0]
 *                                     + scale dS_{t,h,j} q_{t,h} )   response rows j
 * (the latent c_j is both a key and a value, so its gradient has both terms; the rotary
 * part r_j only the key term).  This is the chain rule through the forward's three steps
 * (the product, the softmax, the weighted sum), written for one row at a time.
 */

/* One query row (t, h): exact forward, then dq [D] (NULL: skipped), lse and D.
 * Returns 0, or 1 for a bad page id. */
static int mla_row_bwd(const lso_mla* a, int32_t t, int32_t h, const uint16_t* d_o,
                       double* s, double* o, double* dq, double* lse, double* dd) {
  const int64_t D = a->d_c + a->d_r, nk = a->P + t + 1;
  if (mla_row(a, t, h, s, o, lse)) return 1;
  const uint16_t* g = d_o + ((int64_t)t * a->H + h) * a->d_c;
  double dot = 0.0;
  for (int32_t d = 0; d < a->d_c; ++d) dot += mla_bf16(g[d]) * o[d];
  *dd = dot;
  if (!dq) return 0;
  for (int64_t d = 0; d < D; ++d) dq[d] = 0.0;
  for (int64_t j = 0; j < nk; ++j) {
    const uint16_t* row = mla_key_row(a, j);
    double dp = 0.0;
    for (int32_t d = 0; d < a->d_c; ++d) dp += mla_bf16(g[d]) * mla_bf16(row[d]);
    const double ds = exp(s[j] - *lse) * (dp - dot);
    for (int64_t d = 0; d < D; ++d) dq[d] += a->scale * ds * mla_bf16(row[d]);
  }
  return 0;
}

/* Pass 1 over the rows (t, h) with t >= t0: dq (NULL: skipped; else [R][H][D], rows
 * before t0 untouched), lse and D into lse_all / d_all ([R][H]). */
static int mla_bwd_rows_pass(const lso_mla* a, const uint16_t* d_o, int32_t t0, double* dq,
                             double* lse_all, double* d_all) {
  const int64_t D = a->d_c + a->d_r;
  const int32_t n = (a->R - t0) * a->H;
  int bad = 0, oom = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(a->P + a->R + 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)a->d_c);
    if (!s || !o) {
#pragma omp atomic write
      oom = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int32_t i = 0; i < n; ++i) {
      const int32_t t = t0 + i / a->H, h = i % a->H;
      const int64_t r = (int64_t)t * a->H + h;
      if (!s || !o) continue;
      if (mla_row_bwd(a, t, h, d_o, s, o, dq ? dq + r * D : NULL, lse_all + r, d_all + r)) {
#pragma omp atomic write
        bad = 1;
      }
    }
    free(s);
    free(o);
  }
  return oom ? 2 : (bad ? 1 : 0);
}

/* d lat_j [D] of response row j from the rows' lse and D (rows t >= j). */
static void mla_dlat_key(const lso_mla* a, const uint16_t* d_o, int32_t j,
                         const double* lse_all, const double* d_all, double* out) {
  const int64_t D = a->d_c + a->d_r;
  const uint16_t* row = a->lat_resp + (int64_t)j * D;
  for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
  for (int32_t t = j; t < a->R; ++t) {
    for (int32_t h = 0; h < a->H; ++h) {
      const int64_t r = (int64_t)t * a->H + h;
      const uint16_t* q = a->q + r * D;
      const uint16_t* g = d_o + r * a->d_c;
      double acc = 0.0, dp = 0.0;
      for (int64_t d = 0; d < D; ++d) acc += mla_bf16(q[d]) * mla_bf16(row[d]);
      for (int32_t d = 0; d < a->d_c; ++d) dp += mla_bf16(g[d]) * mla_bf16(row[d]);
      const double p = exp(a->scale * acc - lse_all[r]);
      const double ds = p * (dp - d_all[r]);
      for (int32_t d = 0; d < a->d_c; ++d) out[d] += p * mla_bf16(g[d]);
      for (int64_t d = 0; d < D; ++d) out[d] += a->scale * ds * mla_bf16(q[d]);
    }
  }
}

int lso_mla_bwd(const lso_mla* a, const uint16_t* d_o, double* dq, double* dlat) {
  if (mla_check(a) || (a->R > 0 && (!d_o || !dq || !dlat))) return 1;
  if (a->R == 0) return 0;
  const int64_t D = a->d_c + a->d_r, rows = (int64_t)a->R * a->H;
  double* lse_all = (double*)malloc(sizeof(double) * (size_t)rows);
  double* d_all = (double*)malloc(sizeof(double) * (size_t)rows);
  int rc = (!lse_all || !d_all) ? 2 : mla_bwd_rows_pass(a, d_o, 0, dq, lse_all, d_all);
  if (rc == 0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t j = 0; j < a->R; ++j) mla_dlat_key(a, d_o, j, lse_all, d_all, dlat + j * D);
  }
  free(lse_all);
  free(d_all);
  return rc;
}

int lso_mla_bwd_dq_rows(const lso_mla* a, const uint16_t* d_o, int32_t n, const int32_t* ts,
                        const int32_t* hs, double* dq) {
  if (mla_check(a) || n < 0 || (n > 0 && (!d_o || !ts || !hs || !dq))) return 1;
  const int64_t D = a->d_c + a->d_r;
  int bad = 0, oom = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(a->P + a->R + 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)a->d_c);
    if (!s || !o) {
#pragma omp atomic write
      oom = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int32_t i = 0; i < n; ++i) {
      double lse, dd;
      if (!s || !o) continue;
      if (ts[i] < 0 || ts[i] >= a->R || hs[i] < 0 || hs[i] >= a->H ||
          mla_row_bwd(a, ts[i], hs[i], d_o, s, o, dq + (int64_t)i * D, &lse, &dd)) {
#pragma omp atomic write
        bad = 1;
      }
    }
    free(s);
    free(o);
  }
  return oom ? 2 : (bad ? 1 : 0);
}

int lso_mla_bwd_dlat_keys(const lso_mla* a, const uint16_t* d_o, int32_t n, const int32_t* js,
                          double* dlat) {
  if (mla_check(a) || n < 0 || (n > 0 && (!d_o || !js || !dlat))) return 1;
  if (n == 0) return 0;
  int32_t j0 = a->R;
  for (int32_t i = 0; i < n; ++i) {
    if (js[i] < 0 || js[i] >= a->R) return 1;
    if (js[i] < j0) j0 = js[i];
  }
  const int64_t D = a->d_c + a->d_r, rows = (int64_t)a->R * a->H;
  double* lse_all = (double*)malloc(sizeof(double) * (size_t)rows);
  double* d_all = (double*)malloc(sizeof(double) * (size_t)rows);
  int rc = (!lse_all || !d_all) ? 2 : mla_bwd_rows_pass(a, d_o, j0, NULL, lse_all, d_all);
  if (rc == 0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < n; ++i) mla_dlat_key(a, d_o, js[i], lse_all, d_all, dlat + i * D);
  }
  free(lse_all);
  free(d_all);
  return rc;
}
