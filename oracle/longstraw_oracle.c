/*
 * longstraw_oracle.c -- plain fp64 CPU reference for the response-replay hot path.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the benchmark's
 * CPU-baseline leg.  The product library never links or calls it and the two share
 * no code.  Deliberately slow and literal: no blocking, no fusion, no reordering
 * beyond what each definition states.  OpenMP only runs independent rows (or keys,
 * or tokens) in parallel; every row is computed by one thread in a fixed order, so
 * results do not depend on the thread count.
 *
 * The definitions followed are cited per function (page titles and sections of the
 * LongStraw pages; see longstraw_oracle.h for the full list).
 */
#include "longstraw_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int lso_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- widening */

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* dst[0..n) = exact widening of elements [off, off + n) of an array of type dtype. */
static void load_vec(double* dst, const void* base, int64_t off, int n, int dtype) {
  int i;
  if (dtype == LSO_BF16) {
    const uint16_t* p = (const uint16_t*)base + off;
    for (i = 0; i < n; ++i) dst[i] = bf16_bits_to_double(p[i]);
  } else if (dtype == LSO_F32) {
    const float* p = (const float*)base + off;
    for (i = 0; i < n; ++i) dst[i] = (double)p[i];
  } else {
    const double* p = (const double*)base + off;
    for (i = 0; i < n; ++i) dst[i] = p[i];
  }
}

static double load_one(const void* base, int64_t off, int dtype) {
  double x;
  load_vec(&x, base, off, 1, dtype);
  return x;
}

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  int i;
  for (i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* ---------------------------------------------------------------- capture */

/* Prompt capture writes the prompt's K/V once into resident pages (digest, Method
 * step 1; explainer, "The move: change the graph boundary").  Written as the literal
 * loop: pool[pt[p / ps]][h][p % ps][:] = src[p - start][h][:]. */
int lso_capture_kv(uint16_t* k_pool, uint16_t* v_pool, const int32_t* page_table,
                   int64_t num_pages, int64_t num_logical_pages, int32_t page_size,
                   int32_t hkv, int32_t d, const uint16_t* k, const uint16_t* v,
                   int64_t start_pos, int64_t n) {
  int64_t p;
  int h, e;
  if (page_size <= 0 || hkv <= 0 || d <= 0 || start_pos < 0 || n < 0) return 1;
  for (p = start_pos; p < start_pos + n; ++p) {
    int64_t logical = p / page_size;
    int64_t slot = p % page_size;
    int64_t phys;
    if (logical >= num_logical_pages) return 1;
    phys = page_table[logical];
    if (phys < 0 || phys >= num_pages) return 1;
    for (h = 0; h < hkv; ++h) {
      for (e = 0; e < d; ++e) {
        int64_t dst = ((phys * hkv + h) * page_size + slot) * d + e;
        int64_t src = ((p - start_pos) * hkv + h) * d + e;
        k_pool[dst] = k[src];
        v_pool[dst] = v[src];
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------- attention */

static int attn_check(const lso_attn* a) {
  int64_t lp;
  if (a->hkv <= 0 || a->hq <= 0 || a->d <= 0 || a->R < 0 || a->P < 0) return 1;
  if (a->hq % a->hkv != 0) return 1;
  if (a->P > 0) {
    if (a->page_size <= 0 || a->num_splits <= 0) return 1;
    if ((a->P + a->page_size - 1) / a->page_size > a->num_logical_pages) return 1;
    for (lp = 0; lp < (a->P + a->page_size - 1) / a->page_size; ++lp)
      if (a->page_table[lp] < 0 || a->page_table[lp] >= a->num_pages) return 1;
  }
  return 0;
}

static int64_t prompt_pages(const lso_attn* a) {
  return a->P > 0 ? (a->P + a->page_size - 1) / a->page_size : 0;
}

/* Element offset of prompt key/value `pos` of kv head kvh in the page pool. */
static int64_t pool_offset(const lso_attn* a, int64_t pos, int kvh) {
  int64_t logical = pos / a->page_size;
  int64_t slot = pos % a->page_size;
  int64_t phys = a->page_table[logical];
  return ((phys * a->hkv + kvh) * a->page_size + slot) * a->d;
}

static int64_t resp_offset(const lso_attn* a, int64_t j, int kvh) {
  return (j * a->hkv + kvh) * a->d;
}

/* Per-thread scratch for one row. */
typedef struct {
  double* qd;     /* [d] */
  double* kd;     /* [d] */
  double* acc;    /* [d] */
  double* scores; /* [max keys in one partial] */
  double* part_o; /* [(num_splits + 1) * d] */
  double* part_lse;
} row_scratch;

static int64_t max_partial_keys(const lso_attn* a) {
  int64_t pages = prompt_pages(a);
  int64_t per_split = a->num_splits > 0 ? (pages + a->num_splits - 1) / a->num_splits : 0;
  int64_t m = per_split * (a->page_size > 0 ? a->page_size : 0);
  if (a->R > m) m = a->R;
  return m > 0 ? m : 1;
}

static int scratch_alloc(const lso_attn* a, row_scratch* s) {
  int ns = (a->num_splits > 0 ? a->num_splits : 1) + 1;
  s->qd = (double*)malloc(sizeof(double) * a->d);
  s->kd = (double*)malloc(sizeof(double) * a->d);
  s->acc = (double*)malloc(sizeof(double) * a->d);
  s->scores = (double*)malloc(sizeof(double) * max_partial_keys(a));
  s->part_o = (double*)malloc(sizeof(double) * a->d * ns);
  s->part_lse = (double*)malloc(sizeof(double) * ns);
  return s->qd && s->kd && s->acc && s->scores && s->part_o && s->part_lse ? 0 : 2;
}

static void scratch_free(row_scratch* s) {
  free(s->qd);
  free(s->kd);
  free(s->acc);
  free(s->scores);
  free(s->part_o);
  free(s->part_lse);
}

/* Softmax partial of query qd over one contiguous set of keys: either prompt
 * positions [pos0, pos1) read through the page table, or response keys [0, pos1)
 * when `response` is set.  Writes lse_out = log sum_j exp(s_j) and the normalised
 * o_out = sum_j exp(s_j - lse_out) v_j; an empty set gives lse_out = -inf, o_out = 0.
 * s_j = scale * <q, k_j> (explainer, "Serial replay makes G a schedule": the
 * response graph attends to the whole captured prompt; digest, Qwen implementation:
 * exact attention over the KV pages). */
static void softmax_partial(const lso_attn* a, row_scratch* s, int kvh, int response,
                            int64_t pos0, int64_t pos1, double* o_out, double* lse_out) {
  int64_t n = pos1 - pos0, i;
  double m = -INFINITY, l = 0.0;
  int e;
  if (n <= 0) {
    *lse_out = -INFINITY;
    for (e = 0; e < a->d; ++e) o_out[e] = 0.0;
    return;
  }
  for (i = 0; i < n; ++i) {
    if (response)
      load_vec(s->kd, a->k_resp, resp_offset(a, pos0 + i, kvh), a->d, a->in_dtype);
    else
      load_vec(s->kd, a->k_pool, pool_offset(a, pos0 + i, kvh), a->d, a->pool_dtype);
    s->scores[i] = a->scale * dot(s->qd, s->kd, a->d);
    if (s->scores[i] > m) m = s->scores[i];
  }
  for (e = 0; e < a->d; ++e) s->acc[e] = 0.0;
  for (i = 0; i < n; ++i) {
    double w = exp(s->scores[i] - m);
    l += w;
    if (response)
      load_vec(s->kd, a->v_resp, resp_offset(a, pos0 + i, kvh), a->d, a->in_dtype);
    else
      load_vec(s->kd, a->v_pool, pool_offset(a, pos0 + i, kvh), a->d, a->pool_dtype);
    for (e = 0; e < a->d; ++e) s->acc[e] += w * s->kd[e];
  }
  *lse_out = m + log(l);
  for (e = 0; e < a->d; ++e) o_out[e] = s->acc[e] / l;
}

/* One output row (t, h).  The prompt is cut into num_splits ranges of whole pages
 * and the response keys 0..t (causal, diagonal included) form one more range; each
 * range yields (lse_s, o_s) and the ranges are composed by log-sum-exp, the merge
 * the explainer describes as composing rank-local softmax statistics into the
 * exact global attention output ("Two incompatible architectures", Qwen bullet):
 *   lse = log sum_s exp(lse_s),  o = sum_s exp(lse_s - lse) o_s. */
static void fwd_row(const lso_attn* a, row_scratch* s, int t, int h, double* o, double* lse) {
  int g = a->hq / a->hkv, kvh = h / g, np = 0, i, e;
  int64_t pages = prompt_pages(a);
  double mx = -INFINITY, sum = 0.0, L;
  load_vec(s->qd, a->q, ((int64_t)t * a->hq + h) * a->d, a->d, a->in_dtype);
  if (a->P > 0) {
    int64_t pps = (pages + a->num_splits - 1) / a->num_splits;
    int sp;
    for (sp = 0; sp < a->num_splits; ++sp) {
      int64_t p0 = (int64_t)sp * pps * a->page_size;
      int64_t p1 = (int64_t)(sp + 1) * pps * a->page_size;
      if (p0 > a->P) p0 = a->P;
      if (p1 > a->P) p1 = a->P;
      softmax_partial(a, s, kvh, 0, p0, p1, s->part_o + (int64_t)np * a->d, &s->part_lse[np]);
      ++np;
    }
  }
  softmax_partial(a, s, kvh, 1, 0, (int64_t)t + 1, s->part_o + (int64_t)np * a->d,
                  &s->part_lse[np]);
  ++np;
  for (i = 0; i < np; ++i)
    if (s->part_lse[i] > mx) mx = s->part_lse[i];
  for (i = 0; i < np; ++i)
    if (s->part_lse[i] > -INFINITY) sum += exp(s->part_lse[i] - mx);
  L = mx + log(sum);
  for (e = 0; e < a->d; ++e) o[e] = 0.0;
  for (i = 0; i < np; ++i) {
    double w;
    if (!(s->part_lse[i] > -INFINITY)) continue;
    w = exp(s->part_lse[i] - L);
    for (e = 0; e < a->d; ++e) o[e] += w * s->part_o[(int64_t)i * a->d + e];
  }
  *lse = L;
}

int lso_attn_fwd_rows(const lso_attn* a, int32_t n, const int32_t* ts, const int32_t* hs,
                      double* o, double* lse) {
  int err = attn_check(a), i;
  if (err) return err;
  for (i = 0; i < n; ++i)
    if (ts[i] < 0 || ts[i] >= a->R || hs[i] < 0 || hs[i] >= a->hq) return 1;
#pragma omp parallel
  {
    row_scratch s;
    int ok = scratch_alloc(a, &s) == 0;
    int r;
    if (!ok) {
#pragma omp atomic write
      err = 2;
    }
#pragma omp for schedule(dynamic, 1)
    for (r = 0; r < n; ++r)
      if (ok) fwd_row(a, &s, ts[r], hs[r], o + (int64_t)r * a->d, &lse[r]);
    scratch_free(&s);
  }
  return err;
}

int lso_attn_fwd(const lso_attn* a, double* o, double* lse) {
  int err = attn_check(a);
  int64_t rows = (int64_t)a->R * a->hq;
  if (err) return err;
#pragma omp parallel
  {
    row_scratch s;
    int ok = scratch_alloc(a, &s) == 0;
    int64_t r;
    if (!ok) {
#pragma omp atomic write
      err = 2;
    }
#pragma omp for schedule(dynamic, 1)
    for (r = 0; r < rows; ++r)
      if (ok) fwd_row(a, &s, (int)(r / a->hq), (int)(r % a->hq), o + r * a->d, &lse[r]);
    scratch_free(&s);
  }
  return err;
}

/* dQ of one row given its own forward statistics.  The prompt state is stopgrad
 * (digest, Method, last paragraph: only d(loss)/d(theta) at the captured state is
 * taken), so dQ is the only gradient the prompt keys feed:
 *   P_j  = exp(s_j - lse),  dP_j = <dO, v_j>,  D = <dO, O>,
 *   dS_j = P_j (dP_j - D),  dQ = scale * sum_j dS_j k_j
 * over every prompt key and the response keys j <= t. */
static void dq_row(const lso_attn* a, row_scratch* s, const double* dod, double D, double lse,
                   int t, int h, double* dq) {
  int g = a->hq / a->hkv, kvh = h / g, e;
  int64_t j;
  load_vec(s->qd, a->q, ((int64_t)t * a->hq + h) * a->d, a->d, a->in_dtype);
  for (e = 0; e < a->d; ++e) dq[e] = 0.0;
  for (j = 0; j < a->P + t + 1; ++j) {
    int response = j >= a->P;
    int64_t koff = response ? resp_offset(a, j - a->P, kvh) : pool_offset(a, j, kvh);
    double sc, p, dp, ds;
    load_vec(s->kd, response ? a->k_resp : a->k_pool, koff, a->d,
             response ? a->in_dtype : a->pool_dtype);
    sc = a->scale * dot(s->qd, s->kd, a->d);
    p = exp(sc - lse);
    load_vec(s->acc, response ? a->v_resp : a->v_pool, koff, a->d,
             response ? a->in_dtype : a->pool_dtype);
    dp = dot(dod, s->acc, a->d);
    ds = p * (dp - D);
    for (e = 0; e < a->d; ++e) dq[e] += a->scale * ds * s->kd[e];
  }
}

int lso_attn_bwd_dq_rows(const lso_attn* a, const void* d_o, int32_t do_dtype, int32_t n,
                         const int32_t* ts, const int32_t* hs, double* dq) {
  int err = attn_check(a), i;
  if (err) return err;
  for (i = 0; i < n; ++i)
    if (ts[i] < 0 || ts[i] >= a->R || hs[i] < 0 || hs[i] >= a->hq) return 1;
#pragma omp parallel
  {
    row_scratch s;
    int ok = scratch_alloc(a, &s) == 0;
    double* o = (double*)malloc(sizeof(double) * a->d);
    double* dod = (double*)malloc(sizeof(double) * a->d);
    int r;
    if (!ok || !o || !dod) {
      ok = 0;
#pragma omp atomic write
      err = 2;
    }
#pragma omp for schedule(dynamic, 1)
    for (r = 0; r < n; ++r) {
      double lse, D;
      if (!ok) continue;
      fwd_row(a, &s, ts[r], hs[r], o, &lse);
      load_vec(dod, d_o, ((int64_t)ts[r] * a->hq + hs[r]) * a->d, a->d, do_dtype);
      D = dot(dod, o, a->d);
      dq_row(a, &s, dod, D, lse, ts[r], hs[r], dq + (int64_t)r * a->d);
    }
    free(o);
    free(dod);
    scratch_free(&s);
  }
  return err;
}

/* dK_j, dV_j of response key j (kv head kvh): keys exist only where the response
 * touches them (explainer, "Two incompatible architectures": K/V gradient pages are
 * allocated only when a response backward touches them), summed over the query
 * heads sharing the kv head and the rows t >= j that see key j:
 *   dK_j = scale * sum_{h, t >= j} dS_{t,j} q_t,   dV_j = sum_{h, t >= j} P_{t,j} dO_t.
 * lse_rows / d_rows hold each row's forward statistics ([R][hq]). */
static void dkdv_key(const lso_attn* a, row_scratch* s, const void* d_o, int do_dtype,
                     const double* lse_rows, const double* d_rows, int j, int kvh, double* dk,
                     double* dv, double* dod) {
  int g = a->hq / a->hkv, h, t, e;
  double* vd = s->acc;
  for (e = 0; e < a->d; ++e) dk[e] = dv[e] = 0.0;
  load_vec(s->kd, a->k_resp, resp_offset(a, j, kvh), a->d, a->in_dtype);
  load_vec(vd, a->v_resp, resp_offset(a, j, kvh), a->d, a->in_dtype);
  for (h = kvh * g; h < (kvh + 1) * g; ++h) {
    for (t = j; t < a->R; ++t) {
      int64_t row = (int64_t)t * a->hq + h;
      double sc, p, dp, ds;
      load_vec(s->qd, a->q, row * a->d, a->d, a->in_dtype);
      load_vec(dod, d_o, row * a->d, a->d, do_dtype);
      sc = a->scale * dot(s->qd, s->kd, a->d);
      p = exp(sc - lse_rows[row]);
      dp = dot(dod, vd, a->d);
      ds = p * (dp - d_rows[row]);
      for (e = 0; e < a->d; ++e) {
        dk[e] += a->scale * ds * s->qd[e];
        dv[e] += p * dod[e];
      }
    }
  }
}

/* Forward statistics (lse, D = <dO, O>) of every row (t, h) with t >= t_min. */
static int row_stats(const lso_attn* a, const void* d_o, int do_dtype, int t_min,
                     double* lse_rows, double* d_rows) {
  int err = 0;
  int64_t rows = (int64_t)a->R * a->hq;
#pragma omp parallel
  {
    row_scratch s;
    int ok = scratch_alloc(a, &s) == 0;
    double* o = (double*)malloc(sizeof(double) * a->d);
    double* dod = (double*)malloc(sizeof(double) * a->d);
    int64_t r;
    if (!ok || !o || !dod) {
      ok = 0;
#pragma omp atomic write
      err = 2;
    }
#pragma omp for schedule(dynamic, 1)
    for (r = (int64_t)t_min * a->hq; r < rows; ++r) {
      if (!ok) continue;
      fwd_row(a, &s, (int)(r / a->hq), (int)(r % a->hq), o, &lse_rows[r]);
      load_vec(dod, d_o, r * a->d, a->d, do_dtype);
      d_rows[r] = dot(dod, o, a->d);
    }
    free(o);
    free(dod);
    scratch_free(&s);
  }
  return err;
}

int lso_attn_bwd_dkdv_keys(const lso_attn* a, const void* d_o, int32_t do_dtype, int32_t n,
                           const int32_t* js, const int32_t* kvhs, double* dk, double* dv) {
  int err = attn_check(a), i, jmin = a->R;
  double *lse_rows, *d_rows;
  if (err) return err;
  for (i = 0; i < n; ++i) {
    if (js[i] < 0 || js[i] >= a->R || kvhs[i] < 0 || kvhs[i] >= a->hkv) return 1;
    if (js[i] < jmin) jmin = js[i];
  }
  if (n == 0) return 0;
  lse_rows = (double*)malloc(sizeof(double) * (size_t)a->R * a->hq);
  d_rows = (double*)malloc(sizeof(double) * (size_t)a->R * a->hq);
  if (!lse_rows || !d_rows) {
    free(lse_rows);
    free(d_rows);
    return 2;
  }
  err = row_stats(a, d_o, do_dtype, jmin, lse_rows, d_rows);
  if (!err) {
#pragma omp parallel
    {
      row_scratch s;
      int ok = scratch_alloc(a, &s) == 0;
      double* dod = (double*)malloc(sizeof(double) * a->d);
      int r;
      if (!ok || !dod) {
        ok = 0;
#pragma omp atomic write
        err = 2;
      }
#pragma omp for schedule(dynamic, 1)
      for (r = 0; r < n; ++r)
        if (ok)
          dkdv_key(a, &s, d_o, do_dtype, lse_rows, d_rows, js[r], kvhs[r],
                   dk + (int64_t)r * a->d, dv + (int64_t)r * a->d, dod);
      free(dod);
      scratch_free(&s);
    }
  }
  free(lse_rows);
  free(d_rows);
  return err;
}

int lso_attn_bwd(const lso_attn* a, const void* d_o, int32_t do_dtype, double* dq, double* dk,
                 double* dv) {
  int err = attn_check(a);
  int64_t rows = (int64_t)a->R * a->hq, keys = (int64_t)a->R * a->hkv;
  double *lse_rows, *d_rows;
  if (err) return err;
  if (a->R == 0) return 0;
  lse_rows = (double*)malloc(sizeof(double) * rows);
  d_rows = (double*)malloc(sizeof(double) * rows);
  if (!lse_rows || !d_rows) {
    free(lse_rows);
    free(d_rows);
    return 2;
  }
  err = row_stats(a, d_o, do_dtype, 0, lse_rows, d_rows);
  if (!err) {
#pragma omp parallel
    {
      row_scratch s;
      int ok = scratch_alloc(a, &s) == 0;
      double* dod = (double*)malloc(sizeof(double) * a->d);
      int64_t r;
      if (!ok || !dod) {
        ok = 0;
#pragma omp atomic write
        err = 2;
      }
#pragma omp for schedule(dynamic, 1)
      for (r = 0; r < rows; ++r) {
        if (!ok) continue;
        load_vec(dod, d_o, r * a->d, a->d, do_dtype);
        dq_row(a, &s, dod, d_rows[r], lse_rows[r], (int)(r / a->hq), (int)(r % a->hq),
               dq + r * a->d);
      }
#pragma omp for schedule(dynamic, 1)
      for (r = 0; r < keys; ++r)
        if (ok)
          dkdv_key(a, &s, d_o, do_dtype, lse_rows, d_rows, (int)(r / a->hkv),
                   (int)(r % a->hkv), dk + r * a->d, dv + r * a->d, dod);
      free(dod);
      scratch_free(&s);
    }
  }
  free(lse_rows);
  free(d_rows);
  return err;
}

/* ---------------------------------------------------------------- GRPO */

/* log sum_v exp(z_v) of one row, max-subtracted. */
static double row_lse(const void* logits, int dtype, int64_t row, int V) {
  double m = -INFINITY, s = 0.0;
  int v;
  for (v = 0; v < V; ++v) {
    double z = load_one(logits, row * V + v, dtype);
    if (z > m) m = z;
  }
  for (v = 0; v < V; ++v) s += exp(load_one(logits, row * V + v, dtype) - m);
  return m + log(s);
}

/* The clipped surrogate of the digest's Method section,
 *   L = -(1/G) sum_i (1/R_i) sum_t min(rho_{i,t} A_i, clip(rho_{i,t}, 1-eps, 1+eps) A_i),
 * with rho = exp(logp - logp_old), logp the log-softmax of the logits at the target
 * token, and group-relative advantages A_i = (r_i - mean r) / (std r + adv_eps)
 * (mean and std over the G members of the group, std with std_ddof). */
int lso_grpo(const void* logits, int32_t dtype, int64_t T, int32_t V,
             const int32_t* targets, const double* logp_old, const double* rewards,
             const int32_t* resp_lens, int32_t G, int32_t member_begin, int32_t member_end,
             double eps, double adv_eps, int32_t std_ddof,
             double* loss, double* adv, double* lse, double* logp, double* ratio,
             double* coef, int32_t* zeroed) {
  double mean = 0.0, var = 0.0, sd, total = 0.0;
  double* A;
  double* term;
  int64_t* member_of;
  int64_t t, covered = 0;
  int i, err = 0;
  if (G <= 0 || V <= 0 || T < 0 || member_begin < 0 || member_end > G ||
      member_begin > member_end || std_ddof < 0 || G - std_ddof <= 0 || !loss)
    return 1;
  for (i = member_begin; i < member_end; ++i) {
    if (resp_lens[i] < 0) return 1;
    covered += resp_lens[i];
  }
  if (covered != T) return 1;
  for (t = 0; t < T; ++t)
    if (targets[t] < 0 || targets[t] >= V) return 1;

  A = (double*)malloc(sizeof(double) * G);
  term = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
  member_of = (int64_t*)malloc(sizeof(int64_t) * (T > 0 ? T : 1));
  if (!A || !term || !member_of) {
    free(A);
    free(term);
    free(member_of);
    return 2;
  }
  /* Mean and spread are taken about the first reward (r_i - r_0 is exact for rewards
   * that are fp32 values), which is the same mean mathematically but leaves no rounding
   * residue when every reward is equal: then every deviation is exactly 0 and so is
   * every advantage, instead of ~1e-16 / 1e-6. */
  for (i = 0; i < G; ++i) mean += rewards[i] - rewards[0];
  mean /= G;
  for (i = 0; i < G; ++i) {
    double dev = (rewards[i] - rewards[0]) - mean;
    var += dev * dev;
  }
  var /= (double)(G - std_ddof);
  sd = sqrt(var);
  for (i = 0; i < G; ++i) A[i] = ((rewards[i] - rewards[0]) - mean) / (sd + adv_eps);
  if (adv)
    for (i = 0; i < G; ++i) adv[i] = A[i];

  t = 0;
  for (i = member_begin; i < member_end; ++i) {
    int64_t k;
    for (k = 0; k < resp_lens[i]; ++k) member_of[t++] = i;
  }

#pragma omp parallel for schedule(dynamic, 16)
  for (t = 0; t < T; ++t) {
    int mi = (int)member_of[t];
    double Ai = A[mi];
    double l = row_lse(logits, dtype, t, V);
    double lp = load_one(logits, t * V + targets[t], dtype) - l;
    double rho = exp(lp - logp_old[t]);
    double clipped = rho < 1.0 - eps ? 1.0 - eps : (rho > 1.0 + eps ? 1.0 + eps : rho);
    double unclipped_obj = rho * Ai, clipped_obj = clipped * Ai;
    /* min(.,.) picks the unclipped branch on ties: its gradient then flows. */
    int active = unclipped_obj <= clipped_obj;
    double c = active ? -(Ai * rho) / ((double)G * (double)resp_lens[mi]) : 0.0;
    term[t] = active ? unclipped_obj : clipped_obj;
    if (lse) lse[t] = l;
    if (logp) logp[t] = lp;
    if (ratio) ratio[t] = rho;
    if (coef) coef[t] = c;
    if (zeroed) zeroed[t] = (!active && Ai != 0.0) ? 1 : 0;
  }

  /* Fixed-order reduction: per member, then over members. */
  t = 0;
  for (i = member_begin; i < member_end; ++i) {
    double s = 0.0;
    int64_t k;
    for (k = 0; k < resp_lens[i]; ++k) s += term[t++];
    if (resp_lens[i] > 0) total += s / (double)resp_lens[i];
  }
  *loss = -total / (double)G;
  free(A);
  free(term);
  free(member_of);
  return err;
}

/* d(loss)/d(z_v) of one token: the surrogate depends on the logits only through
 * logp = z_y - lse, and d(logp)/d(z_v) = 1[v == y] - softmax_v. */
int lso_grpo_dlogits_row(const void* logits_row, int32_t dtype, int32_t V, int32_t target,
                         double lse, double coef, double* out) {
  int v;
  if (V <= 0 || target < 0 || target >= V) return 1;
  for (v = 0; v < V; ++v) {
    double p = exp(load_one(logits_row, v, dtype) - lse);
    out[v] = coef * ((v == target ? 1.0 : 0.0) - p);
  }
  return 0;
}

/* Pre-step scoring of GRPO (no gradient): per token the log-probability of the target,
 * logp_t = z_{t,y_t} - logsumexp_v z_{t,v}, and, when reference log-probabilities are
 * given, the per-token KL estimate of the policy from the reference
 *   kl_t = exp(ref_t - logp_t) - (ref_t - logp_t) - 1
 * (non-negative, zero exactly when ref_t = logp_t).  ref_logp and kl may be NULL. */
int lso_grpo_logp(const void* logits, int32_t dtype, int64_t T, int32_t V,
                  const int32_t* targets, const double* ref_logp, double* lse, double* logp,
                  double* kl) {
  int64_t t;
  if (T < 0 || V <= 0 || (kl && !ref_logp)) return 1;
  for (t = 0; t < T; ++t)
    if (targets[t] < 0 || targets[t] >= V) return 1;
#pragma omp parallel for schedule(dynamic, 4)
  for (t = 0; t < T; ++t) {
    const double l = row_lse(logits, dtype, t, V);
    const double lp = load_one(logits, t * V + targets[t], dtype) - l;
    if (lse) lse[t] = l;
    logp[t] = lp;
    if (kl) {
      const double d = ref_logp[t] - lp;
      kl[t] = exp(d) - d - 1.0;
    }
  }
  return 0;
}
