/*
 * gdn_oracle.c -- plain fp64 CPU reference for Gated-DeltaNet replay from a captured
 * recurrent state.
 *
 * TEST INFRASTRUCTURE ONLY (see longstraw_oracle.c): used by the tests, the smoke check
 * and the benchmark's CPU-baseline leg; the product library never links or calls it.
 *
 * LongStraw keeps, for the hybrid model's Gated-DeltaNet layers, only the compact
 * recurrent state at the end of the prompt and replays each response from it with the
 * prompt state stopgrad (digest, "Method" step 1 and "Qwen implementation"; explainer,
 * "Two incompatible architectures", Qwen bullet).  The pages give no equations for the
 * layer; the recurrence is the gated delta rule of Yang, Kautz and Hatamizadeh, "Gated
 * Delta Networks: Improving Mamba2 with Delta Rule" (ICLR 2025), per head:
 *   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   alpha_t = exp(g_t)
 *   o_t = S_t (scale q_t)
 * with S_t a d_v x d_k matrix and S_0 the captured state.  Written as the literal
 * token-by-token loop: no chunking, no reordering.
 *
 * The backward is reverse-mode differentiation of that loop (the adjoint of each step in
 * reverse token order).  With X the gradient of the loss with respect to S_t (from o_t
 * and from S_{t+1}), S_prev = S_{t-1}, kv = S_prev k_t and Xk = X k_t:
 *   dq_t     = scale S_t^T dO_t
 *   dv_t     = beta_t Xk
 *   dbeta_t  = Xk . (v_t - alpha_t kv)
 *   dalpha_t = <X, S_prev> - beta_t (Xk . kv),          dg_t = alpha_t dalpha_t
 *   dk_t     = -alpha_t beta_t (S_prev^T Xk + X^T kv) + beta_t X^T v_t
 *   dS_{t-1} = alpha_t (X - beta_t Xk k_t^T)
 * The gradient that reaches S_0 is what the captured state would receive; the replay
 * drops it (stopgrad) and the oracle returns it only on request, for the pins.
 * The states S_{t-1} needed in reverse order are recomputed from the forward's
 * states stored every kCkpt tokens (the same operations in the same order, so the
 * recomputed states are the forward's, bit for bit).
 */
#include "longstraw_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { kCkpt = 64 };

static double gdn_bf16(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* element e of an array of type dtype (bf16 bits, fp32 or fp64) */
static double gdn_load(const void* base, int64_t e, int32_t dtype) {
  if (dtype == LSO_BF16) return gdn_bf16(((const uint16_t*)base)[e]);
  if (dtype == LSO_F32) return (double)((const float*)base)[e];
  return ((const double*)base)[e];
}

/* One step of the recurrence on S (dv x dk, row-major), in place. */
static void gdn_step(double* S, const double* k, const double* v, double alpha, double beta,
                     int dk, int dv, double* kv) {
  int i, j;
  for (i = 0; i < dv; ++i) {
    double s = 0.0;
    for (j = 0; j < dk; ++j) s += S[(int64_t)i * dk + j] * k[j];
    kv[i] = s;
  }
  for (i = 0; i < dv; ++i)
    for (j = 0; j < dk; ++j) {
      double* x = &S[(int64_t)i * dk + j];
      *x = alpha * (*x - beta * kv[i] * k[j]) + beta * v[i] * k[j];
    }
}

static void gdn_load_vec(double* dst, const void* src, int32_t dtype, int64_t off, int n) {
  int i;
  for (i = 0; i < n; ++i) dst[i] = gdn_load(src, off + i, dtype);
}

int lso_gdn_fwd(const lso_gdn* a, double* o, double* state_out) {
  int h;
  int err = 0;
  if (!a || a->R < 0 || a->H <= 0 || a->dk <= 0 || a->dv <= 0 || !a->state0) return 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (h = 0; h < a->H; ++h) {
    const int dk = a->dk, dv = a->dv, H = a->H;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* q = (double*)malloc(sizeof(double) * dk);
    double* k = (double*)malloc(sizeof(double) * dk);
    double* v = (double*)malloc(sizeof(double) * dv);
    double* kv = (double*)malloc(sizeof(double) * dv);
    int t, i, j;
    if (!S || !q || !k || !v || !kv) {
#pragma omp atomic write
      err = 2;
    } else {
      memcpy(S, a->state0 + (int64_t)h * dk * dv, sizeof(double) * (size_t)dk * dv);
      for (t = 0; t < a->R; ++t) {
        const int64_t r = (int64_t)t * H + h;
        gdn_load_vec(q, a->q, a->in_dtype, r * dk, dk);
        gdn_load_vec(k, a->k, a->in_dtype, r * dk, dk);
        gdn_load_vec(v, a->v, a->in_dtype, r * dv, dv);
        gdn_step(S, k, v, exp(a->g[r]), a->beta[r], dk, dv, kv);
        if (o)
          for (i = 0; i < dv; ++i) {
            double s = 0.0;
            for (j = 0; j < dk; ++j) s += S[(int64_t)i * dk + j] * (a->scale * q[j]);
            o[r * dv + i] = s;
          }
      }
      if (state_out) memcpy(state_out + (int64_t)h * dk * dv, S, sizeof(double) * (size_t)dk * dv);
    }
    free(S);
    free(q);
    free(k);
    free(v);
    free(kv);
  }
  return err;
}

int lso_gdn_bwd(const lso_gdn* a, const void* d_o, int32_t do_dtype, double* dq, double* dk_out,
                double* dv_out, double* dg, double* dbeta, double* dstate0) {
  int h;
  int err = 0;
  if (!a || a->R < 0 || a->H <= 0 || a->dk <= 0 || a->dv <= 0 || !a->state0 || !d_o) return 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (h = 0; h < a->H; ++h) {
    const int dk = a->dk, dv = a->dv, H = a->H, R = a->R;
    const int64_t ss = (int64_t)dk * dv;
    const int nck = R / kCkpt + 1;
    /* ck[c]: state before token c kCkpt; seg[s]: states before tokens of one segment */
    double* ck = (double*)malloc(sizeof(double) * ss * nck);
    double* seg = (double*)malloc(sizeof(double) * ss * (kCkpt + 1));
    double* X = (double*)malloc(sizeof(double) * ss);
    double *q = (double*)malloc(sizeof(double) * dk), *k = (double*)malloc(sizeof(double) * dk);
    double *v = (double*)malloc(sizeof(double) * dv), *kv = (double*)malloc(sizeof(double) * dv);
    double* xk = (double*)malloc(sizeof(double) * dv);
    double* dob = (double*)malloc(sizeof(double) * dv);
    int t, i, j, c;
    if (!ck || !seg || !X || !q || !k || !v || !kv || !xk || !dob) {
#pragma omp atomic write
      err = 2;
    } else {
      /* forward, keeping the state before every kCkpt-th token */
      memcpy(ck, a->state0 + (int64_t)h * ss, sizeof(double) * ss);
      memcpy(seg, ck, sizeof(double) * ss);
      for (t = 0; t < R; ++t) {
        const int64_t r = (int64_t)t * H + h;
        gdn_load_vec(k, a->k, a->in_dtype, r * dk, dk);
        gdn_load_vec(v, a->v, a->in_dtype, r * dv, dv);
        gdn_step(seg, k, v, exp(a->g[r]), a->beta[r], dk, dv, kv);
        if ((t + 1) % kCkpt == 0) memcpy(ck + (int64_t)((t + 1) / kCkpt) * ss, seg, sizeof(double) * ss);
      }
      memset(X, 0, sizeof(double) * ss); /* dL/dS_R: nothing follows the response */
      for (c = (R - 1) / kCkpt; c >= 0 && R > 0; --c) {
        const int t0 = c * kCkpt, t1 = t0 + kCkpt < R ? t0 + kCkpt : R;
        /* seg[s] = state before token t0 + s, s = 0 .. t1 - t0 */
        memcpy(seg, ck + (int64_t)c * ss, sizeof(double) * ss);
        for (t = t0; t < t1; ++t) {
          const int64_t r = (int64_t)t * H + h;
          memcpy(seg + (int64_t)(t - t0 + 1) * ss, seg + (int64_t)(t - t0) * ss, sizeof(double) * ss);
          gdn_load_vec(k, a->k, a->in_dtype, r * dk, dk);
          gdn_load_vec(v, a->v, a->in_dtype, r * dv, dv);
          gdn_step(seg + (int64_t)(t - t0 + 1) * ss, k, v, exp(a->g[r]), a->beta[r], dk, dv, kv);
        }
        for (t = t1 - 1; t >= t0; --t) {
          const int64_t r = (int64_t)t * H + h;
          const double* Sp = seg + (int64_t)(t - t0) * ss;     /* S_{t-1} */
          const double* St = seg + (int64_t)(t - t0 + 1) * ss; /* S_t */
          const double alpha = exp(a->g[r]), beta = a->beta[r];
          double dalpha = 0.0, db = 0.0, xkkv = 0.0;
          gdn_load_vec(q, a->q, a->in_dtype, r * dk, dk);
          gdn_load_vec(k, a->k, a->in_dtype, r * dk, dk);
          gdn_load_vec(v, a->v, a->in_dtype, r * dv, dv);
          gdn_load_vec(dob, d_o, do_dtype, r * dv, dv);
          /* X = dL/dS_t: the later steps' share (already in X) plus o_t's */
          for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j) X[(int64_t)i * dk + j] += dob[i] * (a->scale * q[j]);
          if (dq)
            for (j = 0; j < dk; ++j) {
              double s = 0.0;
              for (i = 0; i < dv; ++i) s += St[(int64_t)i * dk + j] * dob[i];
              dq[r * dk + j] = a->scale * s;
            }
          for (i = 0; i < dv; ++i) {
            double s1 = 0.0, s2 = 0.0;
            for (j = 0; j < dk; ++j) {
              s1 += Sp[(int64_t)i * dk + j] * k[j];
              s2 += X[(int64_t)i * dk + j] * k[j];
            }
            kv[i] = s1;
            xk[i] = s2;
          }
          for (i = 0; i < dv; ++i) {
            xkkv += xk[i] * kv[i];
            db += xk[i] * (v[i] - alpha * kv[i]);
            for (j = 0; j < dk; ++j) dalpha += X[(int64_t)i * dk + j] * Sp[(int64_t)i * dk + j];
          }
          dalpha -= beta * xkkv;
          if (dv_out)
            for (i = 0; i < dv; ++i) dv_out[r * dv + i] = beta * xk[i];
          if (dbeta) dbeta[r] = db;
          if (dg) dg[r] = alpha * dalpha;
          if (dk_out)
            for (j = 0; j < dk; ++j) {
              double a1 = 0.0, a2 = 0.0, a3 = 0.0;
              for (i = 0; i < dv; ++i) {
                a1 += Sp[(int64_t)i * dk + j] * xk[i];
                a2 += X[(int64_t)i * dk + j] * kv[i];
                a3 += X[(int64_t)i * dk + j] * v[i];
              }
              dk_out[r * dk + j] = -alpha * beta * (a1 + a2) + beta * a3;
            }
          /* dL/dS_{t-1} = alpha (X - beta Xk k^T) */
          for (i = 0; i < dv; ++i)
            for (j = 0; j < dk; ++j) {
              double* x = &X[(int64_t)i * dk + j];
              *x = alpha * (*x - beta * xk[i] * k[j]);
            }
        }
      }
      if (dstate0) memcpy(dstate0 + (int64_t)h * ss, X, sizeof(double) * ss);
    }
    free(ck);
    free(seg);
    free(X);
    free(q);
    free(k);
    free(v);
    free(kv);
    free(xk);
    free(dob);
  }
  return err;
}
