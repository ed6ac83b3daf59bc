/*
 * longstraw_oracle.h -- plain fp64 CPU reference for the response-replay hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This header and longstraw_oracle.c are used by the
 * tests, by the smoke check and by the benchmark's CPU-baseline leg. The product
 * library (response_replay_gb300, include/longstraw.h) never includes, links or
 * calls anything here, and nothing here includes the product's headers.
 *
 * What is computed (citations are to the LongStraw pages: the paper digest, page
 * "LongStraw: Long-Context RL Beyond 2M Tokens under a Fixed GPU Budget", and the
 * explainer "LongStraw: fitting million-token RL onto a fixed GPU budget"):
 *
 *   capture   -- the prompt is evaluated once without autograd and its K/V are kept
 *                as resident pages (digest, Method step 1; explainer, "The move:
 *                change the graph boundary").  The oracle is the literal scatter loop.
 *   replay    -- one response branch attends exactly to the captured prompt pages
 *                and causally to itself (digest, Method step 3; explainer, "Serial
 *                replay makes G a schedule"); prompt-side partial softmax statistics
 *                are composed by log-sum-exp into the exact global output (explainer,
 *                "Two incompatible architectures", Qwen bullet; digest, Qwen
 *                implementation).
 *   backward  -- only the conditional response gradient: the prompt state is
 *                stopgrad, so no gradient reaches prompt keys or values (digest,
 *                Method, last paragraph; explainer, Figure 2 caption).
 *   GRPO      -- token-level clipped surrogate with group-relative advantages and the
 *                1/G * 1/R_i normalisation (digest, Method, the L_policy equation).
 *
 * Every floating-point input is widened exactly to double; all arithmetic is fp64.
 * Element types of input arrays: LSO_BF16 (uint16 bit patterns), LSO_F32, LSO_F64.
 *
 * Return codes: 0 ok, 1 invalid argument (sizes, a page id outside the pool, a page
 * index beyond the table), 2 out of memory.
 *
 * Pins (each function is checked against something other than itself; the pages print
 * no numeric values for this path, so none comes from them):
 *   lso_capture_kv          byte-exact scatter, untouched sentinel pages, gather back =
 *                           input, out-of-table positions rejected
 *   lso_attn_fwd            brute-force monolithic softmax on tiny inputs for every split
 *                           count; q = 0 closed form (mean of visible V, lse =
 *                           log(P + t + 1)); P = 0 equals a library causal attention;
 *                           R = 1 equals single-query decode; one page with the identity
 *                           table equals shuffled pages; a hand-worked fixture
 *   lso_attn_fwd_rows       equals lso_attn_fwd on the sampled rows
 *   lso_attn_bwd            central finite differences of <dO, O>; P = 0 equals a library
 *                           autograd of causal attention
 *   lso_attn_bwd_dq_rows,
 *   lso_attn_bwd_dkdv_keys  equal lso_attn_bwd on the sampled rows / keys
 *   lso_grpo                a hand-worked fixture; equal rewards give exactly zero; ratio
 *                           one gives the closed-form loss and coefficients; the clip
 *                           on the favourable side zeroes the gradient; constant logits
 *                           give lse = log V + c; the unclipped limit equals a library
 *                           log-softmax; per-member calls add up to the whole range
 *   lso_grpo_dlogits_row    central finite differences of the loss
 *   lso_grpo_logp           a library log-softmax and the closed-form lse; the KL
 *                           estimate's closed cases
 *   lso_mla_fwd             brute-force softmax over the gathered rows on tiny inputs;
 *                           q = 0 closed form (mean of the visible latents, lse =
 *                           log(P + t + 1)); equals lso_attn_fwd with one KV head, K the
 *                           whole row and V the row with its rotary part zeroed; one page
 *                           with the identity table equals shuffled pages
 *   lso_mla_fwd_rows        equals lso_mla_fwd on the sampled rows
 *   lso_mla_bwd             central finite differences of <dO, O> through lso_mla_fwd
 *                           (steps exact in bf16); one key: dq = 0 and d lat = [dO ; 0]
 *                           summed over the heads; equals lso_attn_bwd with one KV head
 *                           (dq = dQ, d lat = dK + dV)
 *   lso_mla_bwd_dq_rows,
 *   lso_mla_bwd_dlat_keys   equal lso_mla_bwd on the sampled rows / keys
 */
#ifndef LONGSTRAW_ORACLE_H
#define LONGSTRAW_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { LSO_BF16 = 0, LSO_F32 = 1, LSO_F64 = 2 };

/* Paged prompt cache plus one response branch, as the oracle reads them.
 * k_pool / v_pool: [num_pages][hkv][page_size][d], element type pool_dtype.
 * page_table: [num_logical_pages] logical page -> physical page.
 * P: valid prompt tokens (<= num_logical_pages * page_size).
 * q: [R][hq][d]; k_resp, v_resp: [R][hkv][d]; element type in_dtype.
 * Query head h reads key/value head h / (hq / hkv).
 * num_splits: the prompt is cut into this many contiguous ranges of whole logical
 * pages, ceil(pages / num_splits) pages each, whose partial results are merged by
 * log-sum-exp; the response keys form one more partial. */
typedef struct {
  const void* k_pool;
  const void* v_pool;
  int32_t pool_dtype;
  int32_t page_size;
  const int32_t* page_table;
  int64_t num_pages;
  int64_t num_logical_pages;
  int64_t P;
  int32_t hkv;
  int32_t d;
  const void* q;
  const void* k_resp;
  const void* v_resp;
  int32_t in_dtype;
  int32_t R;
  int32_t hq;
  int32_t num_splits;
  double scale;
} lso_attn;

/* Literal scatter: pool[pt[p / ps]][h][p % ps][:] = src[p - start][h][:] for K and V,
 * p in [start, start + n).  Pools and sources are bf16 bit patterns. */
int lso_capture_kv(uint16_t* k_pool, uint16_t* v_pool, const int32_t* page_table,
                   int64_t num_pages, int64_t num_logical_pages, int32_t page_size,
                   int32_t hkv, int32_t d, const uint16_t* k, const uint16_t* v,
                   int64_t start_pos, int64_t n);

/* Forward for every (t, h): o [R][hq][d], lse [R][hq] (natural log). */
int lso_attn_fwd(const lso_attn* a, double* o, double* lse);

/* Forward for the listed (t, h) rows only: o [n][d], lse [n]. */
int lso_attn_fwd_rows(const lso_attn* a, int32_t n, const int32_t* ts, const int32_t* hs,
                      double* o, double* lse);

/* Backward for the whole branch.  d_o: [R][hq][d] (element type do_dtype).
 * dq [R][hq][d]; dk, dv [R][hkv][d] for the response keys only. */
int lso_attn_bwd(const lso_attn* a, const void* d_o, int32_t do_dtype,
                 double* dq, double* dk, double* dv);

/* dQ for the listed (t, h) rows: dq [n][d]. */
int lso_attn_bwd_dq_rows(const lso_attn* a, const void* d_o, int32_t do_dtype, int32_t n,
                         const int32_t* ts, const int32_t* hs, double* dq);

/* dK, dV of the listed response keys (j, kv head): dk, dv [n][d]. */
int lso_attn_bwd_dkdv_keys(const lso_attn* a, const void* d_o, int32_t do_dtype, int32_t n,
                           const int32_t* js, const int32_t* kvhs, double* dk, double* dv);

/* GRPO surrogate over the tokens of members [member_begin, member_end) laid out
 * member-major in logits [T][V] (element type dtype).  rewards and resp_lens hold all
 * G members.  Outputs (any may be NULL except loss):
 *   loss   -- -(1/G) sum_i (1/R_i) sum_t min(rho A_i, clip(rho, 1-eps, 1+eps) A_i)
 *             over the members in range;
 *   adv    [G]  A_i = (r_i - mean r) / (std_ddof-std r + adv_eps);
 *   lse, logp, ratio, coef [T]; coef is dL/d(logp_t) = -(A_i rho_t)/(G R_i) when the
 *             unclipped branch is the active minimum (ties count as active), else 0;
 *   zeroed [T]  1 where the clip zeroes the token's gradient (A != 0, coef == 0). */
int lso_grpo(const void* logits, int32_t dtype, int64_t T, int32_t V,
             const int32_t* targets, const double* logp_old, const double* rewards,
             const int32_t* resp_lens, int32_t G, int32_t member_begin, int32_t member_end,
             double eps, double adv_eps, int32_t std_ddof,
             double* loss, double* adv, double* lse, double* logp, double* ratio,
             double* coef, int32_t* zeroed);

/* One row of dL/dlogits: out[v] = coef * (1[v == target] - exp(z_v - lse)). */
int lso_grpo_dlogits_row(const void* logits_row, int32_t dtype, int32_t V, int32_t target,
                         double lse, double coef, double* out);

/* Pre-step scoring (no gradient): lse_t, logp_t = z_{t,y_t} - lse_t and, given
 * ref_logp, kl_t = exp(ref_t - logp_t) - (ref_t - logp_t) - 1.  lse, ref_logp and kl
 * may be NULL (kl requires ref_logp). */
int lso_grpo_logp(const void* logits, int32_t dtype, int64_t T, int32_t V,
                  const int32_t* targets, const double* ref_logp, double* lse, double* logp,
                  double* kl);

/* Gated-DeltaNet replay from a captured state (gdn_oracle.c): per head h,
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t (scale q_t),
 * S_0 = state0[h] (dv x dk, row-major).  q, k: [R][H][dk], v: [R][H][dv] (in_dtype);
 * g, beta: [R][H] fp64. */
typedef struct {
  const double* state0;  /* [H][dv][dk] */
  const void* q;
  const void* k;
  const void* v;
  int32_t in_dtype;
  const double* g;
  const double* beta;
  int32_t R;
  int32_t H;
  int32_t dk;
  int32_t dv;
  double scale;
} lso_gdn;

/* o [R][H][dv] (may be NULL), state_out [H][dv][dk] (may be NULL): the state after
 * the last token. */
int lso_gdn_fwd(const lso_gdn* a, double* o, double* state_out);

/* Gradients of <dO, o> (d_o [R][H][dv], element type do_dtype): dq, dk [R][H][dk], dv
 * [R][H][dv], dg, dbeta [R][H]; dstate0 [H][dv][dk] is the gradient that would reach
 * the captured state (the replay treats the state as stopgrad).  Any output may be
 * NULL. */
int lso_gdn_bwd(const lso_gdn* a, const void* d_o, int32_t do_dtype, double* dq, double* dk,
                double* dv, double* dg, double* dbeta, double* dstate0);

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int lso_num_threads(void);

/* Latent (MLA-style) pages plus one response branch (mla_oracle.c).
 * lat_pool: bf16 [num_pages][page_size][d_c + d_r], each row a position's latent c
 * (d_c values) then its rotary key (d_r values); page_table [num_logical_pages];
 * P valid prompt positions; q: bf16 [R][H][d_c + d_r] absorbed queries; lat_resp:
 * bf16 [R][d_c + d_r] the response's own rows.  All heads share every row. */
typedef struct {
  const uint16_t* lat_pool;
  int32_t page_size;
  const int32_t* page_table;
  int64_t num_pages;
  int64_t num_logical_pages;
  int64_t P;
  const uint16_t* q;
  const uint16_t* lat_resp;
  int32_t R;
  int32_t H;
  int32_t d_c;
  int32_t d_r;
  double scale;
} lso_mla;

/* o [R][H][d_c] = softmax over keys (P prompt rows, response rows j <= t) of
 * scale <q, row> applied to the rows' first d_c values; lse [R][H] (natural log). */
int lso_mla_fwd(const lso_mla* a, double* o, double* lse);

/* The same for the listed (t, h) rows only: o [n][d_c], lse [n]. */
int lso_mla_fwd_rows(const lso_mla* a, int32_t n, const int32_t* ts, const int32_t* hs,
                     double* o, double* lse);

/* Backward with the prompt rows stopgrad; d_o: bf16 [R][H][d_c].  dq [R][H][d_c + d_r];
 * dlat [R][d_c + d_r], the gradient of the response's own rows. */
int lso_mla_bwd(const lso_mla* a, const uint16_t* d_o, double* dq, double* dlat);

/* dq of the listed (t, h) rows only: dq [n][d_c + d_r]. */
int lso_mla_bwd_dq_rows(const lso_mla* a, const uint16_t* d_o, int32_t n, const int32_t* ts,
                        const int32_t* hs, double* dq);

/* d lat of the listed response rows only: dlat [n][d_c + d_r]. */
int lso_mla_bwd_dlat_keys(const lso_mla* a, const uint16_t* d_o, int32_t n, const int32_t* js,
                          double* dlat);

#ifdef __cplusplus
}
#endif
#endif
