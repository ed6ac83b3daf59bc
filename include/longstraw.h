/*
 * longstraw.h -- C ABI of the GB300 response-replay hot path.
 *
 * LongStraw trains GRPO at million-token contexts by evaluating the shared prompt once
 * without autograd, keeping only the state later tokens need (for full attention: K/V
 * pages), and replaying one response branch at a time under autograd (LongStraw paper
 * digest, "TL;DR" and "Method" steps 1-4; explainer "LongStraw: fitting million-token
 * RL onto a fixed GPU budget", "The move: change the graph boundary" and "Serial replay
 * makes G a schedule").  This library is that replay for one full-attention layer plus
 * the GRPO loss, on one GPU:
 *
 *   ls_capture_kv          write the prompt's K/V into pages behind a page table
 *   ls_replay_attn_fwd     exact attention of one response branch over the captured
 *                          pages plus causal self-attention, split-KV partials merged
 *                          by log-sum-exp
 *   ls_replay_attn_bwd     dQ through prompt and response keys; dK/dV for the
 *                          response's own keys only (the prompt state is stopgrad)
 *   ls_grpo_loss_fwd_bwd   token-level clipped surrogate with group-relative
 *                          advantages and its logits gradient
 *   ls_mla_replay_fwd      the forward over latent (MLA-style) pages, which may be
 *                          held in host memory
 *   ls_mla_replay_bwd      its backward: dq, and the gradient of the response's own
 *                          latent rows (the prompt rows are stopgrad)
 *
 * Conventions shared by every call
 *   - Memory: every pointer argument is DEVICE memory on the current CUDA device unless
 *     stated otherwise, allocated and owned by the caller.  The library allocates no
 *     device memory; temporary space is the caller's `workspace` (size from the
 *     matching *_workspace query, which depends on the current device's SM count).
 *   - Streams: work is enqueued on `stream` (NULL = legacy default stream) and the
 *     calls return without synchronising, except ls_last_device_error.
 *   - Layouts: dense row-major, innermost dimension last, no padding.  bf16 is the
 *     upper half of an IEEE-754 binary32 (1 sign, 8 exponent, 7 fraction bits);
 *     fp32 is binary32.
 *   - Alignment: every device pointer must be 16-byte aligned, except the per-token
 *     arrays of the loss and scoring calls (targets, logp_old, ref_logp, logp_out,
 *     lse_out, kl_out), which need 4 bytes, so that a member's slice of a token-major
 *     buffer can be passed whatever its token offset.
 *   - Errors: arguments are checked on the host first; on failure the call returns
 *     LS_ERR_INVALID_ARG / LS_ERR_UNSUPPORTED / LS_ERR_WORKSPACE and launches
 *     nothing.  A failed launch returns LS_ERR_CUDA.  Conditions only the device can
 *     see (a page id outside the pool, response lengths that do not add up, a
 *     pipeline wait that exceeded its time limit) never trap: the kernel skips the
 *     offending access, records a code in a per-device error word and carries on;
 *     ls_last_device_error() reports and clears it.
 *   - Determinism: no floating-point atomics; the same inputs and launch
 *     configuration give bit-identical outputs.
 *   - Device reset: the library looks up the device addresses of its own device
 *     variables (the error word, the no-alloc scratch) once per device and keeps them
 *     for the life of the process.  cudaDeviceReset() unloads the library's device
 *     image, so these addresses go stale: do not call the library on a device after
 *     resetting it in the same process.
 */
#ifndef LONGSTRAW_H
#define LONGSTRAW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* ls_stream_t;

typedef enum {
  LS_OK = 0,
  LS_ERR_INVALID_ARG = 1,   /* a size, pointer, alignment or dtype is not accepted   */
  LS_ERR_UNSUPPORTED = 2,   /* valid in principle, not built (e.g. head_dim != 128)  */
  LS_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than the query says          */
  LS_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                      */
  LS_ERR_TIMEOUT = 5,       /* a device pipeline wait hit its time limit              */
  LS_ERR_DEVICE_CHECK = 6   /* a device-side argument check failed (bad page id ...)  */
} ls_status;

typedef enum { LS_BF16 = 0, LS_FP32 = 1 } ls_dtype;

/* The captured prompt state of one attention layer: K and V pages plus the page table
 * (the digest's "CP-sharded KV pages" of the Qwen implementation, held whole on one
 * GPU).  Caller-owned; read-only after capture.
 *   k_pool, v_pool  bf16 [num_pages][num_kv_heads][page_size][head_dim]
 *   page_table      int32 [num_logical_pages]: logical page -> physical page in
 *                   [0, num_pages).  Logical page p holds prompt positions
 *                   [p * page_size, (p + 1) * page_size).
 *   num_tokens      P, the valid prompt positions; P <= num_logical_pages * page_size.
 *                   Positions >= P on the last page are never read by attention.
 * Supported: head_dim == 128; page_size a power of two in [16, 4096]; num_pages *
 * num_kv_heads * page_size < 2^31.
 * The pools may live in host memory that the GPU reads directly (pinned, mapped
 * allocations; on a Grace-Blackwell node the Grace memory behind NVLink-C2C): the
 * capture writes and every replay reads them there, with no staging copy.  This is the
 * GB300 counterpart of holding the prompt's pages in CPU memory (explainer, "Two
 * incompatible architectures", GLM bullet).  page_table stays in GPU memory. */
typedef struct {
  void* k_pool;
  void* v_pool;
  const int32_t* page_table;
  int32_t num_pages;
  int32_t num_logical_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int64_t num_tokens;
} ls_kv_cache;

/* ---------------------------------------------------------------- capture
 * Prompt capture keeps the prompt's K/V as resident pages (digest, Method step 1;
 * explainer, "The move: change the graph boundary").  Copies positions
 * [start_pos, start_pos + n) of the prompt:
 *   k_pool[pt[p / ps]][h][p % ps][:] = k[p - start_pos][h][:]   (same for v)
 * k, v: bf16 [n][num_kv_heads][head_dim].  Bit copy.  Can be called in chunks.  A page
 * id outside [0, num_pages) skips that position and sets LS_ERR_DEVICE_CHECK.
 * start_pos + n must not exceed num_logical_pages * page_size. */
ls_status ls_capture_kv(const ls_kv_cache* cache, const void* k, const void* v,
                        int64_t start_pos, int64_t n, ls_stream_t stream);

/* ---------------------------------------------------------------- replay forward
 * Exact attention of one response branch (explainer, "Serial replay makes G a
 * schedule"; digest, Method step 3) over the captured prompt and causally over its own
 * keys; the prompt's split-KV partials are composed by log-sum-exp into the exact
 * output, which the pages do across eight GPUs (explainer, "Two incompatible
 * architectures", Qwen bullet) and this call does on one:
 *   s_{t,j} = softmax_scale * <q_{t,h}, k_{j,h/g}>,  j over all P prompt positions and
 *             response positions j <= t (g = Hq / num_kv_heads)
 *   lse_{t,h} = log sum_j exp(s_{t,j})           (natural log)
 *   o_{t,h}   = sum_j exp(s_{t,j} - lse_{t,h}) v_j
 * q: bf16 [R][Hq][128]; k_resp, v_resp: bf16 [R][num_kv_heads][128] (the response's
 * own keys/values); o: bf16 [R][Hq][128] (round-to-nearest-even); lse: fp32 [R][Hq].
 * num_splits (>= 1) cuts the prompt into that many contiguous ranges of 128-token
 * tiles; the result does not depend on it beyond rounding.  Hq % num_kv_heads == 0.
 * softmax_scale must be finite and > 0 (typically 1/sqrt(128)).
 * R == 0 is a no-op.  P == 0 is plain causal attention of the response. */
ls_status ls_replay_attn_fwd_workspace(const ls_kv_cache* cache, int R, int Hq,
                                       int num_splits, size_t* bytes);
ls_status ls_replay_attn_fwd(const ls_kv_cache* cache, const void* q, const void* k_resp,
                             const void* v_resp, int R, int Hq, float softmax_scale,
                             int num_splits, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, ls_stream_t stream);

/* ls_replay_attn_fwd_members: the same forward for `members` responses of equal length
 * R over the same captured prompt, in one launch.  Pre-step scoring runs every member
 * of a group forward-only before the step (explainer, "Serial replay makes G a
 * schedule": the response branches share the read-only prompt state); batching them
 * lets the members' rows that share a KV head walk each prompt K/V tile together, so
 * the prompt streams from HBM about once for all of them instead of once per member.
 * Member m's rows see the whole prompt and member m's own response keys (j <= t)
 * only; its result equals ls_replay_attn_fwd on member m's slices (up to rounding).
 * q: bf16 [members][R][Hq][128]; k_resp, v_resp: bf16 [members][R][num_kv_heads][128];
 * o: bf16 [members][R][Hq][128]; lse: fp32 [members][R][Hq].  Short responses (the
 * grouped-query-packed regime) pack the members' tokens into shared 128-row tiles, so
 * one K/V tile serves members x g x R rows; there a member's rows also meet the other
 * members' response keys, masked to zero weight, so inputs must be finite (a non-finite
 * value times a zero weight is not zero; the one-response call has the same property
 * for the causally masked keys of its own response).  members >= 0 (0 or R == 0 is a
 * no-op); LS_ERR_UNSUPPORTED when members x R or the work-unit count exceeds 2^30.
 * Other arguments and errors as ls_replay_attn_fwd; ls_replay_attn_fwd is this call
 * with members = 1. */
ls_status ls_replay_attn_fwd_members_workspace(const ls_kv_cache* cache, int R, int members,
                                               int Hq, int num_splits, size_t* bytes);
ls_status ls_replay_attn_fwd_members(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                     const void* v_resp, int R, int members, int Hq,
                                     float softmax_scale, int num_splits, void* o, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     ls_stream_t stream);

/* ---------------------------------------------------------------- replay backward
 * Gradient of the replayed branch with the prompt state stopgrad: only
 * d(loss)/d(theta) at the captured state is formed and the path through the prompt
 * state is dropped (digest, Method, last paragraph; explainer, Figure 2 caption), so
 * prompt keys and values receive no gradient and only the response's own keys do
 * (explainer, "Two incompatible architectures": K/V gradient pages exist only where a
 * response backward touches them).  With P_{t,j} = exp(s_{t,j} - lse_t),
 * D_t = <dO_t, O_t>, dS_{t,j} = P_{t,j} (<dO_t, v_j> - D_t):
 *   dq_t   = softmax_scale * sum_j dS_{t,j} k_j          (prompt and response keys)
 *   dk_j   = softmax_scale * sum_{h in group, t >= j} dS_{t,j} q_t    (response j)
 *   dv_j   = sum_{h in group, t >= j} P_{t,j} dO_t                    (response j)
 * o, lse: the forward's outputs for the same inputs; d_o: bf16 [R][Hq][128].
 * dq: fp32 [R][Hq][128]; dk_resp, dv_resp: fp32 [R][num_kv_heads][128].
 * accumulate != 0 adds into dq/dk_resp/dv_resp instead of overwriting them (serial
 * replay accumulates gradients member by member: digest, Method step 3).
 * The environment variable LS_BWD_PAIR=1, read once per process, runs dQ on pairs of
 * SMs (cluster CTA pairs); the default one-CTA kernel measured faster on every shape
 * tried.  Both give the same results up to summation order; the workspace query and
 * the call must see the same setting. */
ls_status ls_replay_attn_bwd_workspace(const ls_kv_cache* cache, int R, int Hq,
                                       int num_splits, size_t* bytes);
ls_status ls_replay_attn_bwd(const ls_kv_cache* cache, const void* q, const void* k_resp,
                             const void* v_resp, const void* o, const float* lse,
                             const void* d_o, int R, int Hq, float softmax_scale,
                             int num_splits, int accumulate, float* dq, float* dk_resp,
                             float* dv_resp, void* workspace, size_t workspace_bytes,
                             ls_stream_t stream);

/* ---------------------------------------------------------------- ragged members
 * ls_replay_attn_fwd_ragged / ls_replay_attn_bwd_ragged: the replay of `members`
 * responses of different lengths lens[0 .. members) (a HOST array) over the same captured
 * prompt, in one forward and one backward launch.  The members' tokens lie back to back
 * (member m's token t is row off_m + t, off_m = lens[0] + ... + lens[m-1], T = the sum):
 *   q, o, d_o: bf16 [T][Hq][128]; k_resp, v_resp: bf16 [T][num_kv_heads][128];
 *   lse: fp32 [T][Hq]; dq: fp32 [T][Hq][128]; dk_resp, dv_resp: fp32 [T][num_kv_heads][128].
 * Each member sees the whole prompt and its own response keys j <= t only (a
 * block-diagonal causal mask over the concatenation), so member m's results equal the
 * one-response calls on its slices, up to rounding; the work of all members shares one
 * schedule over the GPU (the pages replay members one by one; on one GPU with room for
 * a whole group this fills the SMs better for short and mixed lengths).  As for the
 * batched forward, inputs must be finite: a member's rows meet other members' keys with
 * zero weight, and a non-finite value times zero is not zero.
 * 1 <= members <= 64, lens[m] >= 0 (empty members allowed); T <= 2^30, and for the
 * backward of more than one member T <= 131,072 (LS_ERR_UNSUPPORTED otherwise).  Other
 * arguments, workspace and errors as ls_replay_attn_fwd / ls_replay_attn_bwd, which are
 * these calls with one member. */
ls_status ls_replay_attn_fwd_ragged_workspace(const ls_kv_cache* cache, const int32_t* lens,
                                              int members, int Hq, int num_splits, size_t* bytes);
ls_status ls_replay_attn_fwd_ragged(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                    const void* v_resp, const int32_t* lens, int members, int Hq,
                                    float softmax_scale, int num_splits, void* o, float* lse,
                                    void* workspace, size_t workspace_bytes, ls_stream_t stream);
ls_status ls_replay_attn_bwd_ragged_workspace(const ls_kv_cache* cache, const int32_t* lens,
                                              int members, int Hq, int num_splits, size_t* bytes);
ls_status ls_replay_attn_bwd_ragged(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                    const void* v_resp, const void* o, const float* lse,
                                    const void* d_o, const int32_t* lens, int members, int Hq,
                                    float softmax_scale, int num_splits, int accumulate, float* dq,
                                    float* dk_resp, float* dv_resp, void* workspace,
                                    size_t workspace_bytes, ls_stream_t stream);

/* ---------------------------------------------------------------- GRPO loss
 * The clipped surrogate of the digest's Method section,
 *   L = -(1/G) sum_i (1/R_i) sum_t min(rho_{i,t} A_i, clip(rho_{i,t}, 1-eps, 1+eps) A_i),
 *   rho = exp(logp - logp_old),  logp = logits[target] - logsumexp(logits),
 *   A_i = (r_i - mean r) / (std r + adv_eps)   (group-relative; std with std_ddof;
 *                                             mean/std in fp64),
 * and its gradient dL/dlogits_v = c_t (1[v == target] - softmax_v), where
 * c_t = -A_i rho_t / (G R_i) when the unclipped term is the active minimum (ties
 * included) and 0 when the clip holds the term constant.
 * Serial replay calls this once per member (digest, Method step 3): logits hold the
 * tokens of members [member_begin, member_end) back to back (member-major), while
 * rewards and resp_lens describe all G members so every call sees the whole group.
 *   logits   [T][V] of type dtype; T = sum of resp_lens over the range (checked on the
 *            device: a mismatch sets LS_ERR_DEVICE_CHECK and writes nothing)
 *   targets  int32 [T] in [0, V);  logp_old fp32 [T]
 *   rewards  fp32 [G];  resp_lens int32 [G]
 *   loss     fp32 device scalar: this call's contribution (accumulate_loss != 0 adds
 *            it to the current value)
 *   dlogits  [T][V] of type dtype (may alias nothing else)
 *   logp_out fp32 [T] or NULL
 *   stats    fp32 [4] or NULL: {tokens whose gradient the clip zeroed, sum of rho,
 *            min rho, max rho} over this call's tokens
 * G - std_ddof must be >= 1; 0 <= member_begin <= member_end <= G; V <= 2^30. */
ls_status ls_grpo_workspace(int64_t T, int G, size_t* bytes);
ls_status ls_grpo_loss_fwd_bwd(const void* logits, ls_dtype dtype, int64_t T, int V,
                               const int32_t* targets, const float* logp_old,
                               const float* rewards, const int32_t* resp_lens, int G,
                               int member_begin, int member_end, float eps, float adv_eps,
                               int std_ddof, int accumulate_loss, float* loss, void* dlogits,
                               float* logp_out, float* stats, void* workspace,
                               size_t workspace_bytes, ls_stream_t stream);

/* ls_grpo_loss_fwd_bwd_noalloc: the same computation as ls_grpo_loss_fwd_bwd, for
 * callers that cannot provide or allocate device memory at the point of the call (for
 * example a training loop whose host framework plans all device memory up front and
 * forbids new allocations mid-step).  The paper has no counterpart: this is an
 * interface convenience of this library.  Instead of a caller workspace it uses one
 * fixed scratch array inside the library's device image (4.125 MiB per device, held
 * until process exit); it calls no allocator.  Limits: T <= 262,144 tokens and
 * G <= 1,024 members, otherwise LS_ERR_WORKSPACE is returned and nothing is launched.
 * The first call on a device looks up the array's device address (a runtime query,
 * no allocation); make that first call before any stream capture.  All calls share
 * the array: calls whose kernels could overlap on the GPU race, so order them (one
 * stream, or events).  Nothing in the array needs to start at zero.  Arguments and
 * outputs otherwise as ls_grpo_loss_fwd_bwd. */
ls_status ls_grpo_loss_fwd_bwd_noalloc(const void* logits, ls_dtype dtype, int64_t T, int V,
                                       const int32_t* targets, const float* logp_old,
                                       const float* rewards, const int32_t* resp_lens, int G,
                                       int member_begin, int member_end, float eps,
                                       float adv_eps, int std_ddof, int accumulate_loss,
                                       float* loss, void* dlogits, float* logp_out,
                                       float* stats, ls_stream_t stream);

/* ls_grpo_logp: pre-step scoring without a gradient (LongStraw explainer: the replay
 * is the gradient pass of one member; the log-probabilities a step needs before it,
 * logp_old and a reference policy's, come from forward-only passes like this one).
 *   logp_t = logits[t][targets[t]] - logsumexp_v logits[t][v]
 *   kl_t   = exp(d) - d - 1 with d = ref_logp[t] - logp_t  (when ref_logp is given):
 *            the per-token KL estimate of the policy from the reference, >= 0 and zero
 *            exactly where the two agree (the pages fix no KL form; their 2M-token runs
 *            used beta = 0).
 * logits: [T][V] dtype (bf16 or fp32), targets: int32 [T], ref_logp: fp32 [T] or NULL;
 * outputs fp32 [T]: logp_out (required), lse_out (natural-log logsumexp, optional),
 * kl_out (optional, requires ref_logp).  Each row is read once.  No workspace.
 * Errors: LS_ERR_INVALID_ARG for a bad dtype, T < 0, V <= 0, a missing or unaligned
 * required pointer, or kl_out without ref_logp; a target outside [0, V) records
 * LS_ERR_DEVICE_CHECK (see ls_last_device_error) and yields NaN for that token. */
ls_status ls_grpo_logp(const void* logits, ls_dtype dtype, int64_t T, int V,
                       const int32_t* targets, const float* ref_logp, float* logp_out,
                       float* lse_out, float* kl_out, ls_stream_t stream);

/* ---------------------------------------------------------------- Gated-DeltaNet replay
 * The hybrid model's Gated-DeltaNet layers keep only the compact recurrent state at the
 * end of the prompt, and each response is replayed from it with that state stopgrad
 * (digest, "Method" step 1 and "Qwen implementation"; explainer, "Two incompatible
 * architectures", Qwen bullet).  The pages give no equations for the layer; the
 * recurrence is the gated delta rule (Yang, Kautz & Hatamizadeh, "Gated Delta Networks:
 * Improving Mamba2 with Delta Rule", ICLR 2025), per head h and response token t:
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   S_0 = state0[h]
 *   o_t = S_t (scale q_t)
 * S is a 128 x 128 fp32 matrix (d_v x d_k, row-major).  Heads are independent; for
 * grouped key heads the caller passes each value head's q and k.
 *   state0     fp32 [H][128][128]: the captured state (read only)
 *   q, k, v    bf16 [R][H][128]; k is used as given (the layer normalises it)
 *   g, beta    fp32 [R][H]: log of the decay (g <= 0 in the layer) and the write strength
 *   o          bf16 [R][H][128]
 *   state_out  fp32 [H][128][128] or NULL: the state after the last token (running the
 *              prompt from a zero state with state_out set is the capture)
 * Work is done in 64-token chunks; the result does not depend on R's split into chunks
 * beyond rounding.  R == 0 copies state0 to state_out.  workspace: the *_workspace
 * query's bytes (about 0.33 MB (forward) / 0.6 MB (backward) per head and 64 tokens).
 * Errors as for the attention calls; LS_ERR_UNSUPPORTED when ceil(R / 64) * H > 65535. */
ls_status ls_gdn_replay_fwd_workspace(int R, int H, size_t* bytes);
ls_status ls_gdn_replay_fwd(const float* state0, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, int R, int H, float scale, void* o,
                            float* state_out, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream);

/* ls_gdn_replay_bwd: gradients of the replayed response with the captured state
 * stopgrad (the gradient that would reach state0 is dropped).  d_o: bf16 [R][H][128];
 * dq, dk, dv: fp32 [R][H][128]; dg, dbeta: fp32 [R][H]; accumulate != 0 adds into them.
 * The forward's chunk quantities are recomputed; inputs as for the forward. */
ls_status ls_gdn_replay_bwd_workspace(int R, int H, size_t* bytes);
ls_status ls_gdn_replay_bwd(const float* state0, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const void* d_o, int R, int H,
                            float scale, int accumulate, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream);

/* ---------------------------------------------------------------- latent (MLA) replay
 * The GLM path keeps its multi-head latent attention state as latent pages held in CPU
 * memory and replays each response over them (explainer, "Two incompatible
 * architectures, same transaction", GLM bullet).  The pages give no equations for the
 * layer; it is multi-head latent attention (DeepSeek-V2, 2024) with the key
 * up-projection absorbed into the query.  Every position j keeps one row shared by all
 * heads, its latent c_j (512 values) followed by its rotary key r_j (64 values); the
 * caller passes each head's absorbed query (576 values), and
 *   s_{t,h,j} = softmax_scale * <q_{t,h}, [c_j ; r_j]>,  j over all P prompt rows and
 *               the response rows j <= t
 *   lse_{t,h} = log sum_j exp(s_{t,h,j})        (natural log)
 *   o_{t,h}   = sum_j exp(s_{t,h,j} - lse_{t,h}) c_j   (512 values)
 * The value up-projection and the output projection are weights (the caller's).
 *
 * ls_latent_cache: the captured prompt rows of one latent-attention layer.
 *   pool        bf16 [num_pages][page_size][576]; may be pinned host memory that the
 *               GPU reads directly (on a Grace-Blackwell node, Grace memory behind
 *               NVLink-C2C): capture writes it there and the replay reads it there.
 *   page_table  int32 [num_logical_pages] in GPU memory: logical page -> physical page.
 *   num_tokens  P <= num_logical_pages * page_size.
 * Supported: page_size a power of two in [32, 4096]; num_pages * page_size < 2^31.
 *
 * ls_capture_latent: pool[pt[p / ps]][p % ps][:] = lat[p - start_pos][:] for p in
 * [start_pos, start_pos + n); lat bf16 [n][576].  Bit copy; a page id outside the pool
 * skips the row and sets LS_ERR_DEVICE_CHECK.
 *
 * ls_mla_replay_fwd: the forward of one response of R tokens with H heads.
 * q: bf16 [R][H][576]; lat_resp: bf16 [R][576] (the response's own rows); o: bf16
 * [R][H][512]; lse: fp32 [R][H].  num_splits (>= 1) cuts the prompt into that many
 * ranges of 64-row tiles, merged by log-sum-exp; the result does not depend on it
 * beyond rounding.  softmax_scale finite and > 0.  R == 0 is a no-op; P == 0 is causal
 * attention over the response rows.  Inputs must be finite (a row past a query's
 * causal bound has weight zero, and zero times a non-finite value is not zero).
 * LS_ERR_UNSUPPORTED when R x H >= 2^31.
 *
 * ls_mla_replay_bwd: the backward of ls_mla_replay_fwd with the prompt rows stopgrad
 * (LongStraw paper digest, Method, last paragraph: the captured state takes no
 * gradient).  With P = exp(s - lse), D_{t,h} = <dO_{t,h}, o_{t,h}>, dP_j = <dO, c_j> and
 * dS = P (dP - D):
 *   dq_{t,h} = softmax_scale sum_j dS_{t,h,j} [c_j ; r_j]     (all visible rows j)
 *   dlat_j   = sum_{t >= j} sum_h ( P_{t,h,j} [dO_{t,h} ; 0] + softmax_scale dS_{t,h,j} q_{t,h} )
 * for the response's own rows j (the latent is both key and value; its rotary part is a
 * key only).  q, lat_resp, R, H, softmax_scale and the cache as for the forward; o
 * (bf16 [R][H][512]) and lse (fp32 [R][H]) are the forward's outputs, d_o bf16
 * [R][H][512].  dq: fp32 [R][H][576]; dlat: fp32 [R][576]; both overwritten.
 * num_splits (>= 1) cuts the prompt into ranges of 32-row tiles whose partial dq are
 * added in a fixed order (the result does not depend on it beyond rounding; a given
 * split count gives the same bits every call).  Workspace from
 * ls_mla_replay_bwd_workspace (never zero for R > 0).  R == 0 is a no-op. */
typedef struct {
  void* pool;
  const int32_t* page_table;
  int32_t num_pages;
  int32_t num_logical_pages;
  int32_t page_size;
  int64_t num_tokens;
} ls_latent_cache;

ls_status ls_capture_latent(const ls_latent_cache* cache, const void* lat, int64_t start_pos,
                            int64_t n, ls_stream_t stream);
ls_status ls_mla_replay_fwd_workspace(const ls_latent_cache* cache, int R, int H, int num_splits,
                                      size_t* bytes);
ls_status ls_mla_replay_fwd(const ls_latent_cache* cache, const void* q, const void* lat_resp,
                            int R, int H, float softmax_scale, int num_splits, void* o,
                            float* lse, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream);
ls_status ls_mla_replay_bwd_workspace(const ls_latent_cache* cache, int R, int H, int num_splits,
                                      size_t* bytes);
ls_status ls_mla_replay_bwd(const ls_latent_cache* cache, const void* q, const void* lat_resp,
                            const void* o, const float* lse, const void* d_o, int R, int H,
                            float softmax_scale, int num_splits, float* dq, float* dlat,
                            void* workspace, size_t workspace_bytes, ls_stream_t stream);

/* ---------------------------------------------------------------- checks
 * ls_validate_page_table: enqueue a check that every entry of the page table covering
 * the cache's num_tokens lies in [0, num_pages) and that no physical page is used
 * twice; a failure sets LS_ERR_DEVICE_CHECK in the device error word.
 * ls_last_device_error: synchronise `stream`, return the first device-side error
 * recorded on the current device since the last call (LS_OK if none) and clear it. */
ls_status ls_validate_page_table(const ls_kv_cache* cache, void* workspace,
                                 size_t workspace_bytes, ls_stream_t stream);
ls_status ls_validate_page_table_workspace(const ls_kv_cache* cache, size_t* bytes);
ls_status ls_last_device_error(ls_stream_t stream);

const char* ls_status_string(ls_status status);

/* Diagnostic: number of kernel launches this library has issued in the process (all
 * devices), e.g. to count the launches of one step. */
uint64_t ls_kernel_launches(void);

/* Diagnostic (the pages have no counterpart): enqueue one block that waits, through the
 * pipelines' own bounded mbarrier wait, on a barrier nothing completes.  After the
 * wait's time limit (about 2 s of SM clock) the block records LS_ERR_TIMEOUT in the
 * device error word and exits, so a following ls_last_device_error() returns
 * LS_ERR_TIMEOUT and the context stays usable.  Returns LS_OK once enqueued,
 * LS_ERR_CUDA if the launch fails.  Used by the tests of the failure path. */
ls_status ls_selftest_wait_timeout(ls_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LONGSTRAW_H */
