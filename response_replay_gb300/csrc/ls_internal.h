// ls_internal.h -- host-side interface between the C ABI (ls_api.cu) and the kernel
// translation units.  Not installed; the public interface is include/longstraw.h.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ls_sched.h"

// Bits of the per-device error word (see ls_last_device_error).
#define LS_DEVERR_CHECK 1u    // a device-side argument check failed
#define LS_DEVERR_TIMEOUT 2u  // a pipeline wait exceeded its time limit

// Counts every kernel launch the library makes (reported by ls_kernel_launches).
void ls_note_launch();

// Problem description shared by the replay-attention kernels (device pointers).
struct LsAttnArgs {
  const void* k_pool;        // bf16 [num_pages][hkv][ps][128]
  const void* v_pool;
  const int32_t* page_table; // [num_logical_pages]
  int32_t num_pages;
  int32_t ps_log2;           // page size = 1 << ps_log2
  int64_t P;                 // valid prompt tokens
  int32_t hkv, hq, g;        // g = hq / hkv
  int32_t pack;              // query rows per token in a tile: g (packed) or 1
  int32_t tiles;             // forward: query tiles per unit (2, or 1 when a packed unit's
                             // tokens all fit one tile)
  int32_t R;                 // response tokens (of each member)
  int32_t members;           // forward: responses of equal length R in one launch
  int32_t upm;               // units per member (INT32_MAX unless units are per member)
  int32_t rt;                // tokens the units cover: R, or members x R when the
                             // members' tokens are packed into shared tiles
  const void* q;             // bf16 [members][R][hq][128]
  const void* k_resp;        // bf16 [members][R][hkv][128]
  const void* v_resp;
  float scale_log2;          // softmax_scale * log2(e)
  float scale;               // softmax_scale
  uint32_t* err;             // device error word
};

struct LsFwdOut {
  void* o;                   // bf16 [members][R][hq][128]
  float* lse;                // [members][R][hq]
  float* part_o;             // workspace: [2*ctas][unit_rows][128]
  float* part_lse;           // workspace: [2*ctas][unit_rows]
};

struct LsBwdIn {
  const void* o;             // bf16 [R][hq][128]
  const float* lse;          // [R][hq]
  const void* d_o;           // bf16 [R][hq][128]
  float* delta;              // workspace [R][hq]: D = <dO, O>
  float* dt;                 // workspace [hq][rp]: D transposed, rp = R rounded up to 128
  float* lse2t;              // workspace [hq][rp]: lse log2(e) transposed
  float* dq;                 // [R][hq][128]
  float* dk;                 // [R][hkv][128]
  float* dv;
  float* part_dq;            // workspace: [pieces][unit_rows][128]
  float* part_dkdv;          // workspace: [2*ctas][2][128][128] (response-key kernel)
  int32_t accumulate;
  int32_t pair;              // dQ on CTA pairs (replay_bwd_dq_pair.cu) instead of one CTA
};

// Geometry of the replay kernels (fixed at build time).
int ls_fwd_unit_rows();
int ls_fwd_tile();
int ls_fwd_ctas_per_sm();
int ls_bwd_unit_rows();
int ls_bwd_tile();
int ls_bwd_ctas_per_sm();
int ls_num_units(int R, int hq, int hkv, int unit_rows);
// Forward: grouped-query packing factor (g for short responses, else 1) and units.
int ls_fwd_pack(int R, int hq, int hkv);
int ls_fwd_units(int R, int hq, int hkv);
int ls_fwd_tiles(int R, int hq, int hkv);
// Backward: the same packing for its one-tile units.
int ls_bwd_pack(int R, int hq, int hkv);
int ls_bwd_units(int R, int hq, int hkv);
// Backward dQ on CTA pairs: units of two tiles (one per CTA), their packing, and the
// number of pairs resident at once (the persistent grid).
int ls_bwd_pair_unit_rows();
int ls_bwd_pair_pack(int R, int hq, int hkv);
int ls_bwd_pair_units(int R, int hq, int hkv);
cudaError_t ls_bwd_pair_workers(int* pairs);

cudaError_t ls_launch_capture(const void* k, const void* v, void* k_pool, void* v_pool,
                              const int32_t* page_table, int32_t num_pages, int32_t ps_log2,
                              int32_t hkv, int64_t start_pos, int64_t n, int num_sms,
                              uint32_t* err, cudaStream_t st);

cudaError_t ls_launch_wait_timeout(uint32_t* err, cudaStream_t stream);
cudaError_t ls_launch_grpo_logp(const void* logits, bool is_bf16, int64_t T, int V,
                                const int32_t* targets, const float* ref_logp, float* logp_out,
                                float* lse_out, float* kl_out, uint32_t* err, int num_sms,
                                cudaStream_t stream);
cudaError_t ls_launch_validate_pages(const int32_t* page_table, int32_t num_logical,
                                     int32_t num_pages, uint32_t* seen, uint32_t* err,
                                     cudaStream_t st);

cudaError_t ls_launch_replay_fwd(const LsAttnArgs& a, const LsSched& sc, const LsFwdOut& out,
                                 cudaStream_t st);

cudaError_t ls_launch_bwd_dq(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                             cudaStream_t st);
// sc.ctas counts pairs here.
cudaError_t ls_launch_bwd_dq_pair(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                                  cudaStream_t st);

// Response-key dK / dV (tcgen05) and the bytes of its partial-sum workspace.
size_t ls_dkdv_part_bytes(int R, int hq, int hkv, int num_sms, const LsSegs* segs);
cudaError_t ls_launch_bwd_dkdv(const LsAttnArgs& a, const LsSegs& seg, const LsBwdIn& b,
                               int num_sms, cudaStream_t st);

cudaError_t ls_launch_replay_bwd(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                                 int num_sms, cudaStream_t st);

struct LsGrpoArgs {
  const void* logits;
  int32_t is_bf16;
  int64_t T;
  int32_t V;
  const int32_t* targets;
  const float* logp_old;
  const float* rewards;
  const int32_t* resp_lens;
  int32_t G, member_begin, member_end;
  float eps;
  double adv_eps;
  int32_t std_ddof;
  int32_t accumulate_loss;
  float* loss;
  void* dlogits;
  float* logp_out;
  float* stats;
  void* workspace;
  uint32_t* err;
};
size_t ls_grpo_ws_bytes(int64_t T, int G);
cudaError_t ls_launch_grpo(const LsGrpoArgs& a, int num_sms, cudaStream_t st);

// Gated-DeltaNet replay (gdn_replay.cu): head dims 128 (d_k = d_v), 64-token chunks.
struct LsGdnArgs {
  const float* state0;  // [H][128][128] (d_v x d_k): the captured state
  const void* q;        // bf16 [R][H][128]
  const void* k;
  const void* v;
  const float* g;       // [R][H] log decay
  const float* beta;    // [R][H]
  int32_t R, H;
  float scale;
  uint32_t* err;        // device error word (bounded pipeline waits report here)
};
size_t ls_gdn_ws_bytes(int R, int H, bool bwd);
cudaError_t ls_launch_gdn_fwd(const LsGdnArgs& a, void* o, float* state_out, void* ws,
                              cudaStream_t st);
cudaError_t ls_launch_gdn_bwd(const LsGdnArgs& a, const void* d_o, int accumulate, float* dq,
                              float* dk, float* dv, float* dg, float* dbeta, void* ws,
                              cudaStream_t st);

// Latent (MLA-style) replay forward (mla_replay.cu): rows of 576 bf16 values (512 latent
// + 64 rotary), outputs of 512; units = (128 token-major (t, h) rows) x (half of the
// output columns), unit u covering row tile u >> 1 and half u & 1.
struct LsMlaArgs {
  const void* pool;           // bf16 [num_pages][page_size][576]
  const int32_t* page_table;  // [ceil(P / page_size)]
  int32_t num_pages, ps_log2;
  int64_t P;
  const void* q;              // bf16 [R][H][576]
  const void* lat_resp;       // bf16 [R][576]
  int32_t R, H;
  float scale_log2;           // softmax scale x log2(e)
  void* o;                    // bf16 [R][H][512]
  float* lse;                 // [R][H]
  float* part_o;              // [pieces][128][256] partials of tail-unit pieces
  float* part_lse;            // [pieces][128]
  uint32_t* err;
};
int ls_mla_tile();
int ls_mla_unit_rows();
int ls_mla_half();
cudaError_t ls_launch_mla_fwd(const LsMlaArgs& a, const LsSched& sc, cudaStream_t st);
cudaError_t ls_launch_capture_latent(const void* src, void* pool, const int32_t* page_table,
                                     int32_t num_pages, int32_t ps_log2, int64_t start,
                                     int64_t n, int sms, uint32_t* err, cudaStream_t st);

// Latent replay backward (mla_replay_bwd.cu).
struct LsMlaBwdArgs {
  const void* pool;           // bf16 [num_pages][page_size][576]
  const int32_t* page_table;  // [ceil(P / page_size)]
  int32_t num_pages, ps_log2;
  int64_t P;
  const void* q;              // bf16 [R][H][576]
  const void* lat_resp;       // bf16 [R][576]
  const void* o;              // bf16 [R][H][512], the forward's output
  const float* lse;           // [R][H]
  const void* d_o;            // bf16 [R][H][512]
  int32_t R, H;
  float scale, scale_log2;
  float* delta;               // [R][H]: <dO, o>
  float* dq;                  // [R][H][576]
  float* dlat;                // [R][576]
  float* part_dq;             // [pieces][64][576] partials of tail-unit pieces
  float* part_dlat;           // [2 x d lat CTAs][128][320]
  uint32_t* err;
};
int ls_mla_bwd_tile();
int ls_mla_bwd_unit_rows();
int ls_mla_bwd_part_cols();
int ls_mla_bwd_dlat_ctas(int32_t R, int32_t H, int sms);
cudaError_t ls_launch_mla_bwd(const LsMlaBwdArgs& a, const LsSched& sc, int sms, cudaStream_t st);
