// grpo_noalloc.cu -- ls_grpo_loss_fwd_bwd_noalloc: the fused GRPO loss / logits
// gradient for callers that cannot give the library any device memory of its own.
//
// Some callers cannot call cudaMalloc (or ask their framework for a buffer) at the
// point where they compute the loss: for example a training loop whose device memory
// is planned once by its host framework and then frozen, so that no new allocation
// may appear mid-step, or a plug-in that is only handed its input and output tensors.
// For them this entry point keeps its scratch space in a fixed array that lives in the
// library's own device image; it allocates nothing and frees nothing.
//
// The scratch (per-member advantages and offsets, per-token terms and ratios) is
// kScratchBytes = 4 MiB + 128 KiB per device, which covers any call with
// T <= kMaxTokens (262,144) tokens and G <= kMaxMembers (1,024) members; larger calls
// are rejected with LS_ERR_WORKSPACE before anything is launched.  Every GPU that loads
// the library holds this array until the process exits.  Every call shares it: two
// calls whose kernels overlap on the GPU (different streams without ordering) race on
// it, so order them.  No field of the scratch has to start at zero: each call writes
// every field it later reads, so the contents left by the previous call do no harm.
#include <mutex>

#include "../../include/longstraw.h"
#include "ls_internal.h"

namespace {

constexpr int64_t kMaxTokens = 262144;
constexpr int kMaxMembers = 1024;
constexpr size_t kScratchBytes = (4u << 20) + (128u << 10);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_grpo_scratch[kScratchBytes];

// Device address of g_grpo_scratch for each device (the name itself is only a host
// stand-in); looked up once per device with that device current.
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

ls_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_grpo_scratch) != cudaSuccess || !p) return LS_ERR_CUDA;
    if (ls_grpo_ws_bytes(kMaxTokens, kMaxMembers) > kScratchBytes) return LS_ERR_UNSUPPORTED;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LS_OK;
}

}  // namespace

extern "C" ls_status ls_grpo_loss_fwd_bwd_noalloc(
    const void* logits, ls_dtype dtype, int64_t T, int V, const int32_t* targets,
    const float* logp_old, const float* rewards, const int32_t* resp_lens, int G,
    int member_begin, int member_end, float eps, float adv_eps, int std_ddof,
    int accumulate_loss, float* loss, void* dlogits, float* logp_out, float* stats,
    ls_stream_t stream) {
  if (T < 0 || G <= 0) return LS_ERR_INVALID_ARG;
  if (T > kMaxTokens || G > kMaxMembers) return LS_ERR_WORKSPACE;
  void* scratch = nullptr;
  const ls_status s = scratch_address(&scratch);
  if (s != LS_OK) return s;
  return ls_grpo_loss_fwd_bwd(logits, dtype, T, V, targets, logp_old, rewards, resp_lens, G,
                              member_begin, member_end, eps, adv_eps, std_ddof, accumulate_loss,
                              loss, dlogits, logp_out, stats, scratch, kScratchBytes, stream);
}
