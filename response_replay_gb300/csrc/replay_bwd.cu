// replay_bwd.cu -- replay attention backward with the prompt state stopgrad.
//
// Only the conditional response gradient is formed: the captured prompt state is
// detached (LongStraw paper digest, Method, last paragraph; explainer, Figure 2
// caption), so prompt keys/values get no gradient and K/V gradients exist only for
// the response's own keys (explainer, "Two incompatible architectures", Qwen bullet).
// With P_{t,j} = exp(s_{t,j} - lse_t), D_t = <dO_t, O_t>, dS = P (dO v_j - D_t):
//   dq_t = scale sum_j dS_{t,j} k_j                 over prompt and response keys
//   dk_j = scale sum_{h in group, t >= j} dS_{t,j} q_t,  dv_j = sum P_{t,j} dO_t
//
// Launches:
//   bwd_delta     D = rowsum(dO * O) per (t, h), one warp per row; also writes D and
//                 lse log2(e) transposed ([head][token], padded to whole 128-token tiles
//                 with 0 / +inf) for the response-key kernel.
//   dQ            replay_bwd_dq_pair.cu (CTA pairs) or replay_bwd_dq_tc.cu (one CTA):
//                 q-stationary tcgen05 kernel over prompt and response keys, the
//                 forward's kind of schedule, plus its split combine.
//   dK, dV        replay_bwd_dkdv_tc.cu: key-stationary tcgen05 kernel over the causal
//                 R x R triangle of the response's own keys, plus its split combine.
// Deterministic: no atomics.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace {

constexpr int kD = 128;
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ D = <dO, O>
// delta [R][hq]; dt, lse2t [hq][rp] (transposed; tokens R..rp-1 padded with 0 / +inf).
__global__ void bwd_delta(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
                          const float* __restrict__ lse, int64_t rows, int32_t hq, int32_t R,
                          int32_t rp, float* __restrict__ delta, float* __restrict__ dt,
                          float* __restrict__ lse2t) {
  const int lane = threadIdx.x & 31;
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows;
       r += (int64_t)gridDim.x * (blockDim.x / 32)) {
    const uint2 ov = *reinterpret_cast<const uint2*>(o + r * kD + lane * 4);
    const uint2 dv = *reinterpret_cast<const uint2*>(d_o + r * kD + lane * 4);
    const uint32_t ow[2] = {ov.x, ov.y}, dw[2] = {dv.x, dv.y};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      s += __uint_as_float(ow[i] << 16) * __uint_as_float(dw[i] << 16);
      s += __uint_as_float(ow[i] & 0xffff0000u) * __uint_as_float(dw[i] & 0xffff0000u);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      const int64_t t = r / hq, h = r - t * hq;
      delta[r] = s;
      dt[h * rp + t] = s;
      lse2t[h * rp + t] = lse[r] * kLog2e;
    }
  }
  const int64_t pad = (int64_t)hq * (rp - R);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pad;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t h = i / (rp - R), t = R + (i - h * (rp - R));
    dt[h * rp + t] = 0.f;
    lse2t[h * rp + t] = INFINITY;
  }
}

}  // namespace


cudaError_t ls_launch_replay_bwd(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                                 int num_sms, cudaStream_t st) {
  const int64_t rows = (int64_t)a.R * a.hq;
  int blocks = (int)((rows + 7) / 8);
  if (blocks > num_sms * 16) blocks = num_sms * 16;
  const int32_t rp = (a.R + 127) / 128 * 128;
  bwd_delta<<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(b.o),
                                    static_cast<const __nv_bfloat16*>(b.d_o), b.lse, rows, a.hq,
                                    a.R, rp, b.delta, b.dt, b.lse2t);
  ls_note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = b.pair ? ls_launch_bwd_dq_pair(a, sc, b, st) : ls_launch_bwd_dq(a, sc, b, st);
  if (e != cudaSuccess) return e;
  return ls_launch_bwd_dkdv(a, sc.seg, b, num_sms, st);
}
