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
//   bwd_delta     D = rowsum(dO * O) per (t, h), one warp per row.
//   dQ            replay_bwd_dq_tc.cu: q-stationary tcgen05 kernel over prompt and
//                 response keys, same schedule as the forward, plus its split combine.
//   bwd_dkdv      key-stationary over response keys only: a CTA owns 64 response keys
//                 of one kv head and walks the query blocks t >= j of every query
//                 head in the group; dV += P^T dO, dK += dS^T Q.  This part is the
//                 causal R x R triangle (under 0.2% of the work at P = 2M, R = 4096)
//                 and uses warp-level mma.sync m16n8k16 (bf16 in, fp32 accumulate).
// Deterministic: no atomics.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace {

constexpr int kD = 128;
constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kThreads = 128;
constexpr int kTileBytes = 64 * kD * 2;
constexpr float kLog2e = 1.4426950408889634f;

// 64 rows of bf16 [row][128] (row stride `pitch` elements) into a swizzled tile;
// rows >= nvalid are zero-filled.
__device__ __forceinline__ void load_rows(const __nv_bfloat16* base, int64_t pitch, int nvalid,
                                          uint32_t dst) {
#pragma unroll
  for (int it = 0; it < (64 * 16) / kThreads; ++it) {
    const int i = threadIdx.x + it * kThreads;
    const int r = i >> 4, c = i & 15;
    const bool ok = r < nvalid;
    cp_async16(dst + swz(r, c), base + (ok ? r * pitch + c * 8 : 0), ok ? 16 : 0);
  }
}

// ------------------------------------------------------------------ D = <dO, O>
__global__ void bwd_delta(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
                          int64_t rows, float* __restrict__ delta) {
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
    if (lane == 0) delta[r] = s;
  }
}

// ------------------------------------------------------------------ dK, dV (response keys)
constexpr int kKvSmem = 6 * kTileBytes + 2 * 2 * 64 * 4;  // K, V, 2 x (Q, dO), 2 x (lse2, D)

__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const LsAttnArgs a, const LsBwdIn b) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t ks = smem_u32(smem), vs = ks + kTileBytes;
  const uint32_t qs[2] = {ks + 2 * kTileBytes, ks + 4 * kTileBytes};
  const uint32_t dos[2] = {ks + 3 * kTileBytes, ks + 5 * kTileBytes};
  float* rowstat = reinterpret_cast<float*>(smem + 6 * kTileBytes);  // [2][2][64]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lr = lane >> 2, lc = (lane & 3) * 2;
  const int nKB = (a.R + kBN - 1) / kBN;
  const int kvh = blockIdx.x / nKB;
  const int j0 = (blockIdx.x % nKB) * kBN;
  const int nQB = (a.R + kBM - 1) / kBM;
  const int qb0 = j0 / kBM;
  const int nsteps = a.g * (nQB - qb0);

  // this CTA's 64 response keys / values
  {
    const int nv = a.R - j0 < kBN ? a.R - j0 : kBN;
    load_rows(static_cast<const __nv_bfloat16*>(a.k_resp) + ((int64_t)j0 * a.hkv + kvh) * kD,
              (int64_t)a.hkv * kD, nv, ks);
    load_rows(static_cast<const __nv_bfloat16*>(a.v_resp) + ((int64_t)j0 * a.hkv + kvh) * kD,
              (int64_t)a.hkv * kD, nv, vs);
  }
  auto load_step = [&](int step, int buf) {
    const int h = kvh * a.g + step / (nQB - qb0);
    const int t0 = (qb0 + step % (nQB - qb0)) * kBM;
    const int nv = a.R - t0 < kBM ? a.R - t0 : kBM;
    load_rows(static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)t0 * a.hq + h) * kD,
              (int64_t)a.hq * kD, nv, qs[buf]);
    load_rows(static_cast<const __nv_bfloat16*>(b.d_o) + ((int64_t)t0 * a.hq + h) * kD,
              (int64_t)a.hq * kD, nv, dos[buf]);
    if (tid < 64) {
      const int t = t0 + tid;
      const int64_t row = (int64_t)(t < a.R ? t : a.R - 1) * a.hq + h;
      rowstat[buf * 128 + tid] = b.lse[row] * kLog2e;
      rowstat[buf * 128 + 64 + tid] = b.delta[row];
    }
  };
  float dk[16][4], dv[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[j][e] = dv[j][e] = 0.f;

  load_step(0, 0);
  cp_async_commit();
  for (int step = 0; step < nsteps; ++step) {
    const int buf = step & 1;
    if (step + 1 < nsteps) load_step(step + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int t0 = (qb0 + step % (nQB - qb0)) * kBM;
    const float* l2 = rowstat + buf * 128;
    const float* dd = rowstat + buf * 128 + 64;
    // S^T = K Q^T and dP^T = V dO^T (16 keys x 64 queries per warp)
    float sacc[8][4], pacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[j][e] = pacc[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t ka[4], va[4];
      const uint32_t arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      ldsm_x4(ks + swz(arow, 2 * kk + (lane >> 4)), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(vs + swz(arow, 2 * kk + (lane >> 4)), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int nn = 0; nn < 4; ++nn) {
        uint32_t b0, b1, b2, b3;
        const int brow = nn * 16 + (lane & 7) + (lane >> 4) * 8;
        const int bch = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(qs[buf] + swz(brow, bch), b0, b1, b2, b3);
        mma16816(sacc[2 * nn], ka, b0, b1);
        mma16816(sacc[2 * nn + 1], ka, b2, b3);
        ldsm_x4(dos[buf] + swz(brow, bch), b0, b1, b2, b3);
        mma16816(pacc[2 * nn], va, b0, b1);
        mma16816(pacc[2 * nn + 1], va, b2, b3);
      }
    }
    // P^T and dS^T; key j = j0 + row, query t = t0 + col; visible iff j <= t < R
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = j * 8 + lc + (e & 1);
        const int key = j0 + warp * 16 + lr + (e >> 1) * 8;
        const int t = t0 + col;
        const bool ok = key <= t && t < a.R;
        const float p = ok ? fast_exp2(sacc[j][e] * a.scale_log2 - l2[col]) : 0.f;
        sacc[j][e] = p;
        pacc[j][e] = p * (pacc[j][e] - dd[col]);
      }
    }
    // dV += P^T dO, dK += dS^T Q  (k = queries)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4], sa[4];
      pa[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
      pa[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
      pa[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
      pa[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
      sa[0] = pack_bf16(pacc[2 * kk][0], pacc[2 * kk][1]);
      sa[1] = pack_bf16(pacc[2 * kk][2], pacc[2 * kk][3]);
      sa[2] = pack_bf16(pacc[2 * kk + 1][0], pacc[2 * kk + 1][1]);
      sa[3] = pack_bf16(pacc[2 * kk + 1][2], pacc[2 * kk + 1][3]);
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        uint32_t b0, b1, b2, b3;
        const int trow = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int tch = 2 * dn + (lane >> 4);
        ldsm_x4_t(dos[buf] + swz(trow, tch), b0, b1, b2, b3);
        mma16816(dv[2 * dn], pa, b0, b1);
        mma16816(dv[2 * dn + 1], pa, b2, b3);
        ldsm_x4_t(qs[buf] + swz(trow, tch), b0, b1, b2, b3);
        mma16816(dk[2 * dn], sa, b0, b1);
        mma16816(dk[2 * dn + 1], sa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int key = j0 + warp * 16 + lr + r * 8;
    if (key < a.R) {
      float* pk = b.dk + ((int64_t)key * a.hkv + kvh) * kD;
      float* pv = b.dv + ((int64_t)key * a.hkv + kvh) * kD;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float2 vk = make_float2(dk[j][2 * r] * a.scale, dk[j][2 * r + 1] * a.scale);
        float2 vv = make_float2(dv[j][2 * r], dv[j][2 * r + 1]);
        float2* qk = reinterpret_cast<float2*>(pk + j * 8 + lc);
        float2* qv = reinterpret_cast<float2*>(pv + j * 8 + lc);
        if (b.accumulate) {
          const float2 ok = *qk, ov = *qv;
          vk.x += ok.x; vk.y += ok.y;
          vv.x += ov.x; vv.y += ov.y;
        }
        *qk = vk;
        *qv = vv;
      }
    }
  }
}

}  // namespace


cudaError_t ls_launch_replay_bwd(const LsAttnArgs& a, const LsSched& sc, const LsBwdIn& b,
                                 int num_sms, cudaStream_t st) {
  const int64_t rows = (int64_t)a.R * a.hq;
  int blocks = (int)((rows + 7) / 8);
  if (blocks > num_sms * 16) blocks = num_sms * 16;
  bwd_delta<<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(b.o),
                                    static_cast<const __nv_bfloat16*>(b.d_o), rows, b.delta);
  ls_note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = ls_launch_bwd_dq(a, sc, b, st);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem);
  if (e != cudaSuccess) return e;
  const int nKB = (a.R + kBN - 1) / kBN;
  bwd_dkdv_kernel<<<a.hkv * nKB, kThreads, kKvSmem, st>>>(a, b);
  ls_note_launch();
  return cudaGetLastError();
}
