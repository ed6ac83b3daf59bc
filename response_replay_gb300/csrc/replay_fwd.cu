// replay_fwd.cu -- replay attention forward: one response branch over the captured
// prompt pages plus causal self-attention, split-KV partials merged by log-sum-exp.
//
// Definition (LongStraw explainer, "Serial replay makes G a schedule" and "Two
// incompatible architectures", Qwen bullet; paper digest, Method step 3):
//   s_{t,j} = scale <q_{t,h}, k_{j,h/g}>,  j over all prompt positions and response j <= t
//   lse_t = log sum_j exp(s_{t,j}),  o_t = sum_j exp(s_{t,j} - lse_t) v_j
//
// Kernel: a unit is 64 consecutive response tokens of one query head; a CTA of 4 warps
// owns one unit at a time (16 query rows per warp) and streams 64-key tiles of K and V
// through double-buffered shared memory (cp.async 16-byte gathers through the page
// table; rows past the prompt or response end are zero-filled).  S = Q K^T and O += P V
// run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate); the online
// softmax keeps (max, sum) per row in the log2 domain.  Work is spread by the
// full-waves + split-tail schedule of ls_sched.h; units split across CTAs are merged by
// replay_fwd_combine.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"

namespace {

constexpr int kD = 128;
constexpr int kBM = 64;     // query rows per unit
constexpr int kBN = 64;     // keys per tile
constexpr int kThreads = 128;
constexpr int kTileBytes = kBM * kD * 2;  // 16 KB
constexpr int kSmem = kTileBytes * 5;     // Q + 2 x (K, V)
constexpr float kLn2 = 0.6931471805599453f;

// Decoded unit: query head h (kv head kvh), response tokens [t0, t0 + 64).
struct Unit {
  int h, kvh, t0;
};
__device__ __forceinline__ Unit decode_unit(const LsAttnArgs& a, int u) {
  const int nTB = (a.R + kBM - 1) / kBM;
  Unit x;
  x.h = u / nTB;
  x.t0 = (u % nTB) * kBM;
  x.kvh = x.h / a.g;
  return x;
}

// Gather 64 rows x 256 bytes of K and V into swizzled shared tiles.
// Prompt tile: positions [p0, p0 + 64) through the page table; response tile: keys
// [p0, p0 + 64) of k_resp / v_resp.  Invalid rows are zero-filled.
__device__ __forceinline__ void load_kv_tile(const LsAttnArgs& a, int kvh, bool response,
                                             int64_t p0, uint32_t ks, uint32_t vs) {
  const int tid = threadIdx.x;
  const int64_t ps_mask = (1ll << a.ps_log2) - 1;
#pragma unroll
  for (int it = 0; it < (kBN * 16) / kThreads; ++it) {
    const int i = tid + it * kThreads;
    const int r = i >> 4, c = i & 15;
    const int64_t p = p0 + r;
    const __nv_bfloat16* ksrc = static_cast<const __nv_bfloat16*>(a.k_resp);
    const __nv_bfloat16* vsrc = static_cast<const __nv_bfloat16*>(a.v_resp);
    int64_t off = 0;
    uint32_t bytes = 0;
    if (response) {
      if (p < a.R) {
        off = (p * a.hkv + kvh) * kD + c * 8;
        bytes = 16;
      }
    } else if (p < a.P) {
      const int32_t phys = __ldg(a.page_table + (p >> a.ps_log2));
      if ((uint32_t)phys < (uint32_t)a.num_pages) {
        off = ((((int64_t)phys * a.hkv + kvh) << a.ps_log2) + (p & ps_mask)) * kD + c * 8;
        bytes = 16;
        ksrc = static_cast<const __nv_bfloat16*>(a.k_pool);
        vsrc = static_cast<const __nv_bfloat16*>(a.v_pool);
      } else {
        ls_report(a.err, LS_DEVERR_CHECK);
      }
    }
    cp_async16(ks + swz(r, c), ksrc + off, bytes);
    cp_async16(vs + swz(r, c), vsrc + off, bytes);
  }
}

__device__ __forceinline__ void load_q_tile(const LsAttnArgs& a, const Unit& un, uint32_t qs) {
  const int tid = threadIdx.x;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
  for (int it = 0; it < (kBM * 16) / kThreads; ++it) {
    const int i = tid + it * kThreads;
    const int r = i >> 4, c = i & 15;
    const int t = un.t0 + r;
    const bool ok = t < a.R;
    cp_async16(qs + swz(r, c), q + (ok ? ((int64_t)t * a.hq + un.h) * kD + c * 8 : 0), ok ? 16 : 0);
  }
}

__global__ void __launch_bounds__(kThreads, 2)
replay_fwd_kernel(const LsAttnArgs a, const LsSched sc, const LsFwdOut out) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t qs = smem_u32(smem);
  const uint32_t ks[2] = {qs + kTileBytes, qs + 3 * kTileBytes};
  const uint32_t vs[2] = {qs + 2 * kTileBytes, qs + 4 * kTileBytes};
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lr = lane >> 2;           // fragment row within 8
  const int lc = (lane & 3) * 2;      // fragment column pair

  LsWalk walk(sc, blockIdx.x);
  int u, s;
  bool first, last, complete;
  uint32_t qa[8][4];                  // Q fragments of this warp's 16 rows
  float o[16][4];
  // Row max (log2 domain) and row sum.  The sum runs over up to millions of keys per
  // thread, so it is kept as an unevaluated pair l + lcomp (Fast2Sum per tile): a plain
  // fp32 accumulator loses ~1e-3 relative at P = 2M.
  float m[2], l[2], lcomp[2];
  Unit un{0, 0, 0};
  while (walk.next(&u, &s, &first, &last, &complete)) {
    if (first) {
      un = decode_unit(a, u);
      __syncthreads();                // previous unit's smem reads are done
      load_q_tile(a, un, qs);
      cp_async_commit();
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = lcomp[0] = lcomp[1] = 0.f;
    }
    // KV tile range of this item
    const bool response = (s == sc.nsplit);
    int64_t k0, k1;
    if (response) {
      k0 = 0;
      const int64_t qe = (int64_t)un.t0 + kBM;
      k1 = qe < a.R ? qe : a.R;
    } else {
      int t0, t1;
      sc.split_tiles(s, &t0, &t1);
      k0 = (int64_t)t0 * kBN;
      k1 = (int64_t)t1 * kBN;
      if (k1 > a.P) k1 = a.P;
    }
    const int ntile = (int)((k1 - k0 + kBN - 1) / kBN);
    __syncthreads();                  // K/V buffers free
    if (ntile > 0) load_kv_tile(a, un.kvh, response, k0, ks[0], vs[0]);
    cp_async_commit();
    for (int it = 0; it < ntile; ++it) {
      const int buf = it & 1;
      if (it + 1 < ntile) load_kv_tile(a, un.kvh, response, k0 + (int64_t)(it + 1) * kBN, ks[buf ^ 1], vs[buf ^ 1]);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      if (first && it == 0) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ldsm_x4(qs + swz(warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * kk + (lane >> 4)),
                  qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
      // S = Q K^T  (16 x 64 per warp)
      float sacc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int nn = 0; nn < 4; ++nn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ks[buf] + swz(nn * 16 + (lane & 7) + (lane >> 4) * 8, 2 * kk + ((lane >> 3) & 1)),
                  b0, b1, b2, b3);
          mma16816(sacc[2 * nn], qa[kk], b0, b1);
          mma16816(sacc[2 * nn + 1], qa[kk], b2, b3);
        }
      }
      // mask + online softmax (log2 domain)
      const int64_t kt = k0 + (int64_t)it * kBN;
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t key = kt + j * 8 + lc + (e & 1);
          const int row = warp * 16 + lr + (e >> 1) * 8;
          bool ok;
          if (response) ok = key <= (int64_t)un.t0 + row && key < a.R;
          else ok = key < a.P;
          const float x = ok ? sacc[j][e] * a.scale_log2 : -INFINITY;
          sacc[j][e] = x;
          mx[e >> 1] = fmaxf(mx[e >> 1], x);
        }
      }
      float alpha[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
        const float mn = fmaxf(m[r], mx[r]);
        alpha[r] = fast_exp2(m[r] - mn);
        m[r] = mn;
        l[r] *= alpha[r];
        lcomp[r] *= alpha[r];
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= alpha[0]; o[j][1] *= alpha[0];
        o[j][2] *= alpha[1]; o[j][3] *= alpha[1];
      }
      float ls[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p = fast_exp2(sacc[j][e] - m[e >> 1]);
          sacc[j][e] = p;
          ls[e >> 1] += p;
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {   // Fast2Sum: l + lcomp += ls
        const float t = l[r] + ls[r];
        lcomp[r] += (l[r] - t) + ls[r];
        l[r] = t;
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sacc[2 * kk][0], sacc[2 * kk][1]);
        pa[1] = pack_bf16(sacc[2 * kk][2], sacc[2 * kk][3]);
        pa[2] = pack_bf16(sacc[2 * kk + 1][0], sacc[2 * kk + 1][1]);
        pa[3] = pack_bf16(sacc[2 * kk + 1][2], sacc[2 * kk + 1][3]);
#pragma unroll
        for (int dn = 0; dn < 8; ++dn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vs[buf] + swz(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * dn + (lane >> 4)),
                    b0, b1, b2, b3);
          mma16816(o[2 * dn], pa, b0, b1);
          mma16816(o[2 * dn + 1], pa, b2, b3);
        }
      }
      __syncthreads();                // buffer `buf` may be refilled next iteration
    }
    cp_async_wait<0>();

    if (last) {
      float lt[2], lse[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lt[r] = l[r] + lcomp[r];
        lt[r] += __shfl_xor_sync(0xffffffffu, lt[r], 1);
        lt[r] += __shfl_xor_sync(0xffffffffu, lt[r], 2);
        lse[r] = (m[r] + log2f(lt[r])) * kLn2;
      }
      const float inv[2] = {1.f / lt[0], 1.f / lt[1]};
      if (complete) {
        __nv_bfloat16* og = static_cast<__nv_bfloat16*>(out.o);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int t = un.t0 + warp * 16 + lr + r * 8;
          if (t < a.R) {
            const int64_t row = (int64_t)t * a.hq + un.h;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              *reinterpret_cast<uint32_t*>(og + row * kD + j * 8 + lc) =
                  pack_bf16(o[j][2 * r] * inv[r], o[j][2 * r + 1] * inv[r]);
            }
            if ((lane & 3) == 0) out.lse[row] = lse[r];
          }
        }
      } else {
        const int slot = sc.slot_of(blockIdx.x, u);
        float* po = out.part_o + (int64_t)slot * kBM * kD;
        float* pl = out.part_lse + (int64_t)slot * kBM;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int row = warp * 16 + lr + r * 8;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            *reinterpret_cast<float2*>(po + row * kD + j * 8 + lc) =
                make_float2(o[j][2 * r] * inv[r], o[j][2 * r + 1] * inv[r]);
          if ((lane & 3) == 0) pl[row] = lse[r];
        }
      }
    }
  }
}

// Merge the partial (o, lse) of every tail unit split across CTAs:
//   lse = log sum_c exp(lse_c),  o = sum_c exp(lse_c - lse) o_c.
// One block per tail unit, one thread per head_dim column; fixed merge order.
__global__ void __launch_bounds__(kD) replay_fwd_combine(const LsAttnArgs a, const LsSched sc,
                                                         const LsFwdOut out) {
  const int u = sc.tail_unit0() + blockIdx.x;
  const int64_t ipu = sc.items_per_unit();
  const int64_t i0 = (int64_t)(u - sc.tail_unit0()) * ipu;
  const int c_lo = sc.tail_cta_of(i0), c_hi = sc.tail_cta_of(i0 + ipu - 1);
  if (c_lo == c_hi) return;          // written whole by one CTA
  const Unit un = decode_unit(a, u);
  const int col = threadIdx.x;
  for (int r = 0; r < kBM; ++r) {
    const int t = un.t0 + r;
    if (t >= a.R) break;
    float mx = -INFINITY;
    for (int c = c_lo; c <= c_hi; ++c)
      if (sc.tail_nonempty(c)) mx = fmaxf(mx, out.part_lse[(int64_t)sc.slot_of(c, u) * kBM + r]);
    float sum = 0.f;
    for (int c = c_lo; c <= c_hi; ++c)
      if (sc.tail_nonempty(c)) sum += expf(out.part_lse[(int64_t)sc.slot_of(c, u) * kBM + r] - mx);
    const float lse = mx + logf(sum);
    float acc = 0.f;
    for (int c = c_lo; c <= c_hi; ++c) {
      if (!sc.tail_nonempty(c)) continue;
      const int64_t slot = sc.slot_of(c, u);
      acc += expf(out.part_lse[slot * kBM + r] - lse) * out.part_o[(slot * kBM + r) * kD + col];
    }
    const int64_t row = (int64_t)t * a.hq + un.h;
    static_cast<__nv_bfloat16*>(out.o)[row * kD + col] = __float2bfloat16_rn(acc);
    if (col == 0) out.lse[row] = lse;
  }
}

}  // namespace

int ls_fwd_unit_rows() { return kBM; }
int ls_fwd_tile() { return kBN; }
int ls_fwd_ctas_per_sm() { return 2; }
int ls_num_units(int R, int hq, int hkv, int unit_rows) {
  (void)hkv;
  return hq * ((R + unit_rows - 1) / unit_rows);
}

cudaError_t ls_launch_replay_fwd(const LsAttnArgs& a, const LsSched& sc, const LsFwdOut& out,
                                 cudaStream_t st) {
  cudaError_t e0 = cudaFuncSetAttribute(replay_fwd_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e0 != cudaSuccess) return e0;
  replay_fwd_kernel<<<sc.ctas, kThreads, kSmem, st>>>(a, sc, out);
  ls_note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t tail_units = sc.units - (int64_t)sc.waves * sc.ctas;
  if (tail_units > 0) {
    replay_fwd_combine<<<(unsigned)tail_units, kD, 0, st>>>(a, sc, out);
  ls_note_launch();
    e = cudaGetLastError();
  }
  return e;
}
