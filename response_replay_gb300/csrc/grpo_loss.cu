// grpo_loss.cu -- fused token-level clipped GRPO surrogate and its logits gradient.
//
// Loss (LongStraw paper digest, "Method", the L_policy equation):
//   L = -(1/G) sum_i (1/R_i) sum_t min(rho A_i, clip(rho, 1-eps, 1+eps) A_i),
//   rho = exp(logp - logp_old), logp = z_target - logsumexp(z),
//   A_i = (r_i - mean r) / (std r + adv_eps)  (group-relative advantages).
// Gradient: dL/dz_v = c_t (1[v == target] - softmax_v), c_t = -A_i rho / (G R_i) when
// the unclipped term is the active minimum, 0 when the clip holds the term constant.
//
// Launches:
//   grpo_prep   1 warp  : advantages in fp64 (mean/std about the first reward), member
//                         token offsets, 1/(G R_i); checks that lengths cover T; zeroes
//                         the row kernel's ticket.
//   row kernel  grid    : pass 1 reduces a token row (online max / sum-exp) and gathers
//                         z_target; pass 2 writes dlogits, or zeros without reading the
//                         row when c_t = 0.  HBM: V*b read + V*b written per token, the
//                         algorithmic floor.  Two forms:
//     grpo_stream        one CTA per SM, rows streamed through a shared-memory ring by
//                        bulk copies, the row's last chunks kept for pass 2; its last
//                        CTA to finish (ticket) also reduces the loss.  Used when a row
//                        is a whole number of 16-byte units.
//     grpo_rows          one CTA per row at a time, plain 16-byte loads, pass 2
//                        re-reading the row mostly from L2; any V.
//   grpo_final  1 block : the loss reduction as its own launch, after grpo_rows (or
//                         when T = 0).
// The reduction is a fixed-order fp64 sum of the per-token terms (no floating-point
// atomics), so results are deterministic.
#include <float.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_umma.cuh"

namespace {

constexpr int kRowThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct WsLayout {
  size_t flag, adv, inv_norm, off, term, rho, zeroed, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline WsLayout ws_layout(int64_t T, int G) {
  WsLayout w;
  size_t p = 0;
  w.flag = p;      p = align256(p + 16);
  w.adv = p;       p = align256(p + sizeof(double) * G);
  w.inv_norm = p;  p = align256(p + sizeof(double) * G);
  w.off = p;       p = align256(p + sizeof(int64_t) * (G + 1));
  w.term = p;      p = align256(p + sizeof(double) * (T > 0 ? T : 1));
  w.rho = p;       p = align256(p + sizeof(float) * (T > 0 ? T : 1));
  w.zeroed = p;    p = align256(p + sizeof(float) * (T > 0 ? T : 1));
  w.total = p;
  return w;
}

template <typename P>
__device__ __forceinline__ P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(base) + off);
}

// Sum over the 32 lanes of a warp in a fixed order (the same tree on every call).
__device__ __forceinline__ double warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// One warp: advantages in fp64 about the first reward (lane-strided sums, fixed-order
// tree), member token offsets by a warp scan over the member range, 1/(G R_i), the
// length check, and a zero ticket for the streamed kernel's last-CTA reduction.
__global__ void grpo_prep(const float* __restrict__ rewards, const int32_t* __restrict__ lens,
                          int G, int mb, int me, int std_ddof, double adv_eps, int64_t T,
                          void* ws, uint32_t* err) {
  const int lane = threadIdx.x;
  if (lane >= 32) return;
  const WsLayout w = ws_layout(T, G);
  int32_t* flag = at<int32_t>(ws, w.flag);
  double* adv = at<double>(ws, w.adv);
  double* inv = at<double>(ws, w.inv_norm);
  int64_t* off = at<int64_t>(ws, w.off);
  const double r0 = rewards[0];
  double sum = 0.0;
  for (int i = lane; i < G; i += 32) sum += (double)rewards[i] - r0;
  const double mean = warp_sum(sum) / G;
  double sq = 0.0;
  for (int i = lane; i < G; i += 32) {
    const double dev = ((double)rewards[i] - r0) - mean;
    sq += dev * dev;
  }
  const double var = warp_sum(sq) / (double)(G - std_ddof);
  const double sd = sqrt(var);
  for (int i = lane; i < G; i += 32) adv[i] = (((double)rewards[i] - r0) - mean) / (sd + adv_eps);
  int bad = 0;
  int64_t carry = 0;  // tokens of the members before this chunk
  if (lane == 0) off[0] = 0;
  for (int i0 = mb; i0 < me; i0 += 32) {
    const int i = i0 + lane;
    const int32_t n = i < me ? lens[i] : 0;
    bad |= n < 0;
    int64_t x = n > 0 ? n : 0;  // inclusive scan over the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (i < me) {
      off[i - mb + 1] = carry + x;
      inv[i] = n > 0 ? 1.0 / ((double)G * (double)n) : 0.0;
    }
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  bad = __any_sync(0xffffffffu, bad) || carry != T;
  if (lane == 0) {
    if (bad) ls_report(err, LS_DEVERR_CHECK);
    *flag = !bad;
    *at<uint32_t>(ws, w.flag + 4) = 0u;  // ticket
  }
}

template <typename E>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& u, float* x) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 pack(const float* x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
  __device__ static float load1(const float* p) { return *p; }
  __device__ static void store1(float* p, float x) { *p = x; }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 pack(const float* x) {
    return make_uint4(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                      pack_bf16(x[6], x[7]));
  }
  __device__ static float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void store1(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

// Online (max, sum of exp2) pair in the log2 domain.
struct MS {
  float m, s;
};
__device__ __forceinline__ MS ms_merge(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f};
  return {m, a.s * fast_exp2(a.m - m) + b.s * fast_exp2(b.m - m)};
}
__device__ __forceinline__ void ms_add(MS& a, const float* x2, int n) {
  float mx = x2[0];
  for (int i = 1; i < n; ++i) mx = fmaxf(mx, x2[i]);
  if (mx > a.m) {
    a.s *= fast_exp2(a.m - mx);
    a.m = mx;
  }
  if (a.m == -INFINITY) return;  // only -inf logits so far: they add nothing
  for (int i = 0; i < n; ++i) a.s += fast_exp2(x2[i] - a.m);
}

// Pass 1 over one row: the online (max, sum of exp2) of z log2e, reduced over the block;
// every thread receives the row's pair.  16-byte loads over the aligned body
// [head, tail0), scalar loads for the unaligned head and tail.  red must not be reused
// before the next __syncthreads.
template <typename E>
__device__ MS row_max_sumexp2(const E* __restrict__ zr, int V, int head, int nvec, int tail0,
                              MS* red) {
  using VT = Vec<E>;
  constexpr int NV = VT::N;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint4* zv = reinterpret_cast<const uint4*>(zr + head);
  MS ms = {-INFINITY, 0.f};
  for (int i = tid; i < head; i += kRowThreads) {
    float x = VT::load1(zr + i) * kLog2e;
    ms_add(ms, &x, 1);
  }
  for (int i = tail0 + tid; i < V; i += kRowThreads) {
    float x = VT::load1(zr + i) * kLog2e;
    ms_add(ms, &x, 1);
  }
  for (int i = tid; i < nvec; i += 4 * kRowThreads) {
    uint4 u[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (i + k * kRowThreads < nvec) u[k] = zv[i + k * kRowThreads];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (i + k * kRowThreads < nvec) {
        float x[NV];
        VT::unpack(u[k], x);
#pragma unroll
        for (int e = 0; e < NV; ++e) x[e] *= kLog2e;
        ms_add(ms, x, NV);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS other = {__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.s, o)};
    ms = ms_merge(ms, other);
  }
  if (lane == 0) red[wid] = ms;
  __syncthreads();
  if (wid == 0) {
    MS a = lane < kRowThreads / 32 ? red[lane] : MS{-INFINITY, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      MS other = {__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
      a = ms_merge(a, other);
    }
    if (lane == 0) red[kRowThreads / 32] = a;
  }
  __syncthreads();
  return red[kRowThreads / 32];
}

template <typename E>
__global__ void __launch_bounds__(kRowThreads) grpo_rows(
    const E* __restrict__ logits, int64_t T, int V, const int32_t* __restrict__ targets,
    const float* __restrict__ logp_old, int G, int mb, int me, float eps, E* __restrict__ dlogits,
    float* __restrict__ logp_out, void* ws, uint32_t* err) {
  using VT = Vec<E>;
  constexpr int NV = VT::N;
  const WsLayout w = ws_layout(T, G);
  if (*at<int32_t>(ws, w.flag) == 0) return;
  const double* adv = at<double>(ws, w.adv);
  const double* inv = at<double>(ws, w.inv_norm);
  const int64_t* off = at<int64_t>(ws, w.off);
  double* term_out = at<double>(ws, w.term);
  float* rho_out = at<float>(ws, w.rho);
  float* zeroed_out = at<float>(ws, w.zeroed);

  __shared__ MS red[kRowThreads / 32 + 1];
  __shared__ float s_bcast[2];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nm = me - mb;

  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const E* zr = logits + row * (int64_t)V;
    E* gr = dlogits + row * (int64_t)V;
    // 16-byte aligned body [h, h + nvec*NV), scalar head [0, h) and tail.
    const int h = (int)(((16 - (reinterpret_cast<uintptr_t>(zr) & 15)) & 15) / sizeof(E));
    const int head = h < V ? h : V;
    const int nvec = (V - head) / NV;
    const int tail0 = head + nvec * NV;
    const uint4* zv = reinterpret_cast<const uint4*>(zr + head);

    // ---- pass 1: online max / sum-exp (log2 domain)
    const MS a = row_max_sumexp2<E>(zr, V, head, nvec, tail0, red);
    if (wid == 0) {
      if (lane == 0) {
        // member of this token (binary search over the range's offsets)
        int lo = 0, hi = nm - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (off[mid] <= row) lo = mid; else hi = mid - 1;
        }
        const int mi = mb + lo;
        const float lse2 = a.m + log2f(a.s);
        const int32_t y = targets[row];
        float c = 0.f;
        double term = 0.0;
        float rho = 0.f, zeroed = 0.f;
        if ((uint32_t)y < (uint32_t)V) {
          const float logp = VT::load1(zr + y) - lse2 * kLn2;
          rho = expf(logp - logp_old[row]);
          const float A = (float)adv[mi];
          const float clipped = fminf(fmaxf(rho, 1.f - eps), 1.f + eps);
          const bool active = rho * A <= clipped * A;  // ties: the unclipped branch
          term = (double)(active ? rho : clipped) * adv[mi];
          c = active ? (float)(-adv[mi] * (double)rho * inv[mi]) : 0.f;
          zeroed = (!active && A != 0.f) ? 1.f : 0.f;
          if (logp_out) logp_out[row] = logp;
        } else {
          ls_report(err, LS_DEVERR_CHECK);
          if (logp_out) logp_out[row] = NAN;
        }
        term_out[row] = term;
        rho_out[row] = rho;
        zeroed_out[row] = zeroed;
        s_bcast[0] = c;
        s_bcast[1] = lse2;
      }
    }
    __syncthreads();
    const float c = s_bcast[0], lse2 = s_bcast[1];
    const int32_t y = targets[row];

    // ---- pass 2: dlogits = c (1[v == y] - exp2(z log2e - lse2))
    if (c == 0.f) {
      const uint4 zero = make_uint4(0, 0, 0, 0);
      uint4* gv = reinterpret_cast<uint4*>(gr + head);
      for (int i = tid; i < nvec; i += kRowThreads) __stcs(gv + i, zero);
      for (int i = tid; i < head; i += kRowThreads) VT::store1(gr + i, 0.f);
      for (int i = tail0 + tid; i < V; i += kRowThreads) VT::store1(gr + i, 0.f);
    } else {
      uint4* gv = reinterpret_cast<uint4*>(gr + head);
      // last-read chunk first: the end of the row is the likeliest to still be in L2
      constexpr int kChunk = 4 * kRowThreads;
      for (int i = (nvec - 1) / kChunk * kChunk + tid; i >= 0; i -= kChunk) {
        uint4 u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (i + k * kRowThreads < nvec) u[k] = __ldcs(zv + i + k * kRowThreads);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int vi = i + k * kRowThreads;
          if (vi < nvec) {
            float x[NV];
            VT::unpack(u[k], x);
            const int v0 = head + vi * NV;
#pragma unroll
            for (int e = 0; e < NV; ++e) {
              x[e] = -c * fast_exp2(fmaf(x[e], kLog2e, -lse2));
              if (v0 + e == y) x[e] += c;
            }
            __stcs(gv + vi, VT::pack(x));
          }
        }
      }
      for (int i = tid; i < head; i += kRowThreads) {
        float g = -c * fast_exp2(fmaf(VT::load1(zr + i), kLog2e, -lse2));
        VT::store1(gr + i, i == y ? g + c : g);
      }
      for (int i = tail0 + tid; i < V; i += kRowThreads) {
        float g = -c * fast_exp2(fmaf(VT::load1(zr + i), kLog2e, -lse2));
        VT::store1(gr + i, i == y ? g + c : g);
      }
    }
    __syncthreads();  // red / s_bcast reuse in the next row
  }
}

// Pre-step scoring: logp_t = z_{t,y} - logsumexp z_t for every token row (one read of
// the row), and with reference log-probabilities the per-token KL estimate
// kl_t = exp(d) - d - 1, d = ref_t - logp_t, evaluated as expm1(d) - d (no cancellation
// for small d).  A target outside [0, V) records LS_DEVERR_CHECK and yields NaN.
template <typename E>
__global__ void __launch_bounds__(kRowThreads) grpo_logp_rows(
    const E* __restrict__ logits, int64_t T, int V, const int32_t* __restrict__ targets,
    const float* __restrict__ ref_logp, float* __restrict__ logp_out, float* __restrict__ lse_out,
    float* __restrict__ kl_out, uint32_t* err) {
  using VT = Vec<E>;
  constexpr int NV = VT::N;
  __shared__ MS red[kRowThreads / 32 + 1];
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const E* zr = logits + row * (int64_t)V;
    const int h = (int)(((16 - (reinterpret_cast<uintptr_t>(zr) & 15)) & 15) / sizeof(E));
    const int head = h < V ? h : V;
    const int nvec = (V - head) / NV;
    const int tail0 = head + nvec * NV;
    const MS a = row_max_sumexp2<E>(zr, V, head, nvec, tail0, red);
    if (threadIdx.x == 0) {
      const float lse = (a.m + log2f(a.s)) * kLn2;
      const int32_t y = targets[row];
      float logp = NAN;
      if ((uint32_t)y < (uint32_t)V) {
        logp = VT::load1(zr + y) - lse;
      } else {
        ls_report(err, LS_DEVERR_CHECK);
      }
      logp_out[row] = logp;
      if (lse_out) lse_out[row] = lse;
      if (kl_out) {
        const float d = ref_logp[row] - logp;
        kl_out[row] = expm1f(d) - d;
      }
    }
    __syncthreads();  // red reuse in the next row
  }
}

// Fixed-order reduction of the per-token terms into this call's loss and stats, by
// kThreads threads (tid): lane-strided partials, a shuffle tree per warp, then warp 0
// over the warps' results (sh: [kThreads / 32] x 3 doubles, shf: [kThreads / 32] x 2
// floats of shared memory; sync(): a barrier of the kThreads threads).  The terms may
// come from other CTAs of the same grid: they are read past L1.
template <int kThreads, typename Sync>
__device__ void grpo_reduce(void* ws, int64_t T, int G, int mb, int me, int accumulate,
                            float* loss, float* stats, int tid, double* sh, float* shf,
                            Sync sync) {
  constexpr int kWarps = kThreads / 32;
  const WsLayout w = ws_layout(T, G);
  const double* inv = at<double>(ws, w.inv_norm);
  const int64_t* off = at<int64_t>(ws, w.off);
  const double* term = at<double>(ws, w.term);
  const float* rho = at<float>(ws, w.rho);
  const float* zeroed = at<float>(ws, w.zeroed);
  const int lane = tid & 31, wid = tid >> 5;
  double acc = 0.0, zc = 0.0, rs = 0.0;
  float mn = FLT_MAX, mx = -FLT_MAX;
  const int nm = me - mb;
  for (int m = 0; m < nm; ++m) {
    const double wgt = __ldcg(inv + mb + m) * (double)G;  // 1 / R_i
    const int64_t e = __ldcg(off + m + 1);
    for (int64_t t = __ldcg(off + m) + tid; t < e; t += kThreads) acc += __ldcg(term + t) * wgt;
  }
  for (int64_t t = tid; t < T; t += kThreads) {
    const float r = __ldcg(rho + t);
    zc += __ldcg(zeroed + t);
    rs += r;
    mn = fminf(mn, r);
    mx = fmaxf(mx, r);
  }
  acc = warp_sum(acc);
  zc = warp_sum(zc);
  rs = warp_sum(rs);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sh[wid * 3] = acc;
    sh[wid * 3 + 1] = zc;
    sh[wid * 3 + 2] = rs;
    shf[wid * 2] = mn;
    shf[wid * 2 + 1] = mx;
  }
  sync();
  if (wid == 0) {
    const bool h = lane < kWarps;
    acc = warp_sum(h ? sh[lane * 3] : 0.0);
    zc = warp_sum(h ? sh[lane * 3 + 1] : 0.0);
    rs = warp_sum(h ? sh[lane * 3 + 2] : 0.0);
    mn = h ? shf[lane * 2] : FLT_MAX;
    mx = h ? shf[lane * 2 + 1] : -FLT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      const float contrib = (float)(-acc / (double)G);
      loss[0] = accumulate ? loss[0] + contrib : contrib;
      if (stats) {
        stats[0] = (float)zc;
        stats[1] = (float)rs;
        stats[2] = T > 0 ? mn : 0.f;
        stats[3] = T > 0 ? mx : 0.f;
      }
    }
  }
}

// ---------------------------------------------------------------- streamed row kernel
// Each CTA streams its token rows through shared memory in chunks of two 16-byte vectors
// per consumer thread: a producer warp issues 1-D bulk copies into a ring of chunks (about 200 KB in flight per SM, so
// HBM sees deep queues without holding registers), the consumer warps reduce them, and
// a scalar warp fetches the next row's target, target logit, old (or
// reference) log-probability and member weights while the consumers work, so the end
// of a row waits on no global load.
//   loss form: pass 1 reduces the row to (max, sum exp2), keeping its last chunks (as
//              many as the ring holds) in shared memory; pass 2 writes dlogits of those
//              from shared memory and re-loads only the earlier chunks, most recently
//              read first (the likeliest to still be in L2), with streaming stores.
//   scoring form: pass 1 only, then logp / lse / KL.
// Rows must be 16-byte multiples (V * sizeof(E) % 16 == 0) for the bulk copies; other
// shapes use the one-CTA-per-row kernels above.
// Two shapes: the scoring form runs two CTAs per SM (16 consumer warps, 6 x 16 KB each);
// the loss form runs one CTA per SM (30 consumer warps, 6 x 30 KB), which keeps half as
// many rows live between a row's two passes, so more of pass 2 is served from L2.
template <bool kLoss>
struct StreamCfg {
  static constexpr int kWarps = kLoss ? 30 : 16;  // consumer warps
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kThreads = kConsumers + 64;  // + producer warp + scalar warp
  static constexpr uint32_t kChunkBytes = kConsumers * 32;  // two 16-byte vectors a thread
  static constexpr int kStages = kLoss ? 6 : 6;
  static constexpr int kCtasPerSm = kLoss ? 1 : 2;
  static_assert(kThreads <= 1024, "one CTA holds at most 1024 threads");
  static_assert(kStages * kChunkBytes <= 200 * 1024, "ring too large");
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}
template <int kCount>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kCount) : "memory");
}

// One thread's online (max, sum exp) over raw logits, for the streamed kernels: the max
// with three-operand max instructions, the exponent arguments x log2e - m log2e as one
// packed f32x2 FMA per pair and the sum in two lanes added with packed f32x2 adds.
struct OnlineMS {
  float m = -INFINITY;
  float2 s = {0.f, 0.f};
  template <int N>
  __device__ __forceinline__ void add(const float* x) {
    static_assert(N == 4 || N == 8, "a 16-byte vector of fp32 or bf16");
    float mx;
    if constexpr (N == 8)
      mx = fmax3(fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
    else
      mx = fmaxf(fmax3(x[0], x[1], x[2]), x[3]);
    if (mx > m) {
      const float r = fast_exp2((m - mx) * kLog2e);
      s.x *= r;
      s.y *= r;
      m = mx;
    }
    if (m == -INFINITY) return;  // only -inf logits so far: they add nothing
    const float2 l2 = make_float2(kLog2e, kLog2e);
    const float nm = -m * kLog2e;
    const float2 b = make_float2(nm, nm);
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), l2, b);
      s = __fadd2_rn(s, make_float2(fast_exp2(t.x), fast_exp2(t.y)));
    }
  }
  // the pair in the log2 domain of MS
  __device__ __forceinline__ MS log2_pair() const { return {m * kLog2e, s.x + s.y}; }
};

// dlogits of one 16-byte vector: x <- -c exp2(x log2e - lse2), plus c at lane tl when
// tl >= 0 (the target), with packed f32x2 FMA / multiply.
template <int N>
__device__ __forceinline__ void dlogit_vec(float* x, float c, float lse2, int tl) {
  const float2 l2 = make_float2(kLog2e, kLog2e);
  const float2 b = make_float2(-lse2, -lse2);
  const float2 nc = make_float2(-c, -c);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const float2 t = __ffma2_rn(make_float2(x[i], x[i + 1]), l2, b);
    const float2 g = __fmul2_rn(make_float2(fast_exp2(t.x), fast_exp2(t.y)), nc);
    x[i] = g.x;
    x[i + 1] = g.y;
  }
  if (tl >= 0) {
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (e == tl) x[e] += c;
  }
}

struct RowScalars {
  double adv, inv;  // member advantage and 1 / (G R_i) (loss form)
  float aux;        // old log-probability (loss form) or reference log-probability
  float zt;         // target logit
  int32_t y, pad;
};

struct StreamSmem {
  uint32_t full, empty, info_full, info_empty, red, bc, info, abort, fin, total;
};
__host__ __device__ constexpr StreamSmem stream_smem(int stages, uint32_t chunk_bytes, int warps) {
  StreamSmem l{};
  uint32_t p = (uint32_t)stages * chunk_bytes;
  l.full = p;        p += stages * 8;
  l.empty = p;       p += stages * 8;
  l.info_full = p;   p += 2 * 8;
  l.info_empty = p;  p += 2 * 8;
  l.red = p;         p += 2 * warps * 8;          // [row parity][warp] (max, sum)
  l.bc = p;          p += 16;                     // c, lse2, target of the current row
  l.info = p;        p += 2 * (uint32_t)sizeof(RowScalars);
  l.abort = p;       p += 16;                     // abort flag, last-CTA flag
  l.fin = p;         p += 32 * 3 * 8 + 32 * 2 * 4;  // grpo_reduce scratch
  l.total = p;
  return l;
}

struct StreamArgs {
  const void* logits;
  int64_t T;
  int V;
  const int32_t* targets;
  const float* aux;  // logp_old (loss form), ref_logp or null (scoring form)
  // loss form
  int G, mb, me;
  float eps;
  void* dlogits;
  void* ws;
  // both: per-row log-probability output (optional in the loss form)
  float* logp_out;
  // scoring form
  float* lse_out;
  float* kl_out;
  uint32_t* err;
  // loss form: the last CTA to finish reduces the terms into loss / stats
  int accumulate;
  float* loss;
  float* stats;
};

template <typename E, bool kLoss>
__global__ void __launch_bounds__(StreamCfg<kLoss>::kThreads, StreamCfg<kLoss>::kCtasPerSm)
    grpo_stream(const StreamArgs p) {
  using VT = Vec<E>;
  using Cfg = StreamCfg<kLoss>;
  constexpr int NV = VT::N;
  constexpr int kStages = Cfg::kStages;
  constexpr int kStreamWarps = Cfg::kWarps;
  constexpr int kCons = Cfg::kConsumers;
  constexpr uint32_t kChunkBytes = Cfg::kChunkBytes;
  constexpr uint32_t kChunkElems = kChunkBytes / sizeof(E);
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr StreamSmem L = stream_smem(kStages, kChunkBytes, kStreamWarps);
  const int64_t T = p.T;
  const int V = p.V;
  double* term_out = nullptr;
  float* rho_out = nullptr;
  float* zeroed_out = nullptr;
  const double* adv_ws = nullptr;
  const double* inv_ws = nullptr;
  const int64_t* off = nullptr;
  if constexpr (kLoss) {
    const WsLayout w = ws_layout(T, p.G);
    if (*at<int32_t>(p.ws, w.flag) == 0) return;  // the same for every CTA
    adv_ws = at<double>(p.ws, w.adv);
    inv_ws = at<double>(p.ws, w.inv_norm);
    off = at<int64_t>(p.ws, w.off);
    term_out = at<double>(p.ws, w.term);
    rho_out = at<float>(p.ws, w.rho);
    zeroed_out = at<float>(p.ws, w.zeroed);
  }
  const E* logits = static_cast<const E*>(p.logits);
  const uint32_t row_bytes = (uint32_t)V * sizeof(E);
  const int nch = (int)((row_bytes + kChunkBytes - 1) / kChunkBytes);
  constexpr int npass = kLoss ? 2 : 1;
  // loss form: the last `held` chunks of pass 1 stay in the ring for pass 2
  const int held = kLoss ? (nch < kStages ? nch : kStages) : 0;
  const uint32_t full0 = smem_u32(smem + L.full), empty0 = smem_u32(smem + L.empty);
  const uint32_t ifull0 = smem_u32(smem + L.info_full), iempty0 = smem_u32(smem + L.info_empty);
  MS* red = reinterpret_cast<MS*>(smem + L.red);
  float* bc = reinterpret_cast<float*>(smem + L.bc);
  RowScalars* info = reinterpret_cast<RowScalars*>(smem + L.info);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L.abort);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // a wait that gives up records the error and stops every later wait of the CTA
  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (*abort) return false;
    if (umma::mbar_wait(bar, parity)) return true;
    ls_report(p.err, LS_DEVERR_TIMEOUT);
    *abort = 1;
    return false;
  };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      umma::mbar_init(full0 + 8 * s, 1);
      umma::mbar_init(empty0 + 8 * s, kStreamWarps);
    }
    for (int s = 0; s < 2; ++s) {
      umma::mbar_init(ifull0 + 8 * s, 1);
      umma::mbar_init(iempty0 + 8 * s, 1);
    }
    *abort = 0;
    umma::fence_barrier_init();
  }
  __syncthreads();

  if (wid == kStreamWarps) {
    // ---- producer: the chunk sequence of every row (pass 1 forward, pass 2 reversed)
    if (lane == 0) {
      umma::RingPos<kStages> rp;
      int issued = 0;
      for (int64_t row = blockIdx.x; row < T && !*abort; row += gridDim.x) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(logits + row * (int64_t)V);
        for (int ps = 0; ps < npass; ++ps) {
          // pass 2 re-loads only the chunks that are no longer held in the ring
          const int n = ps == 0 ? nch : nch - held;
          for (int k = 0; k < n; ++k) {
            const int c = ps == 0 ? k : n - 1 - k;
            const uint32_t off_b = (uint32_t)c * kChunkBytes;
            const uint32_t bytes = row_bytes - off_b < kChunkBytes ? row_bytes - off_b : kChunkBytes;
            if (!wait(empty0 + 8 * rp.stage, rp.phase ^ 1u)) break;
            umma::mbar_expect_tx(full0 + 8 * rp.stage, bytes);
            bulk_load(smem_u32(smem + rp.stage * kChunkBytes), src + off_b, bytes,
                      full0 + 8 * rp.stage);
            ++issued;
            rp.advance();
          }
        }
      }
      // no copy may still be landing when the CTA exits: wait for the last fill of each
      // stage (already complete unless a wait above gave up)
      for (int s = 0; s < kStages && s < issued; ++s) {
        rp.stage = rp.stage == 0 ? kStages - 1 : rp.stage - 1;
        if (rp.stage == kStages - 1) rp.phase ^= 1u;
        umma::mbar_wait(full0 + 8 * rp.stage, rp.phase);
      }
    }
    return;
  }
  if (wid == kStreamWarps + 1) {
    // ---- scalar warp: per-row scalars one row ahead of the consumers
    if (lane == 0) {
      int q = 0;
      for (int64_t row = blockIdx.x; row < T; row += gridDim.x, ++q) {
        const int b = q & 1;
        if (!wait(iempty0 + 8 * b, (((uint32_t)q >> 1) & 1u) ^ 1u)) break;
        RowScalars r;
        r.y = p.targets[row];
        r.zt = (uint32_t)r.y < (uint32_t)V ? VT::load1(logits + row * (int64_t)V + r.y) : 0.f;
        r.aux = p.aux ? p.aux[row] : 0.f;
        r.adv = 0.0;
        r.inv = 0.0;
        if constexpr (kLoss) {
          int lo_m = 0, hi_m = p.me - p.mb - 1;  // member of this token
          while (lo_m < hi_m) {
            const int mid = (lo_m + hi_m + 1) >> 1;
            if (off[mid] <= row) lo_m = mid; else hi_m = mid - 1;
          }
          r.adv = adv_ws[p.mb + lo_m];
          r.inv = inv_ws[p.mb + lo_m];
        }
        info[b] = r;
        umma::mbar_arrive(ifull0 + 8 * b);
      }
    }
    return;
  }

  // ---- consumers
  umma::RingPos<kStages> rp;
  int q = 0;
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x, ++q) {
    OnlineMS oms;
    const uint32_t s0 = rp.stage;  // stage of chunk 0; chunk k sits in (s0 + k) % kStages
    for (int k = 0; k < nch; ++k) {
      const uint32_t bytes =
          row_bytes - k * kChunkBytes < kChunkBytes ? row_bytes - k * kChunkBytes : kChunkBytes;
      const int nvec = (int)(bytes / 16);
      if (wait(full0 + 8 * rp.stage, rp.phase)) {
        const uint4* sv = reinterpret_cast<const uint4*>(smem + rp.stage * kChunkBytes);
        for (int i = tid; i < nvec; i += kCons) {
          float x[NV];
          VT::unpack(sv[i], x);
          oms.add<NV>(x);
        }
      }
      __syncwarp();
      if (lane == 0 && k < nch - held) umma::mbar_arrive(empty0 + 8 * rp.stage);
      rp.advance();
    }
    MS ms = oms.log2_pair();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      MS other = {__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.s, o)};
      ms = ms_merge(ms, other);
    }
    MS* rq = red + (q & 1) * kStreamWarps;
    if (lane == 0) rq[wid] = ms;
    consumers_sync<kCons>();
    if (wid == 0) {
      MS a = lane < kStreamWarps ? rq[lane] : MS{-INFINITY, 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        MS other = {__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o)};
        a = ms_merge(a, other);
      }
      if (lane == 0) {
        const int b = q & 1;
        const float lse2 = a.m + log2f(a.s);
        wait(ifull0 + 8 * b, ((uint32_t)q >> 1) & 1u);
        const RowScalars r = info[b];
        umma::mbar_arrive(iempty0 + 8 * b);
        const bool valid = (uint32_t)r.y < (uint32_t)V;
        if (!valid) ls_report(p.err, LS_DEVERR_CHECK);
        const float logp = valid ? r.zt - lse2 * kLn2 : NAN;
        if constexpr (kLoss) {
          float c = 0.f;
          double term = 0.0;
          float rho = 0.f, zeroed = 0.f;
          if (valid) {
            rho = expf(logp - r.aux);
            const float A = (float)r.adv;
            const float clipped = fminf(fmaxf(rho, 1.f - p.eps), 1.f + p.eps);
            const bool active = rho * A <= clipped * A;  // ties: the unclipped branch
            term = (double)(active ? rho : clipped) * r.adv;
            c = active ? (float)(-r.adv * (double)rho * r.inv) : 0.f;
            zeroed = (!active && A != 0.f) ? 1.f : 0.f;
          }
          term_out[row] = term;
          rho_out[row] = rho;
          zeroed_out[row] = zeroed;
          if (p.logp_out) p.logp_out[row] = logp;
          bc[0] = c;
          bc[1] = lse2;
          bc[2] = __int_as_float(r.y);
        } else {
          p.logp_out[row] = logp;
          if (p.lse_out) p.lse_out[row] = lse2 * kLn2;
          if (p.kl_out) {
            const float d = r.aux - logp;
            p.kl_out[row] = expm1f(d) - d;
          }
        }
      }
    }
    if constexpr (kLoss) {
      consumers_sync<kCons>();
      const float c = bc[0], lse2 = bc[1];
      const int y = __float_as_int(bc[2]);
      E* gr = static_cast<E*>(p.dlogits) + row * (int64_t)V;
      // dlogits of chunk ch from ring stage st (whose fill has landed), then release it
      auto p2_chunk = [&](uint32_t st, int ch, bool ok) {
        const uint32_t off_b = (uint32_t)ch * kChunkBytes;
        const uint32_t bytes = row_bytes - off_b < kChunkBytes ? row_bytes - off_b : kChunkBytes;
        const int nvec = (int)(bytes / 16);
        uint4* gv = reinterpret_cast<uint4*>(gr + (size_t)ch * kChunkElems);
        if (c == 0.f) {
          const uint4 zero = make_uint4(0, 0, 0, 0);
          for (int i = tid; i < nvec; i += kCons) __stcs(gv + i, zero);
        } else if (ok) {
          const uint4* sv = reinterpret_cast<const uint4*>(smem + st * kChunkBytes);
          const int ty = y - ch * (int)kChunkElems;  // target's element within the chunk
          for (int i = tid; i < nvec; i += kCons) {
            float x[NV];
            VT::unpack(sv[i], x);
            dlogit_vec<NV>(x, c, lse2, ty >= i * NV && ty < i * NV + NV ? ty - i * NV : -1);
            __stcs(gv + i, VT::pack(x));
          }
        }
        __syncwarp();
        if (lane == 0) umma::mbar_arrive(empty0 + 8 * st);
      };
      // the held chunks first, oldest first (the producer refills their stages in that
      // order), then the re-loaded ones, most recently read first (likeliest in L2)
      for (int j = 0; j < held; ++j) {
        const int ch = nch - held + j;
        p2_chunk((s0 + (uint32_t)ch) % kStages, ch, true);
      }
      for (int k = 0; k < nch - held; ++k) {
        const bool ok = wait(full0 + 8 * rp.stage, rp.phase);
        p2_chunk(rp.stage, nch - held - 1 - k, ok);
        rp.advance();
      }
    }
  }
  if constexpr (kLoss) {
    // The last CTA to finish reduces every row's term into the loss (the ticket was
    // zeroed by the prep launch).  Thread 0 wrote this CTA's terms; the fence orders
    // them before its ticket.
    volatile int* last = abort + 1;
    if (tid == 0) {
      __threadfence();
      const uint32_t t = atomicAdd(at<uint32_t>(p.ws, ws_layout(T, p.G).flag + 4), 1u);
      *last = t == gridDim.x - 1;
    }
    consumers_sync<kCons>();
    if (*last) {
      __threadfence();
      grpo_reduce<kCons>(p.ws, T, p.G, p.mb, p.me, p.accumulate, p.loss, p.stats, tid,
                         reinterpret_cast<double*>(smem + L.fin),
                         reinterpret_cast<float*>(smem + L.fin + 32 * 3 * 8),
                         [] { consumers_sync<kCons>(); });
    }
  }
}

// The reduction as its own launch (T = 0, or the one-CTA-per-row kernel).
__global__ void __launch_bounds__(1024) grpo_final(int64_t T, int G, int mb, int me,
                                                   int accumulate, float* loss, float* stats,
                                                   void* ws) {
  const WsLayout w = ws_layout(T, G);
  if (*at<int32_t>(ws, w.flag) == 0) return;
  __shared__ double sh[32 * 3];
  __shared__ float shf[32 * 2];
  grpo_reduce<1024>(ws, T, G, mb, me, accumulate, loss, stats, threadIdx.x, sh, shf,
                    [] { __syncthreads(); });
}

}  // namespace

size_t ls_grpo_ws_bytes(int64_t T, int G) { return ws_layout(T, G).total; }

namespace {
// The streamed kernels apply when rows are whole 16-byte multiples (the bulk copies'
// granularity; the entry points have already checked the buffers' alignment, re-checked
// here).  Returns false (nothing launched) otherwise; *e is the launch status when it
// returns true.
template <bool kLoss>
bool launch_stream(const StreamArgs& sa, bool is_bf16, int num_sms, cudaStream_t st,
                   cudaError_t* e) {
  const int esz = is_bf16 ? 2 : 4;
  if (((int64_t)sa.V * esz) % 16 != 0 || (reinterpret_cast<uintptr_t>(sa.logits) & 15) ||
      (kLoss && (reinterpret_cast<uintptr_t>(sa.dlogits) & 15)))
    return false;
  using Cfg = StreamCfg<kLoss>;
  constexpr uint32_t smem = stream_smem(Cfg::kStages, Cfg::kChunkBytes, Cfg::kWarps).total;
  const void* fn = is_bf16 ? (const void*)grpo_stream<__nv_bfloat16, kLoss>
                           : (const void*)grpo_stream<float, kLoss>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int64_t ctas = (int64_t)num_sms * Cfg::kCtasPerSm;
  const int64_t grid = sa.T < ctas ? sa.T : ctas;
  if (is_bf16)
    grpo_stream<__nv_bfloat16, kLoss><<<(unsigned)grid, Cfg::kThreads, smem, st>>>(sa);
  else
    grpo_stream<float, kLoss><<<(unsigned)grid, Cfg::kThreads, smem, st>>>(sa);
  ls_note_launch();
  *e = cudaGetLastError();
  return true;
}

StreamArgs loss_stream_args(const LsGrpoArgs& a) {
  StreamArgs sa{};
  sa.logits = a.logits;
  sa.T = a.T;
  sa.V = a.V;
  sa.targets = a.targets;
  sa.aux = a.logp_old;
  sa.G = a.G;
  sa.mb = a.member_begin;
  sa.me = a.member_end;
  sa.eps = a.eps;
  sa.dlogits = a.dlogits;
  sa.ws = a.workspace;
  sa.logp_out = a.logp_out;
  sa.err = a.err;
  sa.accumulate = a.accumulate_loss;
  sa.loss = a.loss;
  sa.stats = a.stats;
  return sa;
}
}  // namespace

cudaError_t ls_launch_grpo(const LsGrpoArgs& a, int num_sms, cudaStream_t st) {
  grpo_prep<<<1, 32, 0, st>>>(a.rewards, a.resp_lens, a.G, a.member_begin, a.member_end,
                              a.std_ddof, a.adv_eps, a.T, a.workspace, a.err);
  ls_note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.T > 0 && launch_stream<true>(loss_stream_args(a), a.is_bf16, num_sms, st, &e)) {
    return e;  // the streamed kernel's last CTA has reduced the loss
  } else if (a.T > 0) {
    int64_t grid = (int64_t)num_sms * 2;
    if (grid > a.T) grid = a.T;
    if (a.is_bf16) {
      grpo_rows<__nv_bfloat16><<<(unsigned)grid, kRowThreads, 0, st>>>(
          static_cast<const __nv_bfloat16*>(a.logits), a.T, a.V, a.targets, a.logp_old, a.G,
          a.member_begin, a.member_end, a.eps, static_cast<__nv_bfloat16*>(a.dlogits),
          a.logp_out, a.workspace, a.err);
  ls_note_launch();
    } else {
      grpo_rows<float><<<(unsigned)grid, kRowThreads, 0, st>>>(
          static_cast<const float*>(a.logits), a.T, a.V, a.targets, a.logp_old, a.G,
          a.member_begin, a.member_end, a.eps, static_cast<float*>(a.dlogits), a.logp_out,
          a.workspace, a.err);
  ls_note_launch();
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  grpo_final<<<1, 1024, 0, st>>>(a.T, a.G, a.member_begin, a.member_end, a.accumulate_loss,
                                 a.loss, a.stats, a.workspace);
  ls_note_launch();
  return cudaGetLastError();
}

cudaError_t ls_launch_grpo_logp(const void* logits, bool is_bf16, int64_t T, int V,
                                const int32_t* targets, const float* ref_logp, float* logp_out,
                                float* lse_out, float* kl_out, uint32_t* err, int num_sms,
                                cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  StreamArgs sa{};
  sa.logits = logits;
  sa.T = T;
  sa.V = V;
  sa.targets = targets;
  sa.aux = ref_logp;
  sa.logp_out = logp_out;
  sa.lse_out = lse_out;
  sa.kl_out = kl_out;
  sa.err = err;
  cudaError_t e = cudaSuccess;
  if (launch_stream<false>(sa, is_bf16, num_sms, st, &e)) return e;
  int64_t grid = (int64_t)num_sms * 2;
  if (grid > T) grid = T;
  if (is_bf16) {
    grpo_logp_rows<__nv_bfloat16><<<(unsigned)grid, kRowThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(logits), T, V, targets, ref_logp, logp_out, lse_out,
        kl_out, err);
  } else {
    grpo_logp_rows<float><<<(unsigned)grid, kRowThreads, 0, st>>>(
        static_cast<const float*>(logits), T, V, targets, ref_logp, logp_out, lse_out, kl_out,
        err);
  }
  ls_note_launch();
  return cudaGetLastError();
}
