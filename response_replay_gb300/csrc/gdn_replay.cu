// gdn_replay.cu -- Gated-DeltaNet replay from a captured recurrent state.
//
// For the hybrid model's Gated-DeltaNet layers LongStraw keeps only the compact
// recurrent state at the end of the prompt (digest, "Method" step 1 and "Qwen
// implementation"; explainer, "Two incompatible architectures", Qwen bullet) and replays
// each response from it with that state stopgrad.  The layer is the gated delta rule
// (Yang, Kautz & Hatamizadeh, "Gated Delta Networks", ICLR 2025), per head:
//   S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t (scale q_t)
// with S a 128 x 128 (d_v x d_k) fp32 matrix and S_0 the captured state.
//
// Chunked form (64-token chunks; within a chunk G_t is the running sum of g, gamma_t =
// exp(G_t), Gam[t][i] = exp(G_t - G_i) for i <= t, lam_i = gamma_C / gamma_i):
//   Ms = (K K^T) * Gam strictly lower,  T = (I + diag(beta) Ms)^-1
//   W  = T diag(beta gamma) K,  U0 = T diag(beta) V,  U = U0 - W S0^T
//   O  = diag(gamma) Q' S0^T + ((Q' K^T) * Gam, lower incl.) U,   Q' = scale Q
//   S_C = gamma_C S0 + U^T diag(lam) K
// Every step that does not depend on the state runs for all (head, chunk) pairs at once
// as batched matrix products; only the state hand-off between chunks is sequential, and
// it splits by rows of S (row i of S_{c+1} needs only row i of S_c), so it runs as one
// warp per (head, row).  The backward is the adjoint of the same steps: the gradient of
// the state is carried from chunk to chunk in reverse (again row by row), the rest is
// batched per chunk.  The gradient reaching S_0 is dropped: the captured state is
// stopgrad.
//
// Arithmetic is fp32 on the CUDA cores (the chunk matrices are 64 x 64 to 128 x 128 and
// the triangular solve is sequential within a column); inputs q, k, v, dO are bf16.
#include <math.h>

#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_umma.cuh"

namespace {

constexpr int kD = 128;   // head dims (d_k = d_v)
constexpr int kC = 64;    // chunk length
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- workspace layout
// Per (head, chunk) pair b = h * nC + c, fp32 blocks of the sizes below.
struct GdnLayout {
  int nC, nb;
  size_t qf, kf, vf, dof;            // [nb][64][128]
  size_t x1, x2, x3, x4, x5, x6;     // [nb][64][128] scratch
  size_t w, u;                       // [nb][64][128]
  size_t ms, tm, p, m1, m2;          // [nb][64][64]
  size_t sc, dsc;                    // [nb][128][128]
  size_t gcum, gam, lam, beta;       // [nb][64]
  size_t total;
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

GdnLayout gdn_layout(int R, int H, bool bwd) {
  GdnLayout L;
  L.nC = (R + kC - 1) / kC;
  L.nb = L.nC * H;
  const size_t cd = (size_t)L.nb * kC * kD * 4, cc = (size_t)L.nb * kC * kC * 4;
  const size_t dd = (size_t)L.nb * kD * kD * 4, c1 = (size_t)L.nb * kC * 4;
  size_t p = 0;
  auto take = [&](size_t n) { const size_t o = p; p = al256(p + n); return o; };
  L.qf = take(cd); L.kf = take(cd); L.vf = take(cd);
  L.dof = bwd ? take(cd) : 0;
  L.x1 = take(cd); L.x2 = take(cd);
  L.x3 = bwd ? take(cd) : 0; L.x4 = bwd ? take(cd) : 0;
  L.x5 = bwd ? take(cd) : 0; L.x6 = bwd ? take(cd) : 0;
  L.w = take(cd); L.u = take(cd);
  L.ms = take(cc); L.tm = take(cc); L.p = take(cc);
  L.m1 = bwd ? take(cc) : 0; L.m2 = bwd ? take(cc) : 0;
  L.sc = take(dd);
  L.dsc = bwd ? take(dd) : 0;
  L.gcum = take(c1); L.gam = take(c1); L.lam = take(c1); L.beta = take(c1);
  L.total = p;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------- chunk inputs
// Grid (nC, H), 128 threads (one per head dim).  Chunk c of head h: qf = scale q, kf, vf
// (and dof when d_o is given) as fp32 [64][128], zeros past R; per token the running log
// decay G, gamma = exp(G), lam = gamma_C / gamma and beta (g = beta = 0 past R, so padding
// neither decays nor writes the state).
__global__ void __launch_bounds__(128) gdn_load(const __nv_bfloat16* __restrict__ q,
                                                const __nv_bfloat16* __restrict__ k,
                                                const __nv_bfloat16* __restrict__ v,
                                                const __nv_bfloat16* __restrict__ d_o,
                                                const float* __restrict__ g,
                                                const float* __restrict__ beta, int R, int H,
                                                float scale, float* qf, float* kf, float* vf,
                                                float* dof, float* gcum, float* gam, float* lam,
                                                float* bet) {
  const int c = blockIdx.x, h = blockIdx.y, nC = gridDim.x, j = threadIdx.x;
  const int64_t b = (int64_t)h * nC + c;
  for (int t = 0; t < kC; ++t) {
    const int tok = c * kC + t;
    const bool ok = tok < R;
    const int64_t src = ((int64_t)tok * H + h) * kD + j;
    const int64_t dst = (b * kC + t) * kD + j;
    qf[dst] = ok ? scale * bf2f(q[src]) : 0.f;
    kf[dst] = ok ? bf2f(k[src]) : 0.f;
    vf[dst] = ok ? bf2f(v[src]) : 0.f;
    if (dof) dof[dst] = ok ? bf2f(d_o[src]) : 0.f;
  }
  __shared__ float gs[kC];
  if (j < kC) {
    const int tok = c * kC + j;
    gs[j] = tok < R ? g[(int64_t)tok * H + h] : 0.f;
    bet[b * kC + j] = tok < R ? beta[(int64_t)tok * H + h] : 0.f;
  }
  __syncthreads();
  if (j == 0) {  // running sum in token order
    float s = 0.f;
    for (int t = 0; t < kC; ++t) {
      s += gs[t];
      gs[t] = s;
    }
  }
  __syncthreads();
  if (j < kC) {
    const float G = gs[j], GC = gs[kC - 1];
    gcum[b * kC + j] = G;
    gam[b * kC + j] = exp2f(G * kLog2e);
    lam[b * kC + j] = exp2f((GC - G) * kLog2e);
  }
}

// ---------------------------------------------------------------- batched products
// C[b] = alpha diag(rs[b]) op(A[b]) op(B[b]) (+ C[b]), op(X) = X or X^T, masked to the
// lower triangle (mask 1: row >= col, 2: row > col; 0: none).  Row-major, leading
// dimensions lda / ldb / ldc, batch strides sA / sB / sC (elements); rs may be NULL.
// 64 x 64 output tiles, 64 threads with 8 x 8 outputs each (rows 8 ty .., columns 8 tx ..),
// K in slabs of 16 (M, N multiples of 64, K of 16: the chunk shapes 64 and 128); four
// 16-byte shared-memory loads feed 64 FMAs.
template <bool TA, bool TB>
__global__ void __launch_bounds__(64) gdn_gemm(const float* __restrict__ A, int lda, int64_t sA,
                                               const float* __restrict__ B, int ldb, int64_t sB,
                                               float* C, int ldc, int64_t sC, int K, float alpha,
                                               const float* __restrict__ rs, int64_t srs,
                                               int accumulate, int mask) {
  __shared__ __align__(16) float As[16][64 + 4];
  __shared__ __align__(16) float Bs[16][64 + 4];
  const int tid = threadIdx.x, tx = tid & 7, ty = tid >> 3;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  const int64_t bz = blockIdx.z;
  A += bz * sA;
  B += bz * sB;
  C += bz * sC;
  if (mask && n0 > m0 + 63) {  // tile entirely above the diagonal
    if (!accumulate)
      for (int e = tid; e < 64 * 64; e += 64) C[(int64_t)(m0 + e / 64) * ldc + n0 + e % 64] = 0.f;
    return;
  }
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  // The next slab is loaded into registers while the current one is multiplied.
  float av[16], bv[16];
  auto load_slab = [&](int k0) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int e = tid + 64 * r;  // 1024 elements of each 64 x 16 / 16 x 64 tile
      if (TA) {  // op(A)[m][k] = A[k][m]: read along m
        av[r] = A[(int64_t)(k0 + e / 64) * lda + m0 + e % 64];
      } else {
        av[r] = A[(int64_t)(m0 + e / 16) * lda + k0 + e % 16];
      }
      if (TB) {  // op(B)[k][n] = B[n][k]
        bv[r] = B[(int64_t)(n0 + e / 16) * ldb + k0 + e % 16];
      } else {
        bv[r] = B[(int64_t)(k0 + e / 64) * ldb + n0 + e % 64];
      }
    }
  };
  load_slab(0);
  for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int e = tid + 64 * r;
      if (TA) As[e / 64][e % 64] = av[r]; else As[e % 16][e / 16] = av[r];
      if (TB) Bs[e % 16][e / 16] = bv[r]; else Bs[e / 64][e % 64] = bv[r];
    }
    __syncthreads();
    if (k0 + 16 < K) load_slab(k0 + 16);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][8 * ty]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][8 * ty + 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][8 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][8 * tx + 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + 8 * ty + i;
    const float sc = alpha * (rs ? rs[bz * srs + m] : 1.f);
#pragma unroll
    for (int j4 = 0; j4 < 2; ++j4) {
      const int n = n0 + 8 * tx + 4 * j4;
      float x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[j] = sc * acc[i][4 * j4 + j];
        if ((mask == 1 && n + j > m) || (mask == 2 && n + j >= m)) x[j] = 0.f;
      }
      float4* p = reinterpret_cast<float4*>(C + (int64_t)m * ldc + n);
      float4 v = make_float4(x[0], x[1], x[2], x[3]);
      if (accumulate) {
        const float4 o = *p;
        v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
      }
      *p = v;
    }
  }
}

// ---------------------------------------------------------------- elementwise steps
// X[b][t][i] *= exp(G_t - G_i) (and beta_t when rowb), on the lower triangle (strict when
// strict), zero above.  Grid nb, 256 threads.
__global__ void __launch_bounds__(256) gdn_decay(float* X, const float* __restrict__ gcum,
                                                 const float* __restrict__ rowb, int strict,
                                                 float* copy_to) {
  const int64_t b = blockIdx.x;
  const float* G = gcum + b * kC;
  for (int e = threadIdx.x; e < kC * kC; e += blockDim.x) {
    const int t = e / kC, i = e % kC;
    float* x = X + b * kC * kC + e;
    float y = 0.f;
    if (i < t || (!strict && i == t)) y = *x * exp2f((G[t] - G[i]) * kLog2e);
    if (copy_to) copy_to[b * kC * kC + e] = y;
    if (rowb) y *= rowb[b * kC + t];
    *x = y;
  }
}

// Y[b][t][:] = a * s1[b][t] * X1[b][t][:] + c * X2[b][t][:]  (X2 may be NULL); grid nb
// (a chunk per CTA), 256 threads.
__global__ void __launch_bounds__(256) gdn_rows(float* Y, const float* X1, const float* s1,
                                                const float* s2, float a, const float* X2,
                                                float c) {
  const int64_t b = blockIdx.x;
#pragma unroll
  for (int q = 0; q < kC * kD / 4 / 256; ++q) {  // the chunk's 64 rows as float4
    const int e4 = threadIdx.x + 256 * q, t = e4 / (kD / 4);
    const float sc = a * (s1 ? s1[b * kC + t] : 1.f) * (s2 ? s2[b * kC + t] : 1.f);
    const int64_t e = b * kC * kD / 4 + e4;
    float4 y = reinterpret_cast<const float4*>(X1)[e];
    y.x *= sc; y.y *= sc; y.z *= sc; y.w *= sc;
    if (X2) {
      const float4 x2 = reinterpret_cast<const float4*>(X2)[e];
      y.x += c * x2.x; y.y += c * x2.y; y.z += c * x2.z; y.w += c * x2.w;
    }
    reinterpret_cast<float4*>(Y)[e] = y;
  }
}

// T = (I + A)^-1 for the unit lower-triangular I + A of each chunk (A strictly lower):
// column j of T is the forward substitution T[t][j] = [t == j] - sum_{j <= i < t} A[t][i]
// T[i][j], independent of the other columns.  Grid nb, 64 threads (one per column).
__global__ void __launch_bounds__(64) gdn_tri_inv(const float* __restrict__ A, float* Tm) {
  __shared__ float As[kC][kC + 1];
  const int64_t b = blockIdx.x;
  const int j = threadIdx.x;
  for (int e = j; e < kC * kC; e += kC) As[e / kC][e % kC] = A[b * kC * kC + e];
  __syncthreads();
  float col[kC];
#pragma unroll
  for (int t = 0; t < kC; ++t) {
    float s = t == j ? 1.f : 0.f;
#pragma unroll
    for (int i = 0; i < t; ++i) s = fmaf(-As[t][i], col[i], s);
    col[t] = t >= j ? s : 0.f;
  }
#pragma unroll
  for (int t = 0; t < kC; ++t) Tm[b * kC * kC + t * kC + j] = col[t];
}

// p[0..63] per lane -> lane l holds the warp sums of entries 2l and 2l + 1 in p[0], p[1].
__device__ __forceinline__ void warp_reduce64(float* p, int lane) {
#pragma unroll
  for (int off = 16, n = 64; off >= 1; off >>= 1, n >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < n / 2; ++j) {
      const float send = up ? p[j] : p[j + n / 2];
      const float keep = up ? p[j + n / 2] : p[j];
      p[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}

// ---------------------------------------------------------------- state hand-off
// Forward: rows of the state, chunk by chunk.  A CTA owns 32 rows of one head's state
// (grid (H, 4), 4 warps of 8 rows; lane l holds columns 4l .. 4l+3 of each row):
//   Sc[b][i][:] = S[i][:]                        (state entering chunk c)
//   u_t = U0[t][i] - W[t] . S[i]                 (written over U0; lane l: t = 2l, 2l+1)
//   S[i] <- gamma_C S[i] + sum_t lam_t u_t K[t]
// Each chunk's W^T and K (32 KB each) arrive by bulk copy into a two-stage ring, one
// chunk ahead, and every value read from shared memory serves the warp's 8 rows: with
// one row per warp the shared-memory pipe was saturated (1.05 ms at R = 4,096, H = 32).
constexpr int kScanCtaRows = 32, kScanWarpRows = 8, kScanWarps = 4;
constexpr int kScanVStride = kScanCtaRows + 4;          // v rows: spread the lanes' stores
constexpr uint32_t kScanChunkBytes = kC * kD * 4;       // one of W^T, K
constexpr size_t kScanFwdSmem = 4 * (size_t)kScanChunkBytes +
                                (size_t)(kScanCtaRows * kD + kC * kScanVStride) * 4 + 64;
__global__ void __launch_bounds__(32 * kScanWarps) gdn_scan_fwd(const float* __restrict__ state0,
                                                                int nC, const float* __restrict__ Wtg,
                                                                const float* __restrict__ kf,
                                                                float* U, const float* __restrict__ gam,
                                                                const float* __restrict__ lam,
                                                                float* Sc, float* state_out,
                                                                uint32_t* err) {
  extern __shared__ __align__(128) uint8_t smraw[];
  float* ring = reinterpret_cast<float*>(smraw);         // stage s: W^T [128][64], K [64][128]
  float* Ssm = ring + 4 * kC * kD;                       // [32][128]: rows entering the chunk
  float* Vsm = Ssm + kScanCtaRows * kD;                  // [64][kScanVStride]: lam_t u_t
  const uint32_t full0 = smem_u32(Vsm + kC * kScanVStride), empty0 = full0 + 16;
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp * kScanWarpRows;                   // the warp's rows: i0 + wr + r
  const int i0 = blockIdx.y * kScanCtaRows;
  if (threadIdx.x == 0) {
    for (int st = 0; st < 2; ++st) {
      umma::mbar_init(full0 + 8 * st, 1);
      umma::mbar_init(empty0 + 8 * st, kScanWarps);
    }
    umma::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int c) {  // chunk c into stage c & 1 (one thread)
    const int st = c & 1;
    const int64_t b = (int64_t)h * nC + c;
    umma::mbar_expect_tx(full0 + 8 * st, 2 * kScanChunkBytes);
    umma::bulk_load(smem_u32(ring + st * 2 * kC * kD), Wtg + b * kC * kD, kScanChunkBytes, full0 + 8 * st);
    umma::bulk_load(smem_u32(ring + st * 2 * kC * kD + kC * kD), kf + b * kC * kD, kScanChunkBytes,
                    full0 + 8 * st);
  };
  int issued = 0;
  if (threadIdx.x == 0 && nC > 0) {
    issue(0);
    issued = 1;
  }
  float S[kScanWarpRows][4];
#pragma unroll
  for (int r = 0; r < kScanWarpRows; ++r) {
    const float4 v = *reinterpret_cast<const float4*>(state0 + ((int64_t)h * kD + i0 + wr + r) * kD + 4 * lane);
    S[r][0] = v.x; S[r][1] = v.y; S[r][2] = v.z; S[r][3] = v.w;
  }
  bool ok = true;
  for (int c = 0; c < nC; ++c) {
    const int64_t b = (int64_t)h * nC + c;
    const int st = c & 1;
    // the next chunk's copies (warp 0; its stage was last read in chunk c - 1)
    if (warp == 0 && c + 1 < nC) {
      ok = c == 0 || umma::mbar_wait(empty0 + 8 * ((c + 1) & 1), ((c - 1) >> 1) & 1);
      if (ok && lane == 0) {
        issue(c + 1);
        issued = c + 2;
      }
    }
    // this chunk's U0 and lam, independent of the state: in flight before the waits
    float u0[kScanWarpRows][2], lm[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = 2 * lane + q;
      lm[q] = lam[b * kC + t];
#pragma unroll
      for (int r = 0; r < kScanWarpRows; ++r) u0[r][q] = U[(b * kC + t) * kD + i0 + wr + r];
    }
    const float gC = gam[b * kC + kC - 1];
    // the state entering the chunk: to Sc, and this warp's rows to shared memory
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r) {
      const float4 v = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
      *reinterpret_cast<float4*>(Sc + (b * kD + i0 + wr + r) * kD + 4 * lane) = v;
      *reinterpret_cast<float4*>(Ssm + (wr + r) * kD + 4 * lane) = v;
    }
    __syncwarp();
    if (!ok || !umma::mbar_wait(full0 + 8 * st, (c >> 1) & 1)) {
      ls_report(err, LS_DEVERR_TIMEOUT);
      ok = false;
      break;
    }
    const float* Wt = ring + st * 2 * kC * kD;
    const float* Ks = Wt + kC * kD;
    // W[t] . S[i] for t = 2 lane, 2 lane + 1
    float acc[kScanWarpRows][2];
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r) acc[r][0] = acc[r][1] = 0.f;
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
      float2 w[4];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) w[kk] = *reinterpret_cast<const float2*>(Wt + (k + kk) * kC + 2 * lane);
#pragma unroll
      for (int r = 0; r < kScanWarpRows; ++r) {
        const float4 sv = *reinterpret_cast<const float4*>(Ssm + (wr + r) * kD + k);
        acc[r][0] = fmaf(w[0].x, sv.x, fmaf(w[1].x, sv.y, fmaf(w[2].x, sv.z, fmaf(w[3].x, sv.w, acc[r][0]))));
        acc[r][1] = fmaf(w[0].y, sv.x, fmaf(w[1].y, sv.y, fmaf(w[2].y, sv.z, fmaf(w[3].y, sv.w, acc[r][1]))));
      }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int t = 2 * lane + q;
      float vr[kScanWarpRows];
#pragma unroll
      for (int r = 0; r < kScanWarpRows; ++r) {
        const float u = u0[r][q] - acc[r][q];
        U[(b * kC + t) * kD + i0 + wr + r] = u;
        vr[r] = lm[q] * u;
      }
      *reinterpret_cast<float4*>(Vsm + t * kScanVStride + wr) = make_float4(vr[0], vr[1], vr[2], vr[3]);
      *reinterpret_cast<float4*>(Vsm + t * kScanVStride + wr + 4) = make_float4(vr[4], vr[5], vr[6], vr[7]);
    }
    __syncwarp();
    // S[i] <- gamma_C S[i] + sum_t v_t K[t]
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) S[r][q] *= gC;
#pragma unroll 4
    for (int t = 0; t < kC; ++t) {
      const float4 kv = *reinterpret_cast<const float4*>(Ks + t * kD + 4 * lane);
      const float4 va = *reinterpret_cast<const float4*>(Vsm + t * kScanVStride + wr);
      const float4 vb = *reinterpret_cast<const float4*>(Vsm + t * kScanVStride + wr + 4);
      const float vv[kScanWarpRows] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
      for (int r = 0; r < kScanWarpRows; ++r) {
        S[r][0] = fmaf(vv[r], kv.x, S[r][0]);
        S[r][1] = fmaf(vv[r], kv.y, S[r][1]);
        S[r][2] = fmaf(vv[r], kv.z, S[r][2]);
        S[r][3] = fmaf(vv[r], kv.w, S[r][3]);
      }
    }
    __syncwarp();
    if (lane == 0) umma::mbar_arrive(empty0 + 8 * st);  // this warp is done with the stage
  }
  if (ok && state_out)
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r)
      *reinterpret_cast<float4*>(state_out + ((int64_t)h * kD + i0 + wr + r) * kD + 4 * lane) =
          make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
  // do not leave while a copy into this CTA's shared memory may be in flight
  if (threadIdx.x == 0)
    for (int c = issued - 2 > 0 ? issued - 2 : 0; c < issued; ++c)
      umma::mbar_wait(full0 + 8 * (c & 1), (c >> 1) & 1);
}

// Backward: rows of dS (the gradient of the state leaving the chunk), chunks in reverse:
//   dSC[b][i][:] = dS[i]
//   a_t = K[t] . dS[i];  dZ_t = dZ0[t][i] + sum_{s >= t} T[s][t] lam_s a_s;  dY_t = beta_t dZ_t
//   dS[i] <- gamma_C dS[i] + sum_t gamma_t (dO[t][i] Q'[t] - dY_t K[t])
// A CTA owns 32 rows of one head's dS (grid (H, 4), 4 warps).  The row update runs with
// 8 rows per warp and 4 columns per lane; the dot products and the triangular product
// run with one row per lane and one 16-token block per warp, reading the rows from
// shared memory (padded: conflict-free) and K and T as broadcasts.  Each chunk's K, Q'
// and T arrive by bulk copy into a two-stage ring one chunk ahead.
constexpr int kBsRowStride = kD + 4;   // dS rows in shared memory
constexpr int kBsAStride = kScanCtaRows + 1;
constexpr uint32_t kBsStageBytes = (2 * kC * kD + kC * kC) * 4;  // K, Q', T of a chunk
constexpr size_t kScanBwdSmem = 2 * (size_t)kBsStageBytes +
                                (size_t)(kScanCtaRows * kBsRowStride + kC * kBsAStride +
                                         2 * kC * kScanVStride) * 4 + 64;
__global__ void __launch_bounds__(32 * kScanWarps) gdn_scan_bwd(int nC, const float* __restrict__ kf,
                                                                const float* __restrict__ qf,
                                                                const float* __restrict__ dof,
                                                                const float* __restrict__ Tm,
                                                                const float* __restrict__ dZ0,
                                                                const float* __restrict__ gam,
                                                                const float* __restrict__ lam,
                                                                const float* __restrict__ bet,
                                                                float* dSC, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t smraw[];
  float* ring = reinterpret_cast<float*>(smraw);              // stage: K, Q' [64][128], T [64][64]
  float* Ssm = ring + 2 * (2 * kC * kD + kC * kC);            // [32][kBsRowStride]
  float* Asm = Ssm + kScanCtaRows * kBsRowStride;             // [64][kBsAStride]: lam_s a_s
  float* Cq = Asm + kC * kBsAStride;                           // [64][kScanVStride]
  float* Ck = Cq + kC * kScanVStride;                         // [64][kScanVStride]
  const uint32_t full0 = smem_u32(Ck + kC * kScanVStride);
  const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp * kScanWarpRows;   // update layout: rows wr .. wr+7, columns 4 lane ..
  const int t0 = 16 * warp;              // dot layout: row lane, tokens t0 .. t0+15
  const int i0 = blockIdx.y * kScanCtaRows;
  if (threadIdx.x == 0) {
    umma::mbar_init(full0, 1);
    umma::mbar_init(full0 + 8, 1);
    umma::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int n) {  // the n-th chunk in reverse order into stage n & 1 (one thread)
    const int st = n & 1;
    const int64_t b = (int64_t)h * nC + (nC - 1 - n);
    float* dst = ring + st * (2 * kC * kD + kC * kC);
    umma::mbar_expect_tx(full0 + 8 * st, kBsStageBytes);
    umma::bulk_load(smem_u32(dst), kf + b * kC * kD, kC * kD * 4, full0 + 8 * st);
    umma::bulk_load(smem_u32(dst + kC * kD), qf + b * kC * kD, kC * kD * 4, full0 + 8 * st);
    umma::bulk_load(smem_u32(dst + 2 * kC * kD), Tm + b * kC * kC, kC * kC * 4, full0 + 8 * st);
  };
  int issued = 0;
  if (threadIdx.x == 0 && nC > 0) {
    issue(0);
    issued = 1;
  }
  float dS[kScanWarpRows][4];
#pragma unroll
  for (int r = 0; r < kScanWarpRows; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) dS[r][q] = 0.f;
  for (int n = 0; n < nC; ++n) {
    const int c = nC - 1 - n, st = n & 1;
    const int64_t b = (int64_t)h * nC + c;
    // this chunk's dZ0, dO (this lane's row, the warp's tokens) and per-token scalars
    float dz0[16], dov[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      dz0[tt] = dZ0[(b * kC + t0 + tt) * kD + i0 + lane];
      dov[tt] = dof[(b * kC + t0 + tt) * kD + i0 + lane];
    }
    const float gC = gam[b * kC + kC - 1];
    // dS entering this step: to dSC and to shared memory
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r) {
      const float4 v = make_float4(dS[r][0], dS[r][1], dS[r][2], dS[r][3]);
      *reinterpret_cast<float4*>(dSC + (b * kD + i0 + wr + r) * kD + 4 * lane) = v;
      *reinterpret_cast<float4*>(Ssm + (wr + r) * kBsRowStride + 4 * lane) = v;
    }
    __syncthreads();  // rows in shared memory; the other stage's last readers are done
    if (threadIdx.x == 0 && n + 1 < nC) {
      issue(n + 1);
      issued = n + 2;
    }
    const bool got = umma::mbar_wait(full0 + 8 * st, (n >> 1) & 1);
    if (!__syncthreads_and(got)) {
      if (threadIdx.x == 0) ls_report(err, LS_DEVERR_TIMEOUT);
      break;
    }
    const float* Ks = ring + st * (2 * kC * kD + kC * kC);
    const float* Qs = Ks + kC * kD;
    const float* Ts = Qs + kC * kD;
    // a_t = K[t] . dS[row lane] for the warp's 16 tokens
    float av[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) av[tt] = 0.f;
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
      const float4 sv = *reinterpret_cast<const float4*>(Ssm + lane * kBsRowStride + k);
#pragma unroll
      for (int tt = 0; tt < 16; ++tt) {
        const float4 kv = *reinterpret_cast<const float4*>(Ks + (t0 + tt) * kD + k);
        av[tt] = fmaf(kv.x, sv.x, fmaf(kv.y, sv.y, fmaf(kv.z, sv.z, fmaf(kv.w, sv.w, av[tt]))));
      }
    }
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) Asm[(t0 + tt) * kBsAStride + lane] = __ldg(lam + b * kC + t0 + tt) * av[tt];
    __syncthreads();
    // z_t = sum_{s >= t} T[s][t] lam_s a_s  (T[s][t] = 0 for s < t)
    float z[16];
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) z[tt] = 0.f;
    for (int s2 = t0; s2 < kC; ++s2) {
      const float bs = Asm[s2 * kBsAStride + lane];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 tv = *reinterpret_cast<const float4*>(Ts + s2 * kC + t0 + 4 * q4);
        z[4 * q4 + 0] = fmaf(tv.x, bs, z[4 * q4 + 0]);
        z[4 * q4 + 1] = fmaf(tv.y, bs, z[4 * q4 + 1]);
        z[4 * q4 + 2] = fmaf(tv.z, bs, z[4 * q4 + 2]);
        z[4 * q4 + 3] = fmaf(tv.w, bs, z[4 * q4 + 3]);
      }
    }
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      const int t = t0 + tt;
      const float gm = __ldg(gam + b * kC + t);
      Cq[t * kScanVStride + lane] = gm * dov[tt];
      Ck[t * kScanVStride + lane] = gm * __ldg(bet + b * kC + t) * (dz0[tt] + z[tt]);
    }
    __syncthreads();
    // dS[i] <- gamma_C dS[i] + sum_t (cq_t Q'[t] - ck_t K[t])
#pragma unroll
    for (int r = 0; r < kScanWarpRows; ++r)
#pragma unroll
      for (int q = 0; q < 4; ++q) dS[r][q] *= gC;
#pragma unroll 2
    for (int t = 0; t < kC; ++t) {
      const float4 kv = *reinterpret_cast<const float4*>(Ks + t * kD + 4 * lane);
      const float4 qv = *reinterpret_cast<const float4*>(Qs + t * kD + 4 * lane);
      const float4 qa = *reinterpret_cast<const float4*>(Cq + t * kScanVStride + wr);
      const float4 qb = *reinterpret_cast<const float4*>(Cq + t * kScanVStride + wr + 4);
      const float4 ka = *reinterpret_cast<const float4*>(Ck + t * kScanVStride + wr);
      const float4 kb = *reinterpret_cast<const float4*>(Ck + t * kScanVStride + wr + 4);
      const float cq[kScanWarpRows] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
      const float ck[kScanWarpRows] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int r = 0; r < kScanWarpRows; ++r) {
        dS[r][0] = fmaf(cq[r], qv.x, fmaf(-ck[r], kv.x, dS[r][0]));
        dS[r][1] = fmaf(cq[r], qv.y, fmaf(-ck[r], kv.y, dS[r][1]));
        dS[r][2] = fmaf(cq[r], qv.z, fmaf(-ck[r], kv.z, dS[r][2]));
        dS[r][3] = fmaf(cq[r], qv.w, fmaf(-ck[r], kv.w, dS[r][3]));
      }
    }
  }
  // do not leave while a copy into this CTA's shared memory may be in flight
  if (threadIdx.x == 0)
    for (int n = issued - 2 > 0 ? issued - 2 : 0; n < issued; ++n)
      umma::mbar_wait(full0 + 8 * (n & 1), (n >> 1) & 1);
}

// ---------------------------------------------------------------- outputs
// o (bf16 [R][H][128]) from the chunk-major fp32 result.  Grid (nC, H), 128 threads.
__global__ void __launch_bounds__(128) gdn_store_o(const float* __restrict__ X, int R, int H,
                                                   __nv_bfloat16* o) {
  const int c = blockIdx.x, h = blockIdx.y, nC = gridDim.x, j = threadIdx.x;
  const int64_t b = (int64_t)h * nC + c;
  for (int t = 0; t < kC; ++t) {
    const int tok = c * kC + t;
    if (tok < R) o[((int64_t)tok * H + h) * kD + j] = __float2bfloat16_rn(X[(b * kC + t) * kD + j]);
  }
}

// dq, dk, dv (fp32 [R][H][128]) from chunk-major results (accumulate adds).
__global__ void __launch_bounds__(128) gdn_store_grads(const float* __restrict__ dQ,
                                                       const float* __restrict__ dK,
                                                       const float* __restrict__ dV, int R, int H,
                                                       float qscale, int accumulate, float* dq,
                                                       float* dk, float* dv) {
  const int c = blockIdx.x, h = blockIdx.y, nC = gridDim.x, j = threadIdx.x;
  const int64_t b = (int64_t)h * nC + c;
  for (int t = 0; t < kC; ++t) {
    const int tok = c * kC + t;
    if (tok >= R) break;
    const int64_t src = (b * kC + t) * kD + j, dst = ((int64_t)tok * H + h) * kD + j;
    const float x = qscale * dQ[src], y = dK[src], z = dV[src];
    dq[dst] = accumulate ? dq[dst] + x : x;
    dk[dst] = accumulate ? dk[dst] + y : y;
    dv[dst] = accumulate ? dv[dst] + z : z;
  }
}

// Per chunk: dbeta and dg.  With dlam_t = U_t . (dSC k_t), the row dots of the chunk and
// the row/column sums of dP * P and dMs * Ms:
//   dG_t = gamma_t dO_t . (S0 q'_t) - gamma_t dY_t . (S0 k_t) + rowsum_t(dP P) -
//          colsum_t(dP P) + rowsum_t(dMs Ms) - colsum_t(dMs Ms) - lam_t dlam_t
//          + [t = C-1] (gamma_C <dSC, S0> + sum_i lam_i dlam_i)
//   dg_j = sum_{t >= j} dG_t;   dbeta_t = dZ_t . Y_t + sum_i dA[t][i] Ms[t][i]
// Grid (nC, H), 256 threads.
struct GdnScalarIn {
  const float *u, *kds, *dof, *qs, *dy, *ks, *dz, *y;  // [nb][64][128]
  const float *dp, *p, *dms, *ms, *da;                 // [nb][64][64]
  const float *sc, *dsc;                               // [nb][128][128]
  const float *gam, *lam;                              // [nb][64]
};
__global__ void __launch_bounds__(256) gdn_scalar_grads(const GdnScalarIn in, int R, int H,
                                                        int accumulate, float* dg, float* dbeta) {
  const int c = blockIdx.x, h = blockIdx.y, nC = gridDim.x;
  const int64_t b = (int64_t)h * nC + c;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float dG[kC], dl[kC], zb[kC], red[8];
  // row dots, one warp per row
  for (int t = warp; t < kC; t += 8) {
    const int64_t r = (b * kC + t) * kD;
    float s_l = 0.f, s_o = 0.f, s_y = 0.f, s_z = 0.f;
    for (int a = lane; a < kD; a += 32) {
      s_l += in.u[r + a] * in.kds[r + a];
      s_o += in.dof[r + a] * in.qs[r + a];
      s_y += in.dy[r + a] * in.ks[r + a];
      s_z += in.dz[r + a] * in.y[r + a];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s_l += __shfl_xor_sync(0xffffffffu, s_l, off);
      s_o += __shfl_xor_sync(0xffffffffu, s_o, off);
      s_y += __shfl_xor_sync(0xffffffffu, s_y, off);
      s_z += __shfl_xor_sync(0xffffffffu, s_z, off);
    }
    if (lane == 0) {
      const float gm = in.gam[b * kC + t];
      dl[t] = s_l;
      dG[t] = gm * s_o - gm * s_y - in.lam[b * kC + t] * s_l;
      zb[t] = s_z;
    }
  }
  // <dSC, S0>
  float sd = 0.f;
  for (int e = tid; e < kD * kD; e += blockDim.x) sd += in.dsc[b * kD * kD + e] * in.sc[b * kD * kD + e];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, off);
  if (lane == 0) red[warp] = sd;
  __syncthreads();
  {
    const float* dp = in.dp + b * kC * kC;
    const float* pp = in.p + b * kC * kC;
    const float* dm = in.dms + b * kC * kC;
    const float* mm = in.ms + b * kC * kC;
    const float* da = in.da + b * kC * kC;
    // row sums: one warp per row (coalesced), reduced by shuffles
    for (int t = warp; t < kC; t += 8) {
      float r1 = 0.f, r2 = 0.f, rb = 0.f;
#pragma unroll
      for (int i = lane; i < kC; i += 32) {
        const float m = mm[t * kC + i];
        r1 += dp[t * kC + i] * pp[t * kC + i];
        r2 += dm[t * kC + i] * m;
        rb += da[t * kC + i] * m;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        r1 += __shfl_xor_sync(0xffffffffu, r1, off);
        r2 += __shfl_xor_sync(0xffffffffu, r2, off);
        rb += __shfl_xor_sync(0xffffffffu, rb, off);
      }
      if (lane == 0) {
        dG[t] += r1 + r2;
        zb[t] += rb;
      }
    }
    __syncthreads();
    // column sums: one thread per column (coalesced across the columns)
    if (tid < kC) {
      const int t = tid;
      float c1 = 0.f, c2 = 0.f;
      for (int i = 0; i < kC; ++i) {
        c1 += dp[i * kC + t] * pp[i * kC + t];
        c2 += dm[i * kC + t] * mm[i * kC + t];
      }
      dG[t] -= c1 + c2;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float sdot = 0.f, sl = 0.f;
    for (int w = 0; w < 8; ++w) sdot += red[w];
    for (int i = 0; i < kC; ++i) sl += in.lam[b * kC + i] * dl[i];
    dG[kC - 1] += in.gam[b * kC + kC - 1] * sdot + sl;
    float run = 0.f;  // dg_j = sum_{t >= j} dG_t
    for (int t = kC - 1; t >= 0; --t) {
      run += dG[t];
      dG[t] = run;
    }
  }
  __syncthreads();
  if (tid < kC) {
    const int tok = c * kC + tid;
    if (tok < R) {
      const int64_t o = (int64_t)tok * H + h;
      dg[o] = accumulate ? dg[o] + dG[tid] : dG[tid];
      dbeta[o] = accumulate ? dbeta[o] + zb[tid] : zb[tid];
    }
  }
}

// ---------------------------------------------------------------- launch helpers
struct Launcher {
  cudaStream_t st;
  cudaError_t err = cudaSuccess;
  void check() {
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err == cudaSuccess) ls_note_launch();
  }
};

// C = alpha diag(rs) op(A) op(B) (+C), all nb batches; M x N output, contraction K.
void gemm(Launcher& L, int nb, bool ta, bool tb, int M, int N, int K, const float* A, int lda,
          int64_t sA, const float* B, int ldb, int64_t sB, float* C, int ldc, int64_t sC,
          float alpha, const float* rs = nullptr, int64_t srs = kC, int accumulate = 0,
          int mask = 0) {
  if (L.err != cudaSuccess) return;
  const dim3 grid(N / 64, M / 64, nb);
  if (!ta && !tb)
    gdn_gemm<false, false><<<grid, 64, 0, L.st>>>(A, lda, sA, B, ldb, sB, C, ldc, sC, K, alpha, rs, srs, accumulate, mask);
  else if (!ta && tb)
    gdn_gemm<false, true><<<grid, 64, 0, L.st>>>(A, lda, sA, B, ldb, sB, C, ldc, sC, K, alpha, rs, srs, accumulate, mask);
  else if (ta && !tb)
    gdn_gemm<true, false><<<grid, 64, 0, L.st>>>(A, lda, sA, B, ldb, sB, C, ldc, sC, K, alpha, rs, srs, accumulate, mask);
  else
    gdn_gemm<true, true><<<grid, 64, 0, L.st>>>(A, lda, sA, B, ldb, sB, C, ldc, sC, K, alpha, rs, srs, accumulate, mask);
  L.check();
}

constexpr int64_t kCD = kC * kD, kCC = kC * kC, kDD = kD * kD;

// The state-independent chunk algebra and the forward state hand-off, shared by the
// forward and the backward (which recomputes it): T, W, U (= U0 - W S0^T after the scan),
// Sc, and P = (Q' K^T) * Gam (lower incl.).
void gdn_common(Launcher& L, const LsGdnArgs& a, const GdnLayout& W_, void* ws,
                const void* d_o, float* state_out) {
  const int nb = W_.nb, nC = W_.nC;
  float* qf = at<float>(ws, W_.qf);
  float* kf = at<float>(ws, W_.kf);
  float* vf = at<float>(ws, W_.vf);
  float* dof = d_o ? at<float>(ws, W_.dof) : nullptr;
  float* gcum = at<float>(ws, W_.gcum);
  float* gam = at<float>(ws, W_.gam);
  float* lam = at<float>(ws, W_.lam);
  float* bet = at<float>(ws, W_.beta);
  gdn_load<<<dim3(nC, a.H), 128, 0, L.st>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), static_cast<const __nv_bfloat16*>(d_o), a.g, a.beta,
      a.R, a.H, a.scale, qf, kf, vf, dof, gcum, gam, lam, bet);
  L.check();
  float* ms = at<float>(ws, W_.ms);
  float* tm = at<float>(ws, W_.tm);
  float* pm = at<float>(ws, W_.p);
  float* x1 = at<float>(ws, W_.x1);
  float* x2 = at<float>(ws, W_.x2);
  float* w = at<float>(ws, W_.w);
  float* u = at<float>(ws, W_.u);
  // A = diag(beta) (K K^T * Gam) strictly lower (in tm for now), Ms kept
  gemm(L, nb, false, true, kC, kC, kD, kf, kD, kCD, kf, kD, kCD, tm, kC, kCC, 1.f);
  if (L.err != cudaSuccess) return;
  gdn_decay<<<nb, 256, 0, L.st>>>(tm, gcum, bet, 1, ms);
  L.check();
  // T = (I + A)^-1, in place of A (read into shared memory first)
  if (L.err != cudaSuccess) return;
  gdn_tri_inv<<<nb, kC, 0, L.st>>>(tm, tm);
  L.check();
  // W = T diag(beta gamma) K,  U0 = T diag(beta) V
  if (L.err != cudaSuccess) return;
  gdn_rows<<<nb, 256, 0, L.st>>>(x1, kf, bet, gam, 1.f, nullptr, 0.f);
  L.check();
  if (L.err != cudaSuccess) return;
  gdn_rows<<<nb, 256, 0, L.st>>>(x2, vf, bet, nullptr, 1.f, nullptr, 0.f);
  L.check();
  // W^T [128][64] per chunk (the state hand-off reads W by columns)
  gemm(L, nb, true, true, kD, kC, kC, x1, kD, kCD, tm, kC, kCC, w, kC, kCD, 1.f);
  gemm(L, nb, false, false, kC, kD, kC, tm, kC, kCC, x2, kD, kCD, u, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return;
  L.err = cudaFuncSetAttribute(gdn_scan_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kScanFwdSmem);
  if (L.err != cudaSuccess) return;
  gdn_scan_fwd<<<dim3(a.H, kD / kScanCtaRows), 32 * kScanWarps, kScanFwdSmem, L.st>>>(
      a.state0, nC, w, kf, u, gam, lam, at<float>(ws, W_.sc), state_out, a.err);
  L.check();
  // P = (Q' K^T) * Gam, lower incl.
  gemm(L, nb, false, true, kC, kC, kD, qf, kD, kCD, kf, kD, kCD, pm, kC, kCC, 1.f);
  if (L.err != cudaSuccess) return;
  gdn_decay<<<nb, 256, 0, L.st>>>(pm, gcum, nullptr, 0, nullptr);
  L.check();
}

}  // namespace

size_t ls_gdn_ws_bytes(int R, int H, bool bwd) { return gdn_layout(R, H, bwd).total; }

cudaError_t ls_launch_gdn_fwd(const LsGdnArgs& a, void* o, float* state_out, void* ws,
                              cudaStream_t st) {
  const GdnLayout W_ = gdn_layout(a.R, a.H, false);
  Launcher L{st};
  gdn_common(L, a, W_, ws, nullptr, state_out);
  const int nb = W_.nb;
  float* x1 = at<float>(ws, W_.x1);
  // O = diag(gamma) Q' S0^T + P U
  gemm(L, nb, false, true, kC, kD, kD, at<float>(ws, W_.qf), kD, kCD, at<float>(ws, W_.sc), kD,
       kDD, x1, kD, kCD, 1.f, at<float>(ws, W_.gam));
  gemm(L, nb, false, false, kC, kD, kC, at<float>(ws, W_.p), kC, kCC, at<float>(ws, W_.u), kD,
       kCD, x1, kD, kCD, 1.f, nullptr, kC, 1);
  if (L.err != cudaSuccess) return L.err;
  gdn_store_o<<<dim3(W_.nC, a.H), kD, 0, st>>>(x1, a.R, a.H, static_cast<__nv_bfloat16*>(o));
  L.check();
  return L.err;
}

cudaError_t ls_launch_gdn_bwd(const LsGdnArgs& a, const void* d_o, int accumulate, float* dq,
                              float* dk, float* dv, float* dg, float* dbeta, void* ws,
                              cudaStream_t st) {
  const GdnLayout W_ = gdn_layout(a.R, a.H, true);
  Launcher L{st};
  gdn_common(L, a, W_, ws, d_o, nullptr);
  const int nb = W_.nb, nC = W_.nC;
  float* qf = at<float>(ws, W_.qf);
  float* kf = at<float>(ws, W_.kf);
  float* vf = at<float>(ws, W_.vf);
  float* dof = at<float>(ws, W_.dof);
  float* gam = at<float>(ws, W_.gam);
  float* lam = at<float>(ws, W_.lam);
  float* bet = at<float>(ws, W_.beta);
  float* gcum = at<float>(ws, W_.gcum);
  float* ms = at<float>(ws, W_.ms);
  float* tm = at<float>(ws, W_.tm);
  float* pm = at<float>(ws, W_.p);
  float* u = at<float>(ws, W_.u);
  float* sc = at<float>(ws, W_.sc);
  float* dsc = at<float>(ws, W_.dsc);
  float* x1 = at<float>(ws, W_.x1);
  float* x2 = at<float>(ws, W_.x2);
  float* x3 = at<float>(ws, W_.x3);
  float* x4 = at<float>(ws, W_.x4);
  float* x5 = at<float>(ws, W_.x5);
  float* x6 = at<float>(ws, W_.x6);
  float* m1 = at<float>(ws, W_.m1);
  float* m2 = at<float>(ws, W_.m2);
  float* w = at<float>(ws, W_.w);
  // x3 = P^T dO;  dZ0 = T^T x3 (in w, free after the forward scan)
  gemm(L, nb, true, false, kC, kD, kC, pm, kC, kCC, dof, kD, kCD, x3, kD, kCD, 1.f);
  gemm(L, nb, true, false, kC, kD, kC, tm, kC, kCC, x3, kD, kCD, w, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return L.err;
  {
    L.err = cudaFuncSetAttribute(gdn_scan_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kScanBwdSmem);
    if (L.err != cudaSuccess) return L.err;
    gdn_scan_bwd<<<dim3(a.H, kD / kScanCtaRows), 32 * kScanWarps, kScanBwdSmem, st>>>(
        nC, kf, qf, dof, tm, w, gam, lam, bet, dsc, a.err);
    L.check();
  }
  // x1 = K S0^T (the state's read-out at k_t);  x2 = Y = V - diag(gamma) x1
  gemm(L, nb, false, true, kC, kD, kD, kf, kD, kCD, sc, kD, kDD, x1, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return L.err;
  gdn_rows<<<nb, 256, 0, st>>>(x2, x1, gam, nullptr, -1.f, vf, 1.f);
  L.check();
  // x4 = K dSC^T;  dU = x3 + diag(lam) x4 (into x3)
  gemm(L, nb, false, true, kC, kD, kD, kf, kD, kCD, dsc, kD, kDD, x4, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return L.err;
  gdn_rows<<<nb, 256, 0, st>>>(x3, x4, lam, nullptr, 1.f, x3, 1.f);
  L.check();
  // x5 = dZ = T^T dU;  x6 = dY = diag(beta) dZ (= dV)
  gemm(L, nb, true, false, kC, kD, kC, tm, kC, kCC, x3, kD, kCD, x5, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return L.err;
  gdn_rows<<<nb, 256, 0, st>>>(x6, x5, bet, nullptr, 1.f, nullptr, 0.f);
  L.check();
  // m1 = dA = -(dZ U^T) strictly lower;  tm <- dMs = diag(beta) dA (T is no longer needed)
  gemm(L, nb, false, true, kC, kC, kD, x5, kD, kCD, u, kD, kCD, m1, kC, kCC, -1.f, nullptr, kC, 0, 2);
  gemm(L, nb, false, true, kC, kC, kD, x5, kD, kCD, u, kD, kCD, tm, kC, kCC, -1.f, bet, kC, 0, 2);
  // m2 = dP = dO U^T lower incl.
  gemm(L, nb, false, true, kC, kC, kD, dof, kD, kCD, u, kD, kCD, m2, kC, kCC, 1.f, nullptr, kC, 0, 1);
  // x3 <- Q' S0^T (for dg; dU is no longer needed)
  gemm(L, nb, false, true, kC, kD, kD, qf, kD, kCD, sc, kD, kDD, x3, kD, kCD, 1.f);
  if (L.err != cudaSuccess) return L.err;
  {
    GdnScalarIn in;
    in.u = u; in.kds = x4; in.dof = dof; in.qs = x3; in.dy = x6; in.ks = x1; in.dz = x5;
    in.y = x2; in.dp = m2; in.p = pm; in.dms = tm; in.ms = ms; in.da = m1; in.sc = sc;
    in.dsc = dsc; in.gam = gam; in.lam = lam;
    gdn_scalar_grads<<<dim3(nC, a.H), 256, 0, st>>>(in, a.R, a.H, accumulate, dg, dbeta);
    L.check();
  }
  if (L.err != cudaSuccess) return L.err;
  // dP * Gam (m2) and dKK = dMs * Gam (tm), lower / strictly lower
  gdn_decay<<<nb, 256, 0, st>>>(m2, gcum, nullptr, 0, nullptr);
  L.check();
  if (L.err != cudaSuccess) return L.err;
  gdn_decay<<<nb, 256, 0, st>>>(tm, gcum, nullptr, 1, nullptr);
  L.check();
  // dQ' = diag(gamma) dO S0 + (dP Gam) K   -> x1 (K S0^T no longer needed)
  gemm(L, nb, false, false, kC, kD, kD, dof, kD, kCD, sc, kD, kDD, x1, kD, kCD, 1.f, gam);
  gemm(L, nb, false, false, kC, kD, kC, m2, kC, kCC, kf, kD, kCD, x1, kD, kCD, 1.f, nullptr, kC, 1);
  // dK = diag(lam) U dSC + (dP Gam)^T Q' - diag(gamma) dY S0 + (dKK + dKK^T) K  -> x4
  gemm(L, nb, false, false, kC, kD, kD, u, kD, kCD, dsc, kD, kDD, x4, kD, kCD, 1.f, lam);
  gemm(L, nb, true, false, kC, kD, kC, m2, kC, kCC, qf, kD, kCD, x4, kD, kCD, 1.f, nullptr, kC, 1);
  gemm(L, nb, false, false, kC, kD, kD, x6, kD, kCD, sc, kD, kDD, x4, kD, kCD, -1.f, gam, kC, 1);
  gemm(L, nb, false, false, kC, kD, kC, tm, kC, kCC, kf, kD, kCD, x4, kD, kCD, 1.f, nullptr, kC, 1);
  gemm(L, nb, true, false, kC, kD, kC, tm, kC, kCC, kf, kD, kCD, x4, kD, kCD, 1.f, nullptr, kC, 1);
  if (L.err != cudaSuccess) return L.err;
  gdn_store_grads<<<dim3(nC, a.H), kD, 0, st>>>(x1, x4, x6, a.R, a.H, a.scale, accumulate, dq, dk,
                                                dv);
  L.check();
  return L.err;
}
