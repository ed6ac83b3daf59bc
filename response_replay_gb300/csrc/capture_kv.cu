// capture_kv.cu -- write the prompt's K/V into pages behind the page table.
//
// Prompt capture keeps the prompt's K/V as resident, read-only pages (LongStraw digest,
// "Method" step 1; explainer, "The move: change the graph boundary").  This is a pure
// HBM copy: 2 * n * hkv * 256 bytes read and written.  Each thread moves 16-byte
// vectors; 16 consecutive threads cover one 256-byte (head, position) row, so reads are
// fully coalesced and writes land as whole 256-byte rows inside a page.
#include "ls_device.cuh"
#include "ls_internal.h"

namespace {

constexpr int kVecPerRow = 16;  // 128 bf16 = 256 bytes = 16 x 16 bytes
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(256) capture_kv_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, const int32_t* __restrict__ page_table, int32_t num_pages,
    int32_t ps_log2, int32_t hkv, int64_t start_pos, int64_t n, uint32_t* err) {
  const int64_t total = n * hkv * kVecPerRow;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t ps_mask = (1ll << ps_log2) - 1;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += stride * kUnroll) {
    uint4 kv[kUnroll], vv[kUnroll];
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = base + u * stride;
      dst[u] = -1;
      if (i < total) {
        const int64_t row = i / kVecPerRow;
        const int c = (int)(i % kVecPerRow);
        const int64_t tok = row / hkv;
        const int h = (int)(row % hkv);
        const int64_t p = start_pos + tok;
        const int32_t phys = __ldg(page_table + (p >> ps_log2));
        if ((uint32_t)phys < (uint32_t)num_pages) {
          dst[u] = ((((int64_t)phys * hkv + h) << ps_log2) + (p & ps_mask)) * kVecPerRow + c;
          kv[u] = __ldcs(k + i);
          vv[u] = __ldcs(v + i);
        } else {
          ls_report(err, LS_DEVERR_CHECK);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (dst[u] >= 0) {
        k_pool[dst[u]] = kv[u];
        v_pool[dst[u]] = vv[u];
      }
    }
  }
}

// Page-table check: every entry in [0, num_pages) and no physical page used twice.
// `seen` is a zeroed bitmap of num_pages bits.
__global__ void validate_pages_kernel(const int32_t* __restrict__ page_table, int32_t num_logical,
                                      int32_t num_pages, uint32_t* seen, uint32_t* err) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < num_logical;
       i += gridDim.x * blockDim.x) {
    const int32_t p = page_table[i];
    if ((uint32_t)p >= (uint32_t)num_pages) {
      ls_report(err, LS_DEVERR_CHECK);
      continue;
    }
    const uint32_t bit = 1u << (p & 31);
    if (atomicOr(seen + (p >> 5), bit) & bit) ls_report(err, LS_DEVERR_CHECK);
  }
}

}  // namespace

cudaError_t ls_launch_capture(const void* k, const void* v, void* k_pool, void* v_pool,
                              const int32_t* page_table, int32_t num_pages, int32_t ps_log2,
                              int32_t hkv, int64_t start_pos, int64_t n, int num_sms,
                              uint32_t* err, cudaStream_t st) {
  const int64_t total = n * hkv * kVecPerRow;
  int64_t blocks = (total + 256 * kUnroll - 1) / (256 * kUnroll);
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  capture_kv_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_pool),
      static_cast<uint4*>(v_pool), page_table, num_pages, ps_log2, hkv, start_pos, n, err);
  ls_note_launch();
  return cudaGetLastError();
}

cudaError_t ls_launch_validate_pages(const int32_t* page_table, int32_t num_logical,
                                     int32_t num_pages, uint32_t* seen, uint32_t* err,
                                     cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(seen, 0, ((size_t)num_pages + 31) / 32 * 4, st);
  if (e != cudaSuccess) return e;
  int blocks = (num_logical + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  validate_pages_kernel<<<blocks, 256, 0, st>>>(page_table, num_logical, num_pages, seen, err);
  ls_note_launch();
  return cudaGetLastError();
}
