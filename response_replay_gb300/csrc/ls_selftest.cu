// ls_selftest.cu -- a check of the bounded-wait path that every tcgen05 kernel relies on:
// one thread waits, through the same mbar_wait the pipelines use, on an mbarrier that
// nothing will ever complete.  The wait must give up after its time limit and the
// kernel must record LS_DEVERR_TIMEOUT in the device error word and return, leaving the
// context usable.  Nothing faults, traps or spins without bound.
#include "ls_device.cuh"
#include "ls_internal.h"
#include "ls_umma.cuh"

namespace {

__global__ void wait_timeout_kernel(uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    umma::mbar_init(b, 1);
    umma::fence_barrier_init();
    if (!umma::mbar_wait(b, 0)) ls_report(err, LS_DEVERR_TIMEOUT);  // no arrival ever comes
  }
}

}  // namespace

cudaError_t ls_launch_wait_timeout(uint32_t* err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  ls_note_launch();
  return cudaGetLastError();
}
