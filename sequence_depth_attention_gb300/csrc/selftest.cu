// Diagnostic of the failure path: one thread waits, through the same bounded
// mbarrier wait the forward kernel uses, on a barrier that nothing arrives on.
// The wait gives up after the requested time and latches MODA_ERR_TIMEOUT in
// the device error word; the kernel then returns normally.
#include "moda_internal.h"
#include "sm103.cuh"

namespace moda {
namespace {

__global__ void selftest_wait_kernel(unsigned int* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sm103::mbar_init(sm103::smem_u32(&bar), 1);
    sm103::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = sm103::mbar_wait_bounded(sm103::smem_u32(&bar), 0, &abort_flag, timeout_ns);
    if (!ok) atomicCAS(err, 0u, (unsigned int)MODA_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned int* err, int timeout_ms, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, (uint64_t)timeout_ms * 1000000ull);
  return cudaGetLastError();
}

}  // namespace moda
