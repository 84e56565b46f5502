// Diagnostic for failure detection: one bounded wait on an mbarrier that
// nothing completes. Every wait of the library's pipelines is bounded the same
// way; this kernel lets a test watch such a wait give up, set the sticky error
// flag and return, and the context stay usable, without faulting or hanging
// the GPU.
#include "dqd_device.cuh"
#include "dqd_internal.h"

namespace dqd {
namespace {

__device__ unsigned int g_selftest_error;

__global__ void selftest_wait_kernel(uint32_t polls) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none comes
    fence_mbar_init();
  }
  __syncthreads();
  bool done = false;
  for (uint32_t i = 0; i < polls && !done; ++i) done = mbar_try_wait(b, 0);
  if (!done && threadIdx.x == 0) atomicOr(&g_selftest_error, kErrWaitTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t polls, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(polls);
  return cudaGetLastError();
}

cudaError_t selftest_take_device_error(uint32_t* flags) {
  uint32_t v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof v);
  if (e != cudaSuccess) return e;
  if (v) e = cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof zero);
  *flags |= v;
  return e;
}

}  // namespace dqd
