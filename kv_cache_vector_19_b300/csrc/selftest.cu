// tq_selftest_bounded_wait: exercises the timeout path every kernel's mbarrier waits share.
// One thread waits on an mbarrier that nothing arrives at; the wait gives up after its time
// limit, the kernel records the sticky timeout flag and returns.  No GPU fault, no hang: the
// failure is made on the device's own terms and read back through tq_get_device_status.
#include <cuda_runtime.h>

#include "dev_common.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

__global__ void bounded_wait_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);   // expects one arrival; none comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !dev::mbar_wait(&bar, 0)) atomicOr(status, kFlagTimeout);
}

}  // namespace

int launch_selftest_wait(const tq_ctx* c, void* stream) {
  bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(c->d_status);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace tq
