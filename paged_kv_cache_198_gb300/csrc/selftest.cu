// selftest.cu -- a kernel that exercises the bounded mbarrier wait the other
// kernels use: it waits on a barrier nothing arrives at, so the wait must give
// up after its limit and record the timeout in the status word.
#include "device.cuh"
#include "kernels.h"

namespace tvl {
namespace {

__global__ void selftest_wait_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // no thread arrives, so the phase never completes
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0)) report(status, kDevTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* status, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace tvl
