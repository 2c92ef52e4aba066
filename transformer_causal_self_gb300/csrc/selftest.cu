// A kernel that waits on a barrier nothing completes, with a time limit: the
// wait runs out, the status word gets the timeout bit, the kernel returns.
// It exercises the failure-detection path of the real kernels (every wait is
// bounded; none traps) without faulting or hanging the GPU.
#include "internal.h"

namespace csattn {
namespace {

__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, nullptr, status, limit_ns);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace csattn
