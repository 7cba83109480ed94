// status.cu -- kernels around the device status word: clearing the bits a
// reader has observed, and the self-test of the bounded mbarrier wait.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"

namespace mx {
namespace {

// Clears only `bits`: a fault that another stream records between the
// host's read of the word and this kernel keeps its bit for the next reader.
__global__ void status_clear_kernel(uint32_t* status, uint32_t bits) {
  atomicAnd(status, ~bits);
}

__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
    // Nothing ever arrives on `bar`: the wait must give up by itself.
    mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  }
}

}  // namespace

cudaError_t launch_status_clear(uint32_t* status, uint32_t bits, cudaStream_t stream) {
  status_clear_kernel<<<1, 1, 0, stream>>>(status, bits);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mx
