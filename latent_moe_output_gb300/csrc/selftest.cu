// Diagnostic kernel for the bounded-wait machinery: one thread waits on an
// mbarrier that nothing ever arrives at, with a caller-chosen limit, through
// the same mbar_wait the tail kernels use. The wait expires, the error word
// gets its timeout bit and the kernel returns, leaving the context usable.
#include "launch.h"
#include "ptx.cuh"

namespace lt {
namespace {

__global__ void wait_probe_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, err, &abort_flag, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, const DeviceInfo& dev, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(dev.err_word, limit_ns);
  return cudaGetLastError();
}

}  // namespace lt
