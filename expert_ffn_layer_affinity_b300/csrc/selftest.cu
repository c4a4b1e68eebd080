// Self-test of the bounded device wait that every pipelined kernel uses.
//
// One CTA of two warps waits on an mbarrier that nothing ever arrives on,
// with a caller-given limit.  The first thread to run out of time records
// MOE_DEV_TIMEOUT in the status word and raises the CTA's abort flag; every
// other waiter sees the flag and returns too, so the kernel ends after about
// the limit and the context stays usable.  This is how a stalled pipeline
// (a copy that never lands, a peer that never arrives) surfaces to the host.
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(64) wait_selftest_kernel(unsigned long long limit_ns,
                                                           int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // phase 0 of a fresh barrier never completes: no arrive is ever made
  const bool done = mbar_wait(smem_u32(&bar), 0u, &abort_flag, status, limit_ns);
  if (done && threadIdx.x == 0) atomicOr(reinterpret_cast<unsigned int*>(status), 0x80000000u);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned long long limit_ns, int32_t* status, cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace moe
