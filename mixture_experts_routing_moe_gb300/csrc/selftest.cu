// Self-test of the failure path the tensor-core kernels share: one bounded mbarrier wait
// (wait_bounded of tcgen05.cuh) on a barrier that nothing ever completes.  The wait gives up after
// about a second of SM clock, records the timeout bit in the status word and returns; the kernel
// then exits normally, so the context stays usable.  No fault, trap or endless loop is involved.
#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace moe {
namespace {

__global__ void moe_wait_selftest_kernel(unsigned* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_f;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);  // one arrival expected; none ever comes
    abort_f = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::wait_bounded(tc::smem_u32(&bar), 0, &abort_f, status);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned* status, cudaStream_t s) {
  moe_wait_selftest_kernel<<<1, 32, 0, s>>>(status);
  return cudaGetLastError();
}

}  // namespace moe
