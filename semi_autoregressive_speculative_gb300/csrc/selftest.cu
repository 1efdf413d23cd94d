// dspark_selftest_bounded_wait: the device-side timeout path, exercised
// without a fault.  One thread waits, through the same bounded mbarrier wait
// (mbar_wait) that the pipelined kernels use on their rings, for a phase that
// nothing ever completes; when the wait gives up it ORs DSPARK_STATUS_TIMEOUT
// into the workspace status word and the kernel returns normally, so the
// context stays usable.
#include "common.h"
#include "device.cuh"

namespace dspark {

__global__ void k_selftest_bounded_wait(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int no_abort;  // the wait's abort word: never set
  if (threadIdx.x == 0) {
    no_abort = 0;
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none ever comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, &no_abort)) report(status, DSPARK_STATUS_TIMEOUT);
}

}  // namespace dspark

extern "C" int dspark_selftest_bounded_wait(void* workspace, void* stream) {
  using namespace dspark;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return DSPARK_ERR_INVALID_ARG;
  k_selftest_bounded_wait<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int32_t*>(workspace));
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
