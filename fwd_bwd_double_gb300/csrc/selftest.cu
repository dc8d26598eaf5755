// Check of the failure-detection path on the GPU, without a fault: one CTA waits on
// an mbarrier that nothing ever completes, through the same bounded wait the
// attention kernels use (with a 20 ms limit instead of 2 s).  The wait gives up,
// sets the CTA's abort flag and this translation unit's status word, and the
// kernel returns normally; the host then reads the status as ATTN_ERR_TIMEOUT.
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace fbd {
namespace {

__device__ unsigned int g_err = 0;

__global__ void __launch_bounds__(32) wait_timeout_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);  // one arrival completes the phase; none ever comes
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const ptx::BoundedWaitT<20000000ull> wait{&abort_flag, &g_err};
  (void)wait(&bar, 0);
}

}  // namespace

cudaError_t selftest_wait_timeout(cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

uint32_t selftest_take_error() {
  uint32_t v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return 0;
  if (v) cudaMemcpyToSymbol(g_err, &z, sizeof(z));
  return v;
}

}  // namespace fbd
