// wna16_check_wait_timeout: the pipelines' bounded wait, run out on purpose.
//
// The GEMM kernels never trap and never wait without a bound: every mbarrier
// wait gives up after a fixed time, raises the CTA's abort flag and sets
// WNA16_DEV_TIMEOUT in the status word; the other roles see the flag, leave
// their loops, and the CTA frees its tensor memory and exits. This kernel runs
// that path with the same wait routine on barriers that nothing arrives on:
// warps 0 and 1 each wait on one (whichever gives up first raises the flag, the
// other leaves through it), warp 2 holds a TMEM allocation for the duration
// and frees it at the end. It ends after about one wait bound.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"
#include "wna16_moe.h"

namespace wna16 {

namespace {

__global__ void __launch_bounds__(96, 1) wait_timeout_kernel(int32_t* status, int32_t* roles_left) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_holder;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&tmem_holder, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp < 2) {
    const bool ok = warp_wait_all(&bars[warp], 0, &abort_flag, status);
    if ((threadIdx.x & 31) == 0 && !ok && roles_left) atomicAdd(roles_left, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_holder, 32);
  }
}

}  // namespace

}  // namespace wna16

using namespace wna16;

extern "C" wna16_status wna16_check_wait_timeout(int32_t* device_status, int32_t* roles_left, void* stream) {
  if (!device_status || (reinterpret_cast<uintptr_t>(device_status) & 3u) ||
      (reinterpret_cast<uintptr_t>(roles_left) & 3u))
    return WNA16_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 96, 0, static_cast<cudaStream_t>(stream)>>>(device_status, roles_left);
  return cudaGetLastError() == cudaSuccess ? WNA16_OK : WNA16_ERR_CUDA;
}
