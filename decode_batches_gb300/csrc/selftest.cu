// Self-test of the bounded waits' expiry path (failure detection without a GPU fault).
//
// Every wait of the layer's kernels on an mbarrier gives up after MOE_WAIT_LIMIT_NS of
// %globaltimer, sets MOE_DEVERR_TIMEOUT in a device error word and lets the kernel return, so a
// lost arrival never hangs the GPU.  In normal runs those waits always complete; this kernel
// makes one expire on purpose and then takes the GEMM kernels' abort teardown: warp 1 holds a
// TMEM allocation (as the MMA warp does), warp 0 waits on phase 0 of an mbarrier that nothing
// arrives on -- the same mbar_wait_warp the pipelines use -- and, once it has given up, the CTA
// passes its final barrier, waits out in-flight copies (abort_quiesce) and frees TMEM.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(64) wait_expiry_selftest_kernel(uint32_t* err, uint32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  uint64_t waited = 0;
  bool completed = true;
  if (warp == 0) {
    const uint64_t t0 = global_timer_ns();
    // phase 0 never completes: no thread arrives on `bar`
    completed = mbar_wait_warp(&bar, 0, &abort_flag, err);
    waited = global_timer_ns() - t0;
  }
  tc_fence_before();
  __syncthreads();
  abort_quiesce(&abort_flag);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
  if (threadIdx.x == 0) {
    result[0] = completed ? 1u : 2u;
    result[1] = static_cast<uint32_t>(waited / 1000000ull);  // milliseconds
    result[2] = abort_flag ? 1u : 0u;                       // the wait raised the CTA's abort flag
  }
}

}  // namespace moe

extern "C" moe_status moe_selftest_wait_expiry(uint32_t* err, uint32_t* result, moe_stream_t stream) {
  if (!err || !result) return moe::fail_message(MOE_ERR_INVALID_ARG, "err and result are required");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  moe::wait_expiry_selftest_kernel<<<1, 64, 0, st>>>(err, result);
  if (cudaGetLastError() != cudaSuccess) return moe::fail_message(MOE_ERR_CUDA, "self-test launch failed");
  return MOE_OK;
}
