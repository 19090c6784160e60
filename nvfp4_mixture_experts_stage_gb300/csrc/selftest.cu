// Self-test of the bounded waits every pipeline role of the GEMM kernels uses: a wait
// on an mbarrier that nothing completes must give up after the limit, report
// MOE_ERR_TIMEOUT and raise the block's abort flag, and another role's wait must then
// return through that flag.
#include "tcgen05.cuh"

namespace moe {

__global__ void __launch_bounds__(64, 1) selftest_bounded_wait_kernel(int32_t* status, int32_t* result) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = wait_bar_bounded(&bar[0], 0, &abort_flag, status);
    result[0] = (!ok && globaltimer_ns() - t0 >= kWaitLimitNs) ? 1 : 0;
  } else if (threadIdx.x == 32) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kWaitLimitNs / 2) {
    }
    const uint64_t t1 = globaltimer_ns();
    const bool ok = wait_bar_bounded(&bar[1], 0, &abort_flag, status);
    result[1] = (!ok && globaltimer_ns() - t1 < kWaitLimitNs) ? 1 : 0;
  }
  // both barriers are left with their phase pending; nothing refers to them afterwards
}

moe_status selftest_bounded_wait(int32_t* status, int32_t* result, cudaStream_t st) {
  selftest_bounded_wait_kernel<<<1, 64, 0, st>>>(status, result);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
