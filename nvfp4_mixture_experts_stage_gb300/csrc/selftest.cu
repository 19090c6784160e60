// Self-tests of device pieces that no layer call exposes on its own:
//   * the bounded waits every pipeline role of the GEMM kernels uses: a wait on an
//     mbarrier that nothing completes must give up after the limit, report
//     MOE_ERR_TIMEOUT and raise the block's abort flag, and another role's wait must
//     then return through that flag;
//   * the two code encoders of the quantisers and the requant epilogue (E2M1 of a
//     scaled value, UE4M3 of a block scale), evaluated on arbitrary fp32 bit patterns
//     so that a test can sweep every input;
//   * the SiLU of the L1 epilogues before its product with up and the BF16 rounding of
//     h, on caller-given gate values (a test sweeps every BF16 gate value).
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

// Pattern first + i for i < n: E2M1 code (sign bit 3, magnitude index bits 2..0) of
// the value as the quantisers encode it, and the UE4M3 byte of the value as a block
// scale is encoded (meaningful for non-negative values).
__global__ void selftest_codecs_kernel(uint32_t first, int64_t n, uint8_t* e2m1, uint8_t* e4m3) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float f = __uint_as_float(first + (uint32_t)i);
    e2m1[i] = (uint8_t)(e2m1x2(f, 0.0f) & 0xFu);
    e4m3[i] = (uint8_t)e4m3_byte(f);
  }
}

moe_status selftest_codecs(uint32_t first, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t st) {
  if (n == 0) return MOE_OK;
  selftest_codecs_kernel<<<num_sms() * 8, 256, 0, st>>>(first, n, e2m1, e4m3);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__global__ void selftest_silu_kernel(const float* g, int64_t n, float* s) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    s[i] = silu_f32(g[i]);
}

moe_status selftest_silu(const float* g, int64_t n, float* s, cudaStream_t st) {
  if (n == 0) return MOE_OK;
  selftest_silu_kernel<<<num_sms() * 4, 256, 0, st>>>(g, n, s);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
