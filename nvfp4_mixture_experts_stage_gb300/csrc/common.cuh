// Shared device helpers of the NVFP4 MoE stage (sm_103a).
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "../../include/moe_stage.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

constexpr int kTileM = 128;
constexpr int kBlock = 16;              // elements per block scale
constexpr float kGsDivisor = 2688.0f;   // 6 * 448

// Programmatic dependent launch.  A kernel launched with launch_ex(..., pdl=true)
// may start while the previous kernel of the stream is still running:
// griddep_wait() blocks until that kernel has completed and its writes are
// visible; griddep_launch_dependents() lets the next such kernel start early.
// Both are no-ops for a kernel launched without the attribute.
MOE_DEV void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEV void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                             Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- per-device launch settings (host) -----------------------------------------
// Launch settings that depend on the device (SM count, a kernel's shared-memory
// opt-in, a cluster kernel's grid) are looked up once per device and cached in
// per-device slots, so one process may drive several devices from several threads.
// Concurrent first calls on a device may both compute a value; the computations are
// idempotent and the slot is written atomically.
constexpr int kMaxDevices = 64;

inline int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices ? d : -1;
}

// A positive int per device (0 = not yet known).
struct PerDeviceInt {
  std::atomic<int> v[kMaxDevices] = {};
  template <class F>
  int get(F&& compute) {
    const int d = current_device();
    if (d < 0) return compute();
    int x = v[d].load(std::memory_order_acquire);
    if (x <= 0) {
      x = compute();
      if (x > 0) v[d].store(x, std::memory_order_release);
    }
    return x;
  }
};

// Runs set_up() (a cudaError_t-returning, idempotent call such as
// cudaFuncSetAttribute) until it first succeeds on each device.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};
  template <class F>
  cudaError_t run(F&& set_up) {
    const int d = current_device();
    const uint64_t bit = d >= 0 ? (1ull << d) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = set_up();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

inline int sm_count_of_current_device() {
  static PerDeviceInt cache;
  return cache.get([] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 1;
    return n;
  });
}

// First error wins.
MOE_DEV void set_status(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// -------------------------------------------------------------------------
// NVFP4 arithmetic, shared by the quantiser, the requantiser and the L1
// requant epilogue.  Order of fp32 operations (all round-to-nearest-even):
//   rg = 1/gs (saturated);  s = (bm*rg)/6;  sb = e4m3_rn_satfinite(s);
//   rb = 1/decode(sb);      v = (|x|*rg)*rb  -> e2m1_rn_satfinite.
// -------------------------------------------------------------------------

// rg = 1/gs, saturated to FLT_MAX; gs == 0 gives rg = 0 (all scales 0, sign-only codes).
MOE_DEV float recip_global_scale(float gs) {
  if (!(gs > 0.0f)) return 0.0f;
  float rg = __frcp_rn(gs);
  return (rg <= 3.402823466e38f) ? rg : 3.402823466e38f;  // +inf -> FLT_MAX
}

// UE4M3 byte of a non-negative fp32 (RNE, saturate to 448).
MOE_DEV uint32_t e4m3_byte(float s) {
  return (uint32_t)__nv_cvt_float_to_fp8(s, __NV_SATFINITE, __NV_E4M3);
}

MOE_DEV float e4m3_value(uint32_t b) {
  __nv_fp8_e4m3 v;
  v.__x = (__nv_fp8_storage_t)b;
  return float(v);
}

// Two fp32 -> one byte of E2M1 sign-magnitude codes (lo = first element, bits 3..0;
// hi = second element, bits 7..4), magnitude RNE saturating at 6, sign kept (also
// for a value that rounds to zero).
MOE_DEV uint32_t e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}

// Block scale byte and the reciprocal of its decoded value (0 if the scale is 0).
MOE_DEV uint32_t block_scale(float bm, float rg, float& rb) {
  float s = __fdiv_rn(__fmul_rn(bm, rg), 6.0f);
  uint32_t sb = e4m3_byte(s);
  float sd = e4m3_value(sb);
  rb = (sd > 0.0f) ? __frcp_rn(sd) : 0.0f;
  return sb;
}

// Scaled code value (x*rg)*rb; for a magnitude |x| this is the code magnitude, for a
// signed x it equals sign(x) times it exactly.  With a zero block scale rb = 0 and
// the result is a signed zero (x*rg is then tiny, never infinite).
MOE_DEV float code_mag(float ax, float rg, float rb) {
  return __fmul_rn(__fmul_rn(ax, rg), rb);
}

// Offset of scale (row m, scale column k) in the swizzled layout of a tensor
// with k_sf scale columns (k_sf % 4 == 0).
MOE_DEV int64_t sf_swizzle_offset(int64_t m, int k, int k_sf) {
  return ((m >> 7) * (k_sf >> 2) + (k >> 2)) * 512 + (m & 31) * 16 + ((m >> 5) & 3) * 4 + (k & 3);
}

MOE_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
MOE_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

MOE_DEV float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

// Bounded waits: give up after this many nanoseconds of wall time.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

MOE_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

}  // namespace moe
