// moe_route for callers that cannot hand the library a workspace.
//
// Some callers have no way to allocate device memory at the point where they
// route tokens: a plugin whose host runtime owns every device allocation and
// passes in only the tensors of the call, or a serving loop that must never
// touch an allocator on its hot path (an allocation can synchronise the device
// or fail under memory pressure).  moe_route needs two scratch tables (per-chunk
// expert counts and the scanned per-chunk bases); this entry point keeps them in
// a fixed array that lives in the library's own device memory instead.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr int64_t kStaticTableInts = MOE_ROUTE_STATIC_TABLE_INTS;  // per table

// Two tables of kStaticTableInts int32 each (2 MiB together), resident on every
// GPU that loads the library until the process exits.  In host code this name
// is only a stand-in for the device object: its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_route_scratch[2 * kStaticTableInts];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device, looked up once per
// device (with that device current) and cached.
moe_status scratch_for_current_device(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_route_static_scratch(const int32_t* topk_ids, const float* topk_w, int64_t T, int topk,
                                               int E, int expert_offset, int32_t* counts, int32_t* offsets,
                                               int32_t* padded_offsets, int32_t* slot_token, float* slot_weight,
                                               int32_t* pair_slot, int64_t capacity, moe_stream_t stream) {
  if (T < 0 || topk < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > moe::kMaxExperts || topk > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets || !padded_offsets || !slot_token || !slot_weight) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !topk_w || !pair_slot)) return MOE_ERR_INVALID_ARG;
  if (capacity < moe_slot_capacity(T, topk, E)) return MOE_ERR_INVALID_ARG;
  const int64_t nchunks = (T * topk + moe::kRouteChunk - 1) / moe::kRouteChunk;
  if (nchunks * E > kStaticTableInts) return MOE_ERR_UNSUPPORTED_SHAPE;  // beyond the fixed scratch
  int32_t* scratch = nullptr;
  moe_status s = scratch_for_current_device(&scratch);
  if (s != MOE_OK) return s;
  // Both tables are written in full (count kernel, then scan kernel) before they
  // are read, so the previous call's contents never leak into this one.
  int32_t* cnt = scratch;
  int32_t* base = scratch + kStaticTableInts;
  cudaStream_t st = stream;
  return moe::launch_route(topk_ids, topk_w, T * topk, topk, E, expert_offset, cnt, base, (int)nchunks, counts,
                           offsets, padded_offsets, slot_token, slot_weight, pair_slot, capacity, nullptr, st) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
