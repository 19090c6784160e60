// C ABI of the NVFP4 MoE stage: argument checks, workspace carving and launches.
// Every entry point only enqueues work on the caller's stream.
#include <cstdio>

#include <algorithm>

#include "kernels.cuh"

using namespace moe;

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline size_t align256(size_t n) { return (n + 255) & ~size_t(255); }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int sm_count() { return sm_count_of_current_device(); }

int64_t route_chunks(int64_t T, int topk) { return ceil_div(T * topk, kRouteChunk); }

// Bump allocator over the caller's workspace.
struct Carve {
  uint8_t* base;
  size_t off = 0;
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += align256(count * sizeof(T));
    return p;
  }
};

constexpr int kAmaxMaxBlocks = 4096;  // amax partials of the large-batch layer path

moe_status quantize_launch(int dst, const void* x, int64_t rows, int K, int64_t ld_x, const uint32_t* amax_bits,
                           const float* gs_fixed, float* gs_out, uint8_t* codes, uint8_t* sf,
                           const int32_t* pair_slot, int topk, const int32_t* slot_token, int64_t capacity,
                           int32_t* status, cudaStream_t st, const uint32_t* amax_partials = nullptr,
                           int n_partials = 0, bool pdl = false) {
  QuantArgs a;
  a.x = reinterpret_cast<const uint4*>(x);
  a.rows = rows;
  a.K = K;
  a.ld_vec = ld_x / 8;
  a.amax_bits = amax_bits;
  a.amax_partials = amax_partials;
  a.n_partials = n_partials;
  a.gs_fixed = gs_fixed;
  a.gs_out = gs_out;
  a.codes = codes;
  a.sf = sf;
  a.pair_slot = pair_slot;
  a.topk = topk;
  a.slot_token = slot_token;
  a.capacity = capacity;
  a.status = status;
  const int64_t warps = rows * ceil_div(K, 256);
  if (warps >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int blocks = (int)std::min<int64_t>(std::max<int64_t>(ceil_div(warps, 8 * 4), 1), (int64_t)sm_count() * 8);
  return launch_quantize(dst, a, blocks, st, pdl) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status amax_launch(const void* x, int64_t rows, int K, int64_t ld_x, uint32_t* amax_bits, cudaStream_t st) {
  if (cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  const int64_t vecs = rows * (K / 8);
  if (vecs == 0) return MOE_OK;
  if (vecs >= (int64_t(1) << 32)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int blocks = (int)std::min<int64_t>(std::max<int64_t>(ceil_div(vecs, 256 * 4), 1), (int64_t)sm_count() * 8);
  return launch_amax(x, rows, K, ld_x, amax_bits, blocks, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status route_impl(const int32_t* ids, const float* w, int64_t T, int topk, int E, int off, int32_t* counts,
                      int32_t* offsets, int32_t* poff, int32_t* slot_token, float* slot_weight, int32_t* pair_slot,
                      int64_t capacity, int32_t* cnt, int32_t* base, int32_t* status, cudaStream_t st) {
  const int nchunks = (int)route_chunks(T, topk);
  return launch_route(ids, w, T * topk, topk, E, off, cnt, base, nchunks, counts, offsets, poff, slot_token,
                      slot_weight, pair_slot, capacity, status, st) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// Record stage event i (if any); inside a graph capture it becomes a record node.
moe_status cast_output(const float* out32, void* out_bf16, int64_t T, int K, cudaStream_t stream, bool pdl) {
  if (T < 0 || K <= 0 || K % 8) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!out32 || !out_bf16 || !aligned(out32, 16) || !aligned(out_bf16, 16)) return MOE_ERR_INVALID_ARG;
  const int64_t n8 = T * K / 8;
  const int blocks = (int)std::min<int64_t>(ceil_div(n8, 256), (int64_t)sm_count() * 8);
  return launch_cast(out32, out_bf16, n8, blocks, stream, pdl) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status combine_rows(const void* y_rows, int64_t ld_y, const int32_t* pair_slot, const float* topk_w, int64_t T,
                        int topk, int K, int64_t capacity, void* out_bf16, int32_t* dev_status, cudaStream_t stream,
                        bool pdl, bool discard_rows = false) {
  if (T < 0 || K <= 0 || K % 8 || topk < 1 || topk > 32 || ld_y < K || ld_y % 8 || capacity < 0)
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y_rows || !pair_slot || !topk_w || !out_bf16 || !aligned(y_rows, 16) || !aligned(out_bf16, 16))
    return MOE_ERR_INVALID_ARG;
  const int64_t n8 = T * K / 8;
  const int blocks = (int)std::min<int64_t>(ceil_div(n8, 256), (int64_t)sm_count() * 8);
  return launch_combine(y_rows, ld_y, pair_slot, topk_w, topk, T, K, capacity, out_bf16, dev_status, blocks, stream,
                        pdl, discard_rows) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status mark(void* const* events, int i, cudaStream_t st) {
  if (!events || !events[i]) return MOE_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = cs == cudaStreamCaptureStatusActive
                      ? cudaEventRecordWithFlags((cudaEvent_t)events[i], st, cudaEventRecordExternal)
                      : cudaEventRecord((cudaEvent_t)events[i], st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

bool shape_ok(int K, int I, int E) {
  return K > 0 && I > 0 && K % 128 == 0 && I % 64 == 0 && E >= 1 && E <= 256;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, bad enum, misalignment or negative size)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (needs K % 128 == 0, I % 64 == 0, 1 <= E <= 256, 1 <= topk <= 32)";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or tensor-map encode failed";
    case MOE_ERR_TIMEOUT: return "device: a bounded wait gave up";
    case MOE_ERR_DEVICE_INDEX: return "device: an index failed its bounds check";
  }
  return "unknown status";
}

size_t moe_quantize_weights_workspace_size(int E, int I, int K) {
  if (E < 1 || I < 1 || K < 1) return 0;
  return align256(moe_stage_workspace_size()) + align256((size_t)E * 2 * I * (K / 16)) +
         align256((size_t)E * K * (I / 16));
}

moe_status moe_quantize_weights(const void* w1, const void* w2, int E, int I, int K, uint8_t* w1_fp4, uint8_t* w1_sf,
                                float* gs_w1_gate, float* gs_w1_up, uint8_t* w2_fp4, uint8_t* w2_sf, float* gs_w2,
                                void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!w1 || !w2 || !w1_fp4 || !w1_sf || !gs_w1_gate || !gs_w1_up || !w2_fp4 || !w2_sf || !gs_w2 || !ws)
    return MOE_ERR_INVALID_ARG;
  if (E < 1 || I < 1 || K < 1 || !aligned(w1, 16) || !aligned(w2, 16)) return MOE_ERR_INVALID_ARG;
  if (I % 64 || K % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < moe_quantize_weights_workspace_size(E, I, K)) return MOE_ERR_WORKSPACE;
  uint8_t* p = static_cast<uint8_t*>(ws);
  void* sws = p;
  p += align256(moe_stage_workspace_size());
  uint8_t* sf1 = p;  // row-major [E, 2I, K/16]
  p += align256((size_t)E * 2 * I * (K / 16));
  uint8_t* sf2 = p;  // row-major [E, K, I/16]
  const uint8_t* x1 = static_cast<const uint8_t*>(w1);
  const uint8_t* x2 = static_cast<const uint8_t*>(w2);
  const size_t sws_bytes = moe_stage_workspace_size();
  for (int e = 0; e < E; ++e) {
    for (int h = 0; h < 2; ++h) {  // gate rows, then up rows
      const int64_t r0 = (int64_t)e * 2 * I + (int64_t)h * I;
      moe_status s = moe_stage_activation(x1 + r0 * K * 2, I, K, K, w1_fp4 + r0 * (K / 2), sf1 + r0 * (K / 16),
                                          MOE_SF_ROWMAJOR, (h ? gs_w1_up : gs_w1_gate) + e, nullptr, sws, sws_bytes,
                                          nullptr, stream);
      if (s != MOE_OK) return s;
    }
    const int64_t r2 = (int64_t)e * K;
    moe_status s = moe_stage_activation(x2 + r2 * I * 2, K, I, I, w2_fp4 + r2 * (I / 2), sf2 + r2 * (I / 16),
                                        MOE_SF_ROWMAJOR, gs_w2 + e, nullptr, sws, sws_bytes, nullptr, stream);
    if (s != MOE_OK) return s;
  }
  moe_status s = moe_prepare_weights(sf1, w1_sf, E, 2 * I, K, MOE_PREP_W1, stream);
  if (s != MOE_OK) return s;
  return moe_prepare_weights(sf2, w2_sf, E, K, I, MOE_PREP_W2, stream);
}

moe_status moe_fold_gate_up_scales(uint8_t* w1_sf, const float* gs_gate, const float* gs_up, float* gs_common,
                                   int E, int I, int K, moe_stream_t stream) {
  if (!w1_sf || !gs_gate || !gs_up || !gs_common || E <= 0 || I <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 16) return MOE_ERR_UNSUPPORTED_SHAPE;
  return launch_fold_gate_up(w1_sf, gs_gate, gs_up, gs_common, E, I, K, (cudaStream_t)stream) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_selftest_bounded_wait(int32_t* dev_status, int32_t* dev_result, moe_stream_t stream) {
  if (!dev_status || !dev_result) return MOE_ERR_INVALID_ARG;
  return selftest_bounded_wait(dev_status, dev_result, (cudaStream_t)stream);
}

moe_status moe_selftest_codecs(uint32_t first_pattern, int64_t n, uint8_t* e2m1_codes, uint8_t* e4m3_bytes,
                               moe_stream_t stream) {
  if (n < 0 || (n > 0 && (!e2m1_codes || !e4m3_bytes))) return MOE_ERR_INVALID_ARG;
  if ((uint64_t)first_pattern + (uint64_t)n > (1ull << 32)) return MOE_ERR_INVALID_ARG;
  return selftest_codecs(first_pattern, n, e2m1_codes, e4m3_bytes, (cudaStream_t)stream);
}

moe_status moe_selftest_silu(const float* g, int64_t n, float* silu_out, moe_stream_t stream) {
  if (n < 0 || (n > 0 && (!g || !silu_out))) return MOE_ERR_INVALID_ARG;
  return selftest_silu(g, n, silu_out, (cudaStream_t)stream);
}

int moe_set_gemm_policy(int policy) {
  if (policy < MOE_GEMM_AUTO || policy > MOE_GEMM_TILED_PAIR) return -1;
  return set_gemm_policy(policy);
}

int64_t moe_slot_capacity(int64_t T, int topk, int E) {
  if (T < 0 || topk < 1 || E < 1) return -1;
  return ceil_div(T * topk + (int64_t)(kTileM - 1) * E, kTileM) * kTileM;
}

size_t moe_route_workspace_size(int64_t T, int topk, int E) {
  if (T < 0 || topk < 1 || E < 1) return 0;
  const int64_t n = route_chunks(T, topk) * E;
  return 2 * align256(std::max<int64_t>(n, 1) * sizeof(int32_t));
}

size_t moe_stage_workspace_size(void) { return 256; }

// Output path of moe_forward.  Small batches scatter w*y with fp32 atomics into an
// accumulator of T*K fp32 (L2-resident) and cast it; once that accumulator outgrows
// a quarter of L2, the atomics would thrash it through HBM (each row receives topk
// scattered updates), so the L2 GEMM writes its BF16 rows instead and one kernel
// combines each token's rows in pair order.
constexpr int64_t kCombineMinOutBytes = 32ll << 20;
static bool use_combine(int64_t T, int K) { return T * K * 4 > kCombineMinOutBytes; }

// Bytes of the output region: the fp32 accumulator, or the BF16 rows of every slot.
static int64_t out_region_bytes(int64_t T, int K, int64_t cap) {
  return std::max<int64_t>(std::max<int64_t>(T * K * 4, 4), use_combine(T, K) ? cap * K * 2 : 0);
}

static size_t forward_layout(Carve& c, int64_t T, int K, int I, int E, int topk, void** parts) {
  const int64_t cap = moe_slot_capacity(T, topk, E);
  parts[0] = c.take<uint32_t>(512);                                  // scalars, claim counters, amax partials
  parts[1] = c.take<uint8_t>(moe_route_workspace_size(T, topk, E));  // route tables
  parts[2] = c.take<int32_t>(E);                                     // counts
  parts[3] = c.take<int32_t>(E + 1);                                 // offsets
  parts[4] = c.take<int32_t>(E + 1);                                 // padded offsets
  parts[5] = c.take<int32_t>(cap);                                   // slot_token
  parts[6] = c.take<float>(cap);                                     // slot_weight
  parts[7] = c.take<int32_t>(std::max<int64_t>(T * topk, 1));        // pair_slot
  parts[8] = c.take<uint8_t>(cap * K / 2);                           // A codes
  parts[9] = c.take<uint8_t>(cap * K / 16);                          // A scales
  parts[10] = c.take<uint16_t>(cap * I);                             // h bf16
  parts[11] = c.take<uint8_t>(cap * I / 2);                          // h codes
  parts[12] = c.take<uint8_t>(cap * I / 16);                         // h scales
  parts[13] = c.take<uint8_t>(out_region_bytes(T, K, cap));         // out32, or L2 rows (combine)
  parts[14] = c.take<uint32_t>(kAmaxMaxBlocks);                      // amax partials (large batches)
  return c.off;
}

size_t moe_workspace_size(int64_t T_max, int K, int I, int E, int topk) {
  if (T_max < 0 || !shape_ok(K, I, E) || topk < 1 || topk > 32) return 0;
  Carve c{nullptr};
  void* parts[15];
  return forward_layout(c, T_max, K, I, E, topk, parts);
}

moe_status moe_prepare_weights(const uint8_t* sf_rowmajor, uint8_t* sf_prepared, int E, int N, int K, int kind,
                               moe_stream_t stream) {
  if (!sf_rowmajor || !sf_prepared || E < 1 || N < 1 || K < 1) return MOE_ERR_INVALID_ARG;
  if (kind != MOE_PREP_W1 && kind != MOE_PREP_W2) return MOE_ERR_INVALID_ARG;
  if (N % 128 || K % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int64_t total = (int64_t)E * N * (K / 16);
  const int blocks = (int)std::min<int64_t>(ceil_div(total, 256), (int64_t)sm_count() * 16);
  return launch_prepare_weight_sf(sf_rowmajor, sf_prepared, E, N, K / 16, kind == MOE_PREP_W1, blocks, stream) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_stage_activation(const void* x, int64_t T, int K, int64_t ld_x, uint8_t* x_fp4, uint8_t* x_sf,
                                int sf_layout, float* gs_out, const float* gs_fixed, void* ws, size_t ws_bytes,
                                int32_t* dev_status, moe_stream_t stream) {
  if (T < 0 || K <= 0 || ld_x < K) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !x_fp4 || !x_sf)) return MOE_ERR_INVALID_ARG;
  if (!gs_out || (!gs_fixed && !ws)) return MOE_ERR_INVALID_ARG;
  if (sf_layout != MOE_SF_ROWMAJOR && sf_layout != MOE_SF_SWIZZLED) return MOE_ERR_INVALID_ARG;
  if (K % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (ld_x % 8 || !aligned(x, 16) || !aligned(x_fp4, 4) || !aligned(x_sf, 4)) return MOE_ERR_INVALID_ARG;
  if (!gs_fixed && ws_bytes < moe_stage_workspace_size()) return MOE_ERR_WORKSPACE;
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws);
  if (!gs_fixed) {
    moe_status s = amax_launch(x, T, K, ld_x, amax, stream);
    if (s != MOE_OK) return s;
  }
  return quantize_launch(sf_layout == MOE_SF_ROWMAJOR ? 0 : 1, x, T, K, ld_x, gs_fixed ? nullptr : amax, gs_fixed,
                         gs_out, x_fp4, x_sf, nullptr, 0, nullptr, 0, dev_status, stream);
}

moe_status moe_stage_activation_to_slots(const void* x, int64_t T, int K, int64_t ld_x, const int32_t* pair_slot,
                                         int topk, int64_t capacity, uint8_t* a_fp4, uint8_t* a_sf, float* gs_out,
                                         const float* gs_fixed, void* ws, size_t ws_bytes, int32_t* dev_status,
                                         moe_stream_t stream) {
  if (T < 0 || K <= 0 || ld_x < K || topk < 1 || topk > 32 || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !pair_slot || !a_fp4 || !a_sf)) return MOE_ERR_INVALID_ARG;
  if (!gs_out || (!gs_fixed && !ws)) return MOE_ERR_INVALID_ARG;
  if (K % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (capacity % kTileM) return MOE_ERR_INVALID_ARG;
  if (ld_x % 8 || !aligned(x, 16) || !aligned(a_fp4, 4) || !aligned(a_sf, 4)) return MOE_ERR_INVALID_ARG;
  if (!gs_fixed && ws_bytes < moe_stage_workspace_size()) return MOE_ERR_WORKSPACE;
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws);
  if (!gs_fixed) {
    moe_status s = amax_launch(x, T, K, ld_x, amax, stream);
    if (s != MOE_OK) return s;
  }
  return quantize_launch(2, x, T, K, ld_x, gs_fixed ? nullptr : amax, gs_fixed, gs_out, a_fp4, a_sf, pair_slot,
                         topk, nullptr, capacity, dev_status, stream);
}

moe_status moe_route(const int32_t* topk_ids, const float* topk_w, int64_t T, int topk, int E, int expert_offset,
                     int32_t* counts, int32_t* offsets, int32_t* padded_offsets, int32_t* slot_token,
                     float* slot_weight, int32_t* pair_slot, int64_t capacity, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  if (T < 0 || topk < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > 256 || topk > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!counts || !offsets || !padded_offsets || !slot_token || !slot_weight || !ws) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !topk_w || !pair_slot)) return MOE_ERR_INVALID_ARG;
  if (capacity < moe_slot_capacity(T, topk, E)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_route_workspace_size(T, topk, E)) return MOE_ERR_WORKSPACE;
  const size_t half = moe_route_workspace_size(T, topk, E) / 2;
  int32_t* cnt = reinterpret_cast<int32_t*>(ws);
  int32_t* base = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(ws) + half);
  return route_impl(topk_ids, topk_w, T, topk, E, expert_offset, counts, offsets, padded_offsets, slot_token,
                    slot_weight, pair_slot, capacity, cnt, base, nullptr, stream);
}

moe_status moe_grouped_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a, const int32_t* offsets,
                               const int32_t* padded_offsets, int E, int64_t capacity, int K, int I,
                               const uint8_t* w1_fp4, const uint8_t* w1_sf, const float* gs_w1_gate,
                               const float* gs_w1_up, int epilogue, void* out_bf16, float* h_amax, uint8_t* h_fp4,
                               uint8_t* h_sf, const float* gs_h, int32_t* dev_status, moe_stream_t stream) {
  if (!a_fp4 || !a_sf || !gs_a || !offsets || !padded_offsets || !w1_fp4 || !w1_sf || !gs_w1_gate || !gs_w1_up)
    return MOE_ERR_INVALID_ARG;
  if (!shape_ok(K, I, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (capacity <= 0 || capacity % kTileM || capacity > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!aligned(a_fp4, 16) || !aligned(w1_fp4, 16) || !aligned(a_sf, 16) || !aligned(w1_sf, 16))
    return MOE_ERR_INVALID_ARG;
  switch (epilogue) {
    case MOE_L1_GATEUP_BF16:
    case MOE_L1_SILU_BF16:
      if (!out_bf16 || !aligned(out_bf16, 16)) return MOE_ERR_INVALID_ARG;
      break;
    case MOE_L1_SILU_REQUANT:
      if (!h_fp4 || !h_sf || !gs_h || !aligned(h_fp4, 16) || !aligned(h_sf, 4)) return MOE_ERR_INVALID_ARG;
      if (out_bf16 && !aligned(out_bf16, 16)) return MOE_ERR_INVALID_ARG;
      break;
    default: return MOE_ERR_INVALID_ARG;
  }
  return launch_gemm_l1(a_fp4, a_sf, gs_a, offsets, padded_offsets, E, capacity, K, I, w1_fp4, w1_sf, gs_w1_gate,
                        gs_w1_up, epilogue, out_bf16, epilogue == MOE_L1_SILU_BF16 ? h_amax : nullptr, h_fp4, h_sf,
                        gs_h, dev_status, stream);
}

moe_status moe_requant(const void* h, int64_t capacity, int I, const int32_t* slot_token, const float* h_amax,
                       float* gs_h_out, uint8_t* h_fp4, uint8_t* h_sf, int32_t* dev_status, moe_stream_t stream) {
  if (!h || !slot_token || !h_amax || !gs_h_out || !h_fp4 || !h_sf || capacity < 0) return MOE_ERR_INVALID_ARG;
  if (I <= 0 || I % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(h, 16) || !aligned(h_fp4, 4) || !aligned(h_sf, 4)) return MOE_ERR_INVALID_ARG;
  return quantize_launch(3, h, capacity, I, I, reinterpret_cast<const uint32_t*>(h_amax), nullptr, gs_h_out, h_fp4,
                         h_sf, nullptr, 0, slot_token, capacity, dev_status, stream);
}

moe_status moe_grouped_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h, const int32_t* offsets,
                               const int32_t* padded_offsets, int E, int64_t capacity, int I, int K,
                               const uint8_t* w2_fp4, const uint8_t* w2_sf, const float* gs_w2, int epilogue,
                               void* y_rows, const int32_t* slot_token, const float* slot_weight, float* out32,
                               int64_t T, int32_t* dev_status, moe_stream_t stream) {
  if (!h_fp4 || !h_sf || !gs_h || !offsets || !padded_offsets || !w2_fp4 || !w2_sf || !gs_w2)
    return MOE_ERR_INVALID_ARG;
  if (!shape_ok(K, I, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (capacity <= 0 || capacity % kTileM || capacity > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!aligned(h_fp4, 16) || !aligned(w2_fp4, 16) || !aligned(h_sf, 16) || !aligned(w2_sf, 16))
    return MOE_ERR_INVALID_ARG;
  if (epilogue == MOE_L2_ROWS_BF16) {
    if (!y_rows || !aligned(y_rows, 16)) return MOE_ERR_INVALID_ARG;
  } else if (epilogue == MOE_L2_SCATTER) {
    if (!slot_token || !slot_weight || !out32 || T < 0 || !aligned(out32, 16)) return MOE_ERR_INVALID_ARG;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return launch_gemm_l2(h_fp4, h_sf, gs_h, offsets, padded_offsets, E, capacity, I, K, w2_fp4, w2_sf, gs_w2,
                        epilogue, y_rows, slot_token, slot_weight, out32, T, dev_status, stream);
}

moe_status moe_cast_output(const float* out32, void* out_bf16, int64_t T, int K, moe_stream_t stream) {
  return cast_output(out32, out_bf16, T, K, stream, false);
}

moe_status moe_combine_rows(const void* y_rows, int64_t ld_y, const int32_t* pair_slot, const float* topk_w, int64_t T,
                            int topk, int K, int64_t capacity, void* out_bf16, int32_t* dev_status,
                            moe_stream_t stream) {
  return combine_rows(y_rows, ld_y, pair_slot, topk_w, T, topk, K, capacity, out_bf16, dev_status, stream, false);
}

moe_status moe_forward(const void* x, int64_t T, int K, int I, int E, const int32_t* topk_ids, const float* topk_w,
                       int topk, int expert_offset, const moe_weights* w, const float* gs_x_fixed, int gs_h_mode,
                       float* gs_h, void* out, int32_t* dev_status, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  return moe_forward_traced(x, T, K, I, E, topk_ids, topk_w, topk, expert_offset, w, gs_x_fixed, gs_h_mode, gs_h,
                            out, dev_status, ws, ws_bytes, nullptr, stream);
}

moe_status moe_forward_traced(const void* x, int64_t T, int K, int I, int E, const int32_t* topk_ids,
                              const float* topk_w, int topk, int expert_offset, const moe_weights* w,
                              const float* gs_x_fixed, int gs_h_mode, float* gs_h, void* out, int32_t* dev_status,
                              void* ws, size_t ws_bytes, void* const* stage_events, moe_stream_t stream) {
  if (T < 0 || !w || !gs_h || !ws) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(K, I, E) || topk < 1 || topk > 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T > 0 && (!x || !topk_ids || !topk_w || !out)) return MOE_ERR_INVALID_ARG;
  if (gs_h_mode != MOE_GS_DYNAMIC && gs_h_mode != MOE_GS_FIXED) return MOE_ERR_INVALID_ARG;
  if (!w->w1_fp4 || !w->w1_sf || !w->gs_w1_gate || !w->gs_w1_up || !w->w2_fp4 || !w->w2_sf || !w->gs_w2)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < moe_workspace_size(T, K, I, E, topk)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;

  Carve c{reinterpret_cast<uint8_t*>(ws)};
  void* parts[15];
  forward_layout(c, T, K, I, E, topk, parts);
  const int64_t cap = moe_slot_capacity(T, topk, E);
  uint32_t* scal = reinterpret_cast<uint32_t*>(parts[0]);
  float* h_amax = reinterpret_cast<float*>(scal + 1);
  float* gs_x = reinterpret_cast<float*>(scal + 2);
  const size_t rhalf = moe_route_workspace_size(T, topk, E) / 2;
  int32_t* rcnt = reinterpret_cast<int32_t*>(parts[1]);
  int32_t* rbase = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(parts[1]) + rhalf);
  int32_t* counts = reinterpret_cast<int32_t*>(parts[2]);
  int32_t* offsets = reinterpret_cast<int32_t*>(parts[3]);
  int32_t* poff = reinterpret_cast<int32_t*>(parts[4]);
  int32_t* slot_token = reinterpret_cast<int32_t*>(parts[5]);
  float* slot_weight = reinterpret_cast<float*>(parts[6]);
  int32_t* pair_slot = reinterpret_cast<int32_t*>(parts[7]);
  uint8_t* a_fp4 = reinterpret_cast<uint8_t*>(parts[8]);
  uint8_t* a_sf = reinterpret_cast<uint8_t*>(parts[9]);
  void* h_bf16 = parts[10];
  uint8_t* h_fp4 = reinterpret_cast<uint8_t*>(parts[11]);
  uint8_t* h_sf = reinterpret_cast<uint8_t*>(parts[12]);
  float* out32 = reinterpret_cast<float*>(parts[13]);
  const bool combine = use_combine(T, K);  // parts[13] then holds the L2 rows [cap, K] BF16
  // the weight-streaming GEMMs' tile-claim counters (L1, L2), zeroed by the small-batch
  // prologue; larger batches walk static ranges (no counter)
  int32_t* claims = reinterpret_cast<int32_t*>(scal + 8);
  const bool small = T * topk <= kSmallRoutePairsMax;
  int32_t* claim_l1 = small ? claims : nullptr;
  int32_t* claim_l2 = small ? claims + 1 : nullptr;

  moe_status s;
  // Kernels after the first run as programmatic dependents of their predecessor (each
  // waits for it before touching its results, and may start early) unless stage
  // events are recorded between them (events 0 and 6 sit outside the kernel chain).
  bool pdl = true;
  for (int i = 1; stage_events && i < 6; ++i) pdl = pdl && stage_events[i] == nullptr;
  if (mark(stage_events, 0, stream) != MOE_OK) return MOE_ERR_CUDA;
  if (small) {
    // one launch: routing (block 0) + per-block amax of x + zeroing of out32 and of the
    // tile-claim counters
    uint32_t* partials = scal + 256;
    const int64_t vecs = T * (K / 8), n4 = T * K / 4;
    const int nb = (int)std::min<int64_t>(std::max<int64_t>(ceil_div(std::max(vecs, n4), 2048), 1), 256);
    PrologueArgs pa;
    pa.ids = topk_ids;
    pa.w = topk_w;
    pa.P = (int)(T * topk);
    pa.topk = topk;
    pa.E = E;
    pa.off = expert_offset;
    pa.counts = counts;
    pa.offsets = offsets;
    pa.padded_offsets = poff;
    pa.slot_token = slot_token;
    pa.slot_weight = slot_weight;
    pa.pair_slot = pair_slot;
    pa.capacity = cap;
    pa.status = dev_status;
    pa.x = reinterpret_cast<const uint4*>(x);
    pa.rows = T;
    pa.vec_per_row = K / 8;
    pa.ld_vec = K / 8;
    pa.amax_partials = gs_x_fixed ? nullptr : partials;
    pa.out32 = combine ? nullptr : out32;
    pa.out32_n4 = combine ? 0 : n4;
    pa.zero_words = claims;
    pa.n_zero_words = 2;
    pa.fill_padding = gs_h_mode == MOE_GS_DYNAMIC;
    if (launch_forward_prologue(pa, nb, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if ((s = mark(stage_events, 1, stream)) != MOE_OK) return s;
    // A programmatic dependent launched only once the prologue's amax blocks have exited
    // (launched beside them, its blocks were placed on the few SMs they left free and ran
    // several times slower).
    s = quantize_launch(2, x, T, K, K, nullptr, gs_x_fixed, gs_x, a_fp4, a_sf, pair_slot, topk, nullptr, cap,
                        dev_status, stream, gs_x_fixed ? nullptr : partials, nb, pdl);
  } else {
    if (!combine && cudaMemsetAsync(out32, 0, (size_t)T * K * sizeof(float), stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    s = route_impl(topk_ids, topk_w, T, topk, E, expert_offset, counts, offsets, poff, slot_token, slot_weight,
                   pair_slot, cap, rcnt, rbase, dev_status, stream);
    if (s != MOE_OK || (s = mark(stage_events, 1, stream)) != MOE_OK) return s;
    // the amax of x runs beside the routing (per-block partials, no zeroed word); the
    // quantiser reduces the partials
    uint32_t* partials = reinterpret_cast<uint32_t*>(parts[14]);
    int nparts = 0;
    if (!gs_x_fixed) {
      const int64_t vecs = T * (K / 8);
      if (vecs >= (int64_t(1) << 32)) return MOE_ERR_UNSUPPORTED_SHAPE;
      nparts = (int)std::min<int64_t>(std::max<int64_t>(ceil_div(vecs, 256 * 4), 1),
                                      std::min<int64_t>((int64_t)sm_count() * 8, kAmaxMaxBlocks));
      if (launch_amax(x, T, K, K, nullptr, nparts, stream, partials, pdl) != cudaSuccess) return MOE_ERR_CUDA;
    }
    s = quantize_launch(2, x, T, K, K, nullptr, gs_x_fixed, gs_x, a_fp4, a_sf, pair_slot, topk, nullptr, cap,
                        dev_status, stream, gs_x_fixed ? nullptr : partials, nparts, pdl);
  }
  if (s != MOE_OK || (s = mark(stage_events, 2, stream)) != MOE_OK) return s;
  if (gs_h_mode == MOE_GS_DYNAMIC) {
    s = launch_gemm_l1(a_fp4, a_sf, gs_x, offsets, poff, E, cap, K, I, w->w1_fp4, w->w1_sf, w->gs_w1_gate,
                       w->gs_w1_up, MOE_L1_SILU_BF16, h_bf16, h_amax, nullptr, nullptr, nullptr, dev_status, stream,
                       pdl, claim_l1);
    if (s != MOE_OK || (s = mark(stage_events, 3, stream)) != MOE_OK) return s;
    s = quantize_launch(3, h_bf16, cap, I, I, reinterpret_cast<const uint32_t*>(h_amax), nullptr, gs_h, h_fp4, h_sf,
                        nullptr, 0, slot_token, cap, dev_status, stream, nullptr, 0, pdl);
  } else {
    s = launch_gemm_l1(a_fp4, a_sf, gs_x, offsets, poff, E, cap, K, I, w->w1_fp4, w->w1_sf, w->gs_w1_gate,
                       w->gs_w1_up, MOE_L1_SILU_REQUANT, nullptr, nullptr, h_fp4, h_sf, gs_h, dev_status, stream,
                       pdl, claim_l1);
    if (s != MOE_OK || (s = mark(stage_events, 3, stream)) != MOE_OK) return s;
  }
  if (s != MOE_OK || (s = mark(stage_events, 4, stream)) != MOE_OK) return s;
  if (combine)
    s = launch_gemm_l2(h_fp4, h_sf, gs_h, offsets, poff, E, cap, I, K, w->w2_fp4, w->w2_sf, w->gs_w2,
                       MOE_L2_ROWS_BF16, parts[13], nullptr, nullptr, nullptr, T, dev_status, stream, pdl, claim_l2);
  else
    s = launch_gemm_l2(h_fp4, h_sf, gs_h, offsets, poff, E, cap, I, K, w->w2_fp4, w->w2_sf, w->gs_w2, MOE_L2_SCATTER,
                       nullptr, slot_token, slot_weight, out32, T, dev_status, stream, pdl, claim_l2);
  if (s != MOE_OK || (s = mark(stage_events, 5, stream)) != MOE_OK) return s;
  s = combine ? combine_rows(parts[13], K, pair_slot, topk_w, T, topk, K, cap, out, dev_status, stream, pdl,
                             true)  // the rows are this call's workspace: dead once combined
              : cast_output(out32, out, T, K, stream, pdl);
  if (s != MOE_OK) return s;
  return mark(stage_events, 6, stream);
}

}  // extern "C"
