// Declarations shared between the kernel translation units and the C ABI layer.
#pragma once

#include "common.cuh"

namespace moe {

// ---- quant.cu ----
enum QuantDst : int {
  kDstRowMajorSf = 0,  // codes [rows, K/2], scales [rows, K/16]
  kDstSwizzledSf = 1,  // codes [rows, K/2], scales swizzled
  kDstSlots = 2,       // row t -> slots pair_slot[t*topk + j] (swizzled scales)
  kDstMasked = 3,      // row r written iff slot_token[r] >= 0 (swizzled scales)
};

struct QuantArgs {
  const uint4* x;             // rows of bf16, 16-byte vectors
  int64_t rows;
  int K;                      // elements per row (multiple of 64)
  int64_t ld_vec;             // row stride in 16-byte vectors
  const uint32_t* amax_bits;  // dynamic: fp32 bits of max|x|  (or NULL)
  const uint32_t* amax_partials;  // dynamic: per-block maxima (fp32 bits) to reduce (or NULL)
  int n_partials;
  const float* gs_fixed;      // fixed global scale (or NULL)
  float* gs_out;              // written by one thread (or NULL)
  uint8_t* codes;
  uint8_t* sf;
  const int32_t* pair_slot;   // kDstSlots
  int topk;
  const int32_t* slot_token;  // kDstMasked
  int64_t capacity;           // kDstSlots: bound on slot indices
  int32_t* status;
};

// Host launchers (each translation unit launches its own kernels).
// partials: each block's maximum to partials[blockIdx.x] instead of an atomic max into
// *amax_bits; pdl: a programmatic dependent of the previous kernel (see amax_bf16_kernel).
cudaError_t launch_amax(const void* x, int64_t rows, int K, int64_t ld_x, uint32_t* amax_bits, int blocks,
                        cudaStream_t st, uint32_t* partials = nullptr, bool pdl = false);
// pdl: launched as a programmatic dependent of the previous kernel in the stream
// (only where that kernel and everything before it is known; see moe_forward).
cudaError_t launch_quantize(int dst, const QuantArgs& a, int blocks, cudaStream_t st, bool pdl = false);
cudaError_t launch_cast(const float* in, void* out, int64_t n8, int blocks, cudaStream_t st, bool pdl = false);
cudaError_t launch_combine(const void* y, int64_t ld_y, const int32_t* pair_slot, const float* w, int topk, int64_t T,
                           int K, int64_t capacity, void* out, int32_t* status, int blocks, cudaStream_t st,
                           bool pdl = false, bool discard_rows = false);
cudaError_t launch_prepare_weight_sf(const uint8_t* src, uint8_t* dst, int E, int N, int k_sf, int gateup,
                                     int blocks, cudaStream_t st);

// ---- route.cu ----
constexpr int kRouteChunk = 256;  // pairs per warp
constexpr int kRouteWarps = 8;    // warps per block (count / place)
constexpr int kMaxExperts = 256;

// Routes the pairs and initialises every slot of [0, capacity) (padding: token -1,
// weight 0); one single-block kernel up to 8192 pairs, count/scan/place above.
cudaError_t launch_route(const int32_t* ids, const float* w, int64_t P, int topk, int E, int off, int32_t* cnt,
                         int32_t* base, int nchunks, int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                         int32_t* slot_token, float* slot_weight, int32_t* pair_slot, int64_t capacity,
                         int32_t* status, cudaStream_t st);

// Small-batch start of the layer: routing + amax partials + zeroing out32, one launch.
constexpr int kSmallRoutePairsMax = 8192;
struct PrologueArgs {
  const int32_t* ids;
  const float* w;
  int P, topk, E, off;
  int32_t* counts;
  int32_t* offsets;
  int32_t* padded_offsets;
  int32_t* slot_token;
  float* slot_weight;
  int32_t* pair_slot;
  int64_t capacity;
  int32_t* status;
  const uint4* x;            // activations (16-byte vectors)
  int64_t rows;
  int vec_per_row;
  int64_t ld_vec;
  uint32_t* amax_partials;   // [amax_blocks] fp32 bits, or NULL (fixed global scale)
  float* out32;
  int64_t out32_n4;          // float4 count to zero
  int32_t* zero_words;       // words block 0 zeroes (the GEMMs' tile-claim counters), or NULL
  int n_zero_words;
  int fill_padding;          // write slot_token -1 / slot_weight 0 into the padding slots (only the
                             // masked requantisation of h reads them; the GEMMs stop at each
                             // expert's slot count)
};
cudaError_t launch_forward_prologue(const PrologueArgs& a, int amax_blocks, cudaStream_t st);

// ---- gemm.cu ----
moe_status launch_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a, const int32_t* offsets,
                          const int32_t* padded_offsets, int E, int64_t cap, int K, int I, const uint8_t* w1_fp4,
                          const uint8_t* w1_sf, const float* gs_g, const float* gs_u, int epilogue, void* out_bf16,
                          float* h_amax, uint8_t* h_fp4, uint8_t* h_sf, const float* gs_h, int32_t* status,
                          cudaStream_t st, bool pdl = false, int32_t* tile_claim = nullptr);
moe_status launch_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h, const int32_t* offsets,
                          const int32_t* padded_offsets, int E, int64_t cap, int I, int K, const uint8_t* w2_fp4,
                          const uint8_t* w2_sf, const float* gs_w2, int epilogue, void* y_rows,
                          const int32_t* slot_token, const float* slot_weight, float* out32, int64_t T,
                          int32_t* status, cudaStream_t st, bool pdl = false, int32_t* tile_claim = nullptr);

// ---- gemm_stream.cu (weight-streaming kernel for small per-expert slot counts) ----
bool stream_gemm_supported(int Kred);
moe_status launch_stream_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a, const int32_t* offsets,
                                 const int32_t* padded_offsets, int E, int64_t cap, int K, int I,
                                 const uint8_t* w1_fp4, const uint8_t* w1_sf, const float* gs_g, const float* gs_u,
                                 int epilogue, void* out_bf16, float* h_amax, uint8_t* h_fp4, uint8_t* h_sf,
                                 const float* gs_h, int32_t* status, cudaStream_t st, bool pdl = false,
                                 int32_t* tile_claim = nullptr);
moe_status launch_stream_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h, const int32_t* offsets,
                                 const int32_t* padded_offsets, int E, int64_t cap, int I, int K,
                                 const uint8_t* w2_fp4, const uint8_t* w2_sf, const float* gs_w2, int epilogue,
                                 void* y_rows, const int32_t* slot_token, const float* slot_weight, float* out32,
                                 int64_t T, int32_t* status, cudaStream_t st, bool pdl = false,
                                 int32_t* tile_claim = nullptr);

// Gate/up scale fold (set-up, quant.cu).
cudaError_t launch_fold_gate_up(uint8_t* sf, const float* gg, const float* gu, float* common, int E, int I, int K,
                                cudaStream_t st);

// Bounded-wait self-test (selftest.cu).
moe_status selftest_bounded_wait(int32_t* status, int32_t* result, cudaStream_t st);
moe_status selftest_codecs(uint32_t first, int64_t n, uint8_t* e2m1, uint8_t* e4m3, cudaStream_t st);
moe_status selftest_silu(const float* g, int64_t n, float* s, cudaStream_t st);

// Which grouped-GEMM kernel runs (process-wide; moe_set_gemm_policy).
int gemm_policy();
int set_gemm_policy(int policy);
bool use_stream_gemm(int64_t cap, int E, int Kred);
int stream_chunk(int64_t cap, int E);

}  // namespace moe
