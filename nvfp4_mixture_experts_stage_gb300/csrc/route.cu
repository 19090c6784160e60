// Token -> slot routing on the device, with no host synchronisation.
//
// Method: nvfp4-megamoe-kernel commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py
// ("global expert ids": subtract the rank's first expert id, drop foreign ids),
// of src ("1-D slot_expert_ids / slot_token"), of vllm/nvfp4_cutedsl.py ("CUDA
// graph" commits: sort pairs by expert, bincount + cumsum int32 offsets on the
// device, zero-weight padding) and of tests ("token layout": rows grouped
// [expert 0 | expert 1 | ...]).
//
// Large batches: one cooperative launch over chunks of 256 (token, k) pairs, one chunk
// per warp at a time, in three phases separated by grid-wide barriers:
//   count: warp-level histogram (__match_any_sync groups equal experts, the group
//          leader adds the group size) -> cnt[e][chunk];
//   scan:  per expert a warp-level prefix sum over chunks gives each chunk's first
//          rank; every block then scans the expert totals into offsets and 128-padded
//          offsets;
//   place: each warp walks its chunks again in order, ranks pairs within the 32-pair
//          group by popcount of the lower lanes of its match group, and writes
//          slot_token / slot_weight / pair_slot; the blocks fill the padding slots.
// Processing every chunk in order and every group in lane order makes the placement
// stable: slots of an expert follow ascending t*topk + j.  Small batches route in one
// block (route_small_kernel).
#include <algorithm>

#include <cooperative_groups.h>

#include "kernels.cuh"

namespace moe {

__device__ __forceinline__ int local_expert(const int32_t* ids, int64_t idx, int64_t P, int off, int E) {
  if (idx >= P) return -1;
  const int l = __ldg(ids + idx) - off;
  return (l >= 0 && l < E) ? l : -1;
}

namespace cg = cooperative_groups;

// Per-warp histogram of one chunk's local experts into hist[0..E) (shared memory).
__device__ __forceinline__ void chunk_histogram(const int32_t* __restrict__ ids, int64_t base, int64_t P, int off,
                                                int E, int* hist) {
  const int lane = threadIdx.x & 31;
  int loc[kRouteChunk / 32];
#pragma unroll
  for (int g = 0; g < kRouteChunk / 32; ++g) loc[g] = local_expert(ids, base + g * 32 + lane, P, off, E);
#pragma unroll
  for (int g = 0; g < kRouteChunk / 32; ++g) {
    const unsigned grp = __match_any_sync(0xFFFFFFFFu, loc[g]);
    if (loc[g] >= 0 && lane == __ffs(grp) - 1) hist[loc[g]] += __popc(grp);
    __syncwarp();
  }
}

// Launched cooperatively with blockDim kRouteWarps * 32 and a grid that fits on the GPU
// at once.  cnt, base: E * nchunks ints of scratch.
__global__ void __launch_bounds__(kRouteWarps * 32) route_fused_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t P, int topk, int E, int off,
    int32_t* __restrict__ cnt, int32_t* __restrict__ base, int nchunks, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets, int32_t* __restrict__ slot_token,
    float* __restrict__ slot_weight, int32_t* __restrict__ pair_slot, int64_t capacity, int32_t* status) {
  __shared__ int run[kRouteWarps][kMaxExperts];
  __shared__ int s_cnt[kMaxExperts], s_poff[kMaxExperts + 1];
  // the layer's next kernel (the amax of x) reads nothing routed and may start now
  griddep_launch_dependents();
  cg::grid_group grid = cg::this_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kRouteWarps + warp, nw = gridDim.x * kRouteWarps;

  // count
  for (int chunk = gw; chunk < nchunks; chunk += nw) {
    for (int e = lane; e < E; e += 32) run[warp][e] = 0;
    __syncwarp();
    chunk_histogram(ids, (int64_t)chunk * kRouteChunk, P, off, E, run[warp]);
    __syncwarp();
    for (int e = lane; e < E; e += 32) cnt[(int64_t)e * nchunks + chunk] = run[warp][e];
    __syncwarp();
  }
  grid.sync();

  // scan over chunks, per expert (256 chunk counts loaded together per round)
  for (int e = gw; e < E; e += nw) {
    int running = 0;
    const int32_t* row = cnt + (int64_t)e * nchunks;
    int32_t* brow = base + (int64_t)e * nchunks;
    for (int c0 = 0; c0 < nchunks; c0 += 256) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + 32 * i + lane;
        v[i] = c < nchunks ? __ldcg(row + c) : 0;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int incl = v[i];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
          if (lane >= d) incl += t;
        }
        const int c = c0 + 32 * i + lane;
        if (c < nchunks) brow[c] = running + incl - v[i];
        running += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
    }
    if (lane == 0) counts[e] = running;
  }
  grid.sync();

  // every block: the expert-level scan (offsets and 128-padded offsets)
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = __ldcg(counts + e);
  __syncthreads();
  if (warp == 0) {
    int rsum = 0, prun = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? s_cnt[e] : 0;
      const int pv = (v + kTileM - 1) / kTileM * kTileM;
      int incl = v, pincl = pv;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        const int pt = __shfl_up_sync(0xFFFFFFFFu, pincl, d);
        if (lane >= d) { incl += t; pincl += pt; }
      }
      if (e < E) {
        s_poff[e] = prun + pincl - pv;
        if (blockIdx.x == 0) {
          offsets[e] = rsum + incl - v;
          padded_offsets[e] = prun + pincl - pv;
        }
      }
      rsum += __shfl_sync(0xFFFFFFFFu, incl, 31);
      prun += __shfl_sync(0xFFFFFFFFu, pincl, 31);
    }
    if (lane == 0) {
      s_poff[E] = prun;
      if (blockIdx.x == 0) {
        offsets[E] = rsum;
        padded_offsets[E] = prun;
      }
    }
  }
  __syncthreads();

  // place
  const unsigned lower = (1u << lane) - 1u;
  for (int chunk = gw; chunk < nchunks; chunk += nw) {
    for (int e = lane; e < E; e += 32) run[warp][e] = s_poff[e] + __ldcg(base + (int64_t)e * nchunks + chunk);
    __syncwarp();
    const int64_t base_idx = (int64_t)chunk * kRouteChunk;
    int loc[kRouteChunk / 32];
    float wt[kRouteChunk / 32];
#pragma unroll
    for (int g = 0; g < kRouteChunk / 32; ++g) {
      const int64_t idx = base_idx + g * 32 + lane;
      loc[g] = local_expert(ids, idx, P, off, E);
      wt[g] = idx < P ? __ldg(w + idx) : 0.0f;
    }
#pragma unroll
    for (int g = 0; g < kRouteChunk / 32; ++g) {
      const int64_t idx = base_idx + g * 32 + lane;
      const int l = loc[g];
      const unsigned grp = __match_any_sync(0xFFFFFFFFu, l);
      int slot = -1;
      if (l >= 0) slot = run[warp][l] + __popc(grp & lower);
      __syncwarp();
      if (l >= 0 && lane == __ffs(grp) - 1) run[warp][l] += __popc(grp);
      __syncwarp();
      if (idx < P) {
        if (slot >= capacity) {
          set_status(status, MOE_ERR_DEVICE_INDEX);
          slot = -1;
        }
        pair_slot[idx] = slot;
        if (slot >= 0) {
          slot_token[slot] = (int32_t)(idx / topk);
          slot_weight[slot] = wt[g];
        }
      }
    }
    __syncwarp();
  }

  // padding slots: the tail of each expert's padded range, then everything past the last
  for (int e = gw; e < E; e += nw)
    for (int p = s_poff[e] + s_cnt[e] + lane; p < s_poff[e + 1] && p < capacity; p += 32) {
      slot_token[p] = -1;
      slot_weight[p] = 0.0f;
    }
  for (int64_t p = s_poff[E] + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < capacity;
       p += (int64_t)gridDim.x * blockDim.x) {
    slot_token[p] = -1;
    slot_weight[p] = 0.0f;
  }
}

// Whole routing in one block of 32 warps for up to kSmallRoutePairs pairs (decode
// batches): warp w owns the contiguous pairs [w*G*32, (w+1)*G*32) in groups of 32,
// counts them per expert, a per-expert scan over the 32 warps gives each warp its
// first rank, a scan over experts gives the offsets, then the warps place their
// pairs in order (stable) and the block fills the padding slots.
constexpr int kSmallRoutePairs = 8192;
constexpr int kSmallGroups = kSmallRoutePairs / (32 * 32);  // 32-pair groups per warp (max)

// One block of 1024 threads; wcnt: 32*E ints of shared memory.
__device__ __forceinline__ void route_small_block(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int P, int topk, int E, int off,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets,
    int32_t* __restrict__ slot_token, float* __restrict__ slot_weight, int32_t* __restrict__ pair_slot,
    int64_t capacity, int32_t* status, int* wcnt, bool fill_padding = true) {
  __shared__ int s_cnt[kMaxExperts], s_off[kMaxExperts + 1], s_poff[kMaxExperts + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (P + 1023) / 1024;  // groups per warp
  for (int i = threadIdx.x; i < 32 * E; i += 1024) wcnt[i] = 0;
  int loc[kSmallGroups];
  float wt[kSmallGroups];
#pragma unroll
  for (int g = 0; g < kSmallGroups; ++g) {
    const int idx = (warp * G + g) * 32 + lane;
    const bool in = g < G && idx < P;
    loc[g] = in ? local_expert(ids, idx, P, off, E) : -1;
    wt[g] = in ? __ldg(w + idx) : 0.0f;
  }
  __syncthreads();
  int* mine = wcnt + warp * E;
#pragma unroll
  for (int g = 0; g < kSmallGroups; ++g) {
    if (g >= G) break;
    const unsigned grp = __match_any_sync(0xFFFFFFFFu, loc[g]);
    if (loc[g] >= 0 && lane == __ffs(grp) - 1) mine[loc[g]] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();
  // per expert: exclusive scan over the 32 warps (warp-parallel over experts)
  for (int e = warp; e < E; e += 32) {
    const int v = wcnt[lane * E + e];
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += t;
    }
    wcnt[lane * E + e] = incl - v;
    if (lane == 31) s_cnt[e] = incl;
  }
  __syncthreads();
  if (warp == 0) {
    int run = 0, prun = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < E ? s_cnt[e] : 0;
      const int pv = (v + kTileM - 1) / kTileM * kTileM;
      int incl = v, pincl = pv;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        const int pt = __shfl_up_sync(0xFFFFFFFFu, pincl, d);
        if (lane >= d) { incl += t; pincl += pt; }
      }
      if (e < E) {
        s_off[e] = run + incl - v;
        s_poff[e] = prun + pincl - pv;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      prun += __shfl_sync(0xFFFFFFFFu, pincl, 31);
    }
    if (lane == 0) {
      s_off[E] = run;
      s_poff[E] = prun;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += 1024) {
    if (e < E) counts[e] = s_cnt[e];
    offsets[e] = s_off[e];
    padded_offsets[e] = s_poff[e];
  }
  // place: running slot of (warp, expert) = padded offset + ranks of earlier warps
  for (int e = lane; e < E; e += 32) mine[e] += s_poff[e];
  __syncwarp();
  const unsigned lower = (1u << lane) - 1u;
#pragma unroll
  for (int g = 0; g < kSmallGroups; ++g) {
    if (g >= G) break;
    const int idx = (warp * G + g) * 32 + lane;
    const int l = loc[g];
    const unsigned grp = __match_any_sync(0xFFFFFFFFu, l);
    int slot = -1;
    if (l >= 0) slot = mine[l] + __popc(grp & lower);
    __syncwarp();
    if (l >= 0 && lane == __ffs(grp) - 1) mine[l] += __popc(grp);
    __syncwarp();
    if (idx < P) {
      if (slot >= capacity) {
        set_status(status, MOE_ERR_DEVICE_INDEX);
        slot = -1;
      }
      pair_slot[idx] = slot;
      if (slot >= 0) {
        slot_token[slot] = idx / topk;
        slot_weight[slot] = wt[g];
      }
    }
  }
  // padding slots: the tail of each expert's padded range, then everything past the last
  if (!fill_padding) return;
  for (int e = warp; e < E; e += 32)
    for (int p = s_poff[e] + s_cnt[e] + lane; p < s_poff[e + 1] && p < capacity; p += 32) {
      slot_token[p] = -1;
      slot_weight[p] = 0.0f;
    }
  for (int64_t p = s_poff[E] + threadIdx.x; p < capacity; p += 1024) {
    slot_token[p] = -1;
    slot_weight[p] = 0.0f;
  }
}

__global__ void __launch_bounds__(1024) route_small_kernel(
    const int32_t* __restrict__ ids, const float* __restrict__ w, int P, int topk, int E, int off,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ padded_offsets,
    int32_t* __restrict__ slot_token, float* __restrict__ slot_weight, int32_t* __restrict__ pair_slot,
    int64_t capacity, int32_t* status) {
  extern __shared__ int sm[];
  route_small_block(ids, w, P, topk, E, off, counts, offsets, padded_offsets, slot_token, slot_weight, pair_slot,
                    capacity, status, sm);
}

// The start of the layer for small batches, in one launch: block 0 routes (as
// route_small_kernel) and zeroes the GEMMs' tile-claim counters; the other blocks take
// the per-block max |x| (written to amax_partials[block-1], no atomics, so nothing has
// to be cleared first) and zero the fp32 output accumulator.  Only block 0 triggers the
// dependent launch.
__global__ void __launch_bounds__(1024) forward_prologue_kernel(PrologueArgs a) {
  extern __shared__ int sm[];
  if (blockIdx.x == 0) {
    // The quantiser after this kernel is a programmatic dependent: it launches once this
    // block has passed here and every other block has exited (those blocks never
    // trigger), so its blocks spread over the SMs the amax blocks have left, and wait
    // for this block's routing tables in griddep_wait().
    griddep_launch_dependents();
    if (threadIdx.x < a.n_zero_words) a.zero_words[threadIdx.x] = 0;
    route_small_block(a.ids, a.w, a.P, a.topk, a.E, a.off, a.counts, a.offsets, a.padded_offsets, a.slot_token,
                      a.slot_weight, a.pair_slot, a.capacity, a.status, sm, a.fill_padding != 0);
    return;
  }
  const uint32_t nb = gridDim.x - 1, b = blockIdx.x - 1;
  const uint32_t stride = nb * blockDim.x;
  // zero out32 (float4 stores)
  float4* o = reinterpret_cast<float4*>(a.out32);
  for (int64_t i = (int64_t)b * blockDim.x + threadIdx.x; i < a.out32_n4; i += stride) o[i] = make_float4(0, 0, 0, 0);
  if (!a.amax_partials) return;
  // max |x| over this block's share of the 16-byte vectors
  const uint32_t vpr = (uint32_t)a.vec_per_row;
  const uint32_t total = (uint32_t)(a.rows * a.vec_per_row);
  uint32_t m = 0;
  for (uint32_t v = b * blockDim.x + threadIdx.x; v < total; v += stride) {
    const uint32_t r = v / vpr;
    const uint4 q = __ldg(a.x + (int64_t)r * a.ld_vec + (v - r * vpr));
    m = __vmaxu2(m, q.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, q.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, q.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, q.w & 0x7FFF7FFFu);
  }
  m = max(m & 0xFFFFu, m >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) a.amax_partials[b] = v << 16;  // bf16 magnitude -> fp32 bits
  }
}

cudaError_t launch_forward_prologue(const PrologueArgs& a, int amax_blocks, cudaStream_t st) {
  static PerDeviceOnce configured;
  cudaError_t e = configured.run([] {
    return cudaFuncSetAttribute(forward_prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                32 * kMaxExperts * (int)sizeof(int));
  });
  if (e != cudaSuccess) return e;
  forward_prologue_kernel<<<1 + amax_blocks, 1024, 32 * a.E * sizeof(int), st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_route(const int32_t* ids, const float* w, int64_t P, int topk, int E, int off, int32_t* cnt,
                         int32_t* base, int nchunks, int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                         int32_t* slot_token, float* slot_weight, int32_t* pair_slot, int64_t capacity,
                         int32_t* status, cudaStream_t st) {
  // one block up to 4096 pairs: above that its scattered slot stores (all from one SM)
  // take longer than the three launches of the chunked path (8192 pairs: 20 us against
  // ~12 us); the layer's fused prologue still routes up to 8192 pairs in its block 0
  if (P <= kSmallRoutePairs / 2) {
    static PerDeviceOnce configured;
    cudaError_t e = configured.run([] {
      return cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  32 * kMaxExperts * (int)sizeof(int));
    });
    if (e != cudaSuccess) return e;
    route_small_kernel<<<1, 1024, 32 * E * sizeof(int), st>>>(ids, w, (int)P, topk, E, off, counts, offsets,
                                                              padded_offsets, slot_token, slot_weight, pair_slot,
                                                              capacity, status);
    return cudaGetLastError();
  }
  // one cooperative launch: as many blocks as fit on the GPU at once (at most one per
  // group of kRouteWarps chunks)
  static PerDeviceInt resident;
  const int max_blocks = resident.get([] {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_fused_kernel, kRouteWarps * 32, 0) !=
            cudaSuccess ||
        per_sm < 1)
      return 0;
    return per_sm * sm_count_of_current_device();
  });
  if (max_blocks <= 0) return cudaErrorCooperativeLaunchTooLarge;
  const int blocks = std::max(1, std::min(max_blocks, (nchunks + kRouteWarps - 1) / kRouteWarps));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kRouteWarps * 32);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_fused_kernel, ids, w, P, topk, E, off, cnt, base, nchunks, counts, offsets,
                            padded_offsets, slot_token, slot_weight, pair_slot, capacity, status);
}

}  // namespace moe
