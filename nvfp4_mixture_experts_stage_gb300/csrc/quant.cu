// NVFP4 quantisation kernels: global amax, block quantisation (row-major,
// swizzled, into slot rows, or of masked slot rows), output cast and the
// one-time weight-scale rearrangement.
//
// Method: nvfp4-megamoe-kernel commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py
// ("three bugs fixed" commit: sign-magnitude E2M1 nibbles, scale = block_max/6;
// "global scale" commit: gs = amax/(6*448) normalises before blocking), commits of
// tests ("float4_e2m1fn_x2": two codes per byte along K) and of src (the
// scale-factor atom layout of the block-scaled MMA).
//
// Data movement: one warp owns a 256-element segment of a row per step; lane l
// holds elements [8l, 8l+8) as one 16-byte load, so lanes (2i, 2i+1) form the
// 16-element block i and the warp's loads and code stores are fully coalesced
// (512 B in, 128 B out).  Four consecutive block scales of a row are assembled
// into one 32-bit store by lane 8j (they are contiguous in both scale layouts).
#include <algorithm>

#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// max |x| over a BF16 matrix -> fp32 bits: atomically max-ed into *amax_bits (which must
// hold 0 or a previous non-negative value on entry), or, with partials, each block's
// maximum to partials[blockIdx.x] (no zeroed word needed).  It reads only x, so as a
// programmatic dependent it may run beside the kernel before it; it waits for that
// kernel only at its end, so a kernel waiting for this one also sees the one before.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint4* __restrict__ x, int64_t T,
                                                        int vec_per_row, int64_t ld_vec,
                                                        uint32_t* amax_bits, uint32_t* partials) {
  griddep_launch_dependents();
  // vector index v -> (row, column); 32-bit division (the host keeps T*vec_per_row < 2^32)
  const uint32_t total = (uint32_t)(T * vec_per_row);
  const uint32_t vpr = (uint32_t)vec_per_row;
  const uint32_t stride = gridDim.x * blockDim.x;
  auto addr = [&](uint32_t v) {
    const uint32_t r = v / vpr;
    return x + (int64_t)r * ld_vec + (v - r * vpr);
  };
  uint32_t m = 0;
  uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  // 4 independent loads in flight per thread
  for (; i + 3 * stride < total; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldg(addr(i + u * stride));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      m = __vmaxu2(m, v[u].x & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].y & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].z & 0x7FFF7FFFu);
      m = __vmaxu2(m, v[u].w & 0x7FFF7FFFu);
    }
  }
  for (; i < total; i += stride) {
    const uint4 v = __ldg(addr(i));
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
  }
  // bf16 magnitude bits order like the magnitudes (non-NaN inputs)
  m = max(m & 0xFFFFu, m >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) {
      if (partials)
        partials[blockIdx.x] = v << 16;  // bf16 -> fp32 bits
      else if (v)
        atomicMax(amax_bits, v << 16);
    }
  }
  griddep_wait();
}

// ---------------------------------------------------------------------------
// Block quantisation.
// ---------------------------------------------------------------------------
template <int DST>
__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a) {
  griddep_wait();  // everything read below comes from earlier kernels
  griddep_launch_dependents();
  // 1/decode(b) for every block-scale byte b (scales are non-negative and <= 448, so
  // b <= 0x7E; b = 0 gives 0): the same values the per-block reciprocal would give
  __shared__ float s_rb[128];
  if (threadIdx.x < 128) s_rb[threadIdx.x] = threadIdx.x ? __frcp_rn(e4m3_value(threadIdx.x)) : 0.0f;
  float amax_f = 0.0f;
  if (!a.gs_fixed) {
    if (a.amax_partials) {  // reduce the per-block maxima (non-negative: bits order like values)
      uint32_t m = 0;
      for (int i = threadIdx.x & 31; i < a.n_partials; i += 32) m = max(m, __ldg(a.amax_partials + i));
      amax_f = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, m));
    } else {
      amax_f = __uint_as_float(*a.amax_bits);
    }
  }
  const float gs = a.gs_fixed ? __ldg(a.gs_fixed) : __fdiv_rn(amax_f, kGsDivisor);
  const float rg = recip_global_scale(gs);
  if (a.gs_out && blockIdx.x == 0 && threadIdx.x == 0) *a.gs_out = gs;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  // segment s (256 elements of one row) -> (row, seg); a warp takes segments warp0,
  // warp0 + nwarps, ...: row and seg advance incrementally (no division in the loop)
  const uint32_t nseg = (uint32_t)((a.K + 255) >> 8);
  const uint32_t total = (uint32_t)(a.rows * nseg);
  const uint32_t warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t drow = nwarps / nseg, dseg = nwarps - drow * nseg;
  uint32_t cur_row = warp0 / nseg, cur_seg = warp0 - cur_row * nseg;
  const int k_sf = a.K >> 4;
  const int half_k = a.K >> 1;

  constexpr int U = 4;
  for (uint32_t base = warp0; base < total; base += nwarps * U) {
    uint4 v[U];
    int64_t row[U];
    int col[U];
    bool live[U];  // the segment belongs to a row that is quantised (warp-uniform)
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t s = base + u * nwarps;
      row[u] = cur_row;
      col[u] = (int)cur_seg * 256 + lane * 8;  // first element of this lane
      cur_row += drow;
      cur_seg += dseg;
      if (cur_seg >= nseg) { cur_seg -= nseg; ++cur_row; }
      live[u] = s < total;
      if (live[u] && DST == kDstMasked) live[u] = __ldg(a.slot_token + row[u]) >= 0;
      const bool ok = live[u] && col[u] < a.K;
      v[u] = ok ? __ldcs(a.x + row[u] * a.ld_vec + (col[u] >> 3)) : make_uint4(0, 0, 0, 0);
      if (!ok) col[u] = -1;
    }
    // slots of each segment's token, fetched up front so the loads overlap (top-k <= 8)
    int32_t ps[U][8];
    if (DST == kDstSlots && a.topk <= 8) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          ps[u][j] = (col[u] >= 0 && j < a.topk) ? __ldg(a.pair_slot + row[u] * a.topk + j) : -1;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!live[u]) continue;  // a padding row (masked) or past the end: the whole warp skips it
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) { f[2 * i] = bf16lo(w[i]); f[2 * i + 1] = bf16hi(w[i]); }
      float m = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
      const float bm = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      const uint32_t sb = e4m3_byte(__fdiv_rn(__fmul_rn(bm, rg), 6.0f));
      const float rb = s_rb[sb];
      // (x*rg)*rb is sign(x) * ((|x|*rg)*rb) exactly, and the E2M1 conversion rounds
      // the magnitude and keeps the sign (also of a value that rounds to zero)
      uint32_t code = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        code |= e2m1x2(__fmul_rn(__fmul_rn(f[2 * i], rg), rb), __fmul_rn(__fmul_rn(f[2 * i + 1], rg), rb)) << (8 * i);
      // scale word of 4 blocks, assembled on lane 8j from lanes 8j, 8j+2, 8j+4, 8j+6
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
      const uint32_t sfw = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
      if (col[u] < 0) continue;
      const bool sf_lane = (lane & 7) == 0;
      const int ks = col[u] >> 4;  // scale column of this lane's block
      if (DST == kDstSlots) {
        auto put = [&](int32_t p) {
          if (p < 0) return;
          if (p >= a.capacity) { set_status(a.status, MOE_ERR_DEVICE_INDEX); return; }
          *reinterpret_cast<uint32_t*>(a.codes + (int64_t)p * half_k + (col[u] >> 1)) = code;
          if (sf_lane) *reinterpret_cast<uint32_t*>(a.sf + sf_swizzle_offset(p, ks, k_sf)) = sfw;
        };
        if (a.topk <= 8) {
#pragma unroll
          for (int j = 0; j < 8; ++j) put(ps[u][j]);
        } else {
          for (int j = 0; j < a.topk; ++j) put(__ldg(a.pair_slot + row[u] * a.topk + j));
        }
      } else {
        *reinterpret_cast<uint32_t*>(a.codes + row[u] * half_k + (col[u] >> 1)) = code;
        if (sf_lane) {
          const int64_t off = (DST == kDstRowMajorSf) ? row[u] * k_sf + ks
                                                      : sf_swizzle_offset(row[u], ks, k_sf);
          *reinterpret_cast<uint32_t*>(a.sf + off) = sfw;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Block quantisation of token rows into their slots (top-k <= 8): a warp takes a run of
// 1024 consecutive elements of one token row; lane l holds elements [32l, 32l+32) (two
// whole 16-element blocks, so no block maximum crosses lanes) and writes their 16 code
// bytes with one 16-byte store per slot; lanes 2m and 2m+1 together hold the four block
// scales of one scale word, which lane 2m stores.  The token's slots are looked up once
// per run (lane j holds slot j) with each slot's code-row and scale-atom offsets.  The
// arithmetic of every element is the one of quantize_kernel.
// ---------------------------------------------------------------------------
constexpr int kRunElems = 1024;

__global__ void __launch_bounds__(256, 4) quantize_slots_kernel(QuantArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float s_rb[128];
  if (threadIdx.x < 128) s_rb[threadIdx.x] = threadIdx.x ? __frcp_rn(e4m3_value(threadIdx.x)) : 0.0f;
  float amax_f = 0.0f;
  if (!a.gs_fixed) {
    if (a.amax_partials) {
      uint32_t m = 0;
      for (int i = threadIdx.x & 31; i < a.n_partials; i += 32) m = max(m, __ldg(a.amax_partials + i));
      amax_f = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, m));
    } else {
      amax_f = __uint_as_float(*a.amax_bits);
    }
  }
  const float gs = a.gs_fixed ? __ldg(a.gs_fixed) : __fdiv_rn(amax_f, kGsDivisor);
  const float rg = recip_global_scale(gs);
  if (a.gs_out && blockIdx.x == 0 && threadIdx.x == 0) *a.gs_out = gs;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const uint32_t nrun = (uint32_t)((a.K + kRunElems - 1) / kRunElems);
  const uint32_t total = (uint32_t)(a.rows * nrun);
  const uint32_t warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  const uint32_t drow = nwarps / nrun, drun = nwarps - drow * nrun;
  uint32_t cur_row = warp0 / nrun, cur_run = warp0 - cur_row * nrun;
  const int k_sf = a.K >> 4;
  const int half_k = a.K >> 1;
  const int atom_row = (k_sf >> 2) * 512;  // bytes of scale atoms per 128 slot rows

  for (uint32_t t = warp0; t < total; t += nwarps) {
    const int64_t row = cur_row;
    const int col = (int)cur_run * kRunElems + lane * 32;  // first element of this lane
    cur_row += drow;
    cur_run += drun;
    if (cur_run >= nrun) { cur_run -= nrun; ++cur_row; }
    // K is a multiple of 64, so a lane's 32 elements are all inside the row or all past it
    const bool in = col < a.K;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = in ? __ldcs(a.x + row * a.ld_vec + (col >> 3) + i) : make_uint4(0, 0, 0, 0);
    int32_t pj = lane < a.topk ? __ldg(a.pair_slot + row * a.topk + lane) : -1;
    if (pj >= a.capacity) {
      set_status(a.status, MOE_ERR_DEVICE_INDEX);
      pj = -1;
    }
    // slot j's code row and scale-atom position (scale column 0); the launcher keeps
    // capacity * K / 2 below 2^31, so 32-bit offsets hold them
    int32_t cbase[8];
    int32_t sbase[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int32_t p = __shfl_sync(0xFFFFFFFFu, pj, j);
      cbase[j] = p >= 0 ? p * half_k : -1;
      sbase[j] = (p >> 7) * atom_row + (p & 31) * 16 + ((p >> 5) & 3) * 4;
    }
    // two blocks of 16: codes and scale bytes
    uint32_t code[4];
    uint32_t sb2 = 0;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float f[16];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 q = v[2 * b + i];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { f[8 * i + 2 * k] = bf16lo(w[k]); f[8 * i + 2 * k + 1] = bf16hi(w[k]); }
      }
      float bm = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(f[i]));
      const uint32_t sb = e4m3_byte(__fdiv_rn(__fmul_rn(bm, rg), 6.0f));
      const float rb = s_rb[sb];
      sb2 |= sb << (8 * b);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t c = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          c |= e2m1x2(__fmul_rn(__fmul_rn(f[8 * h + 2 * i], rg), rb), __fmul_rn(__fmul_rn(f[8 * h + 2 * i + 1], rg), rb))
               << (8 * i);
        code[2 * b + h] = c;
      }
    }
    // scale word of blocks 4m..4m+3 on lane 2m: its two bytes, then lane 2m+1's two
    const uint32_t sfw = sb2 | (__shfl_down_sync(0xFFFFFFFFu, sb2, 1) << 16);
    if (!in) continue;
    const bool sf_lane = (lane & 1) == 0;
    const int ks = col >> 4;  // scale column of this lane's first block (a multiple of 4 on sf lanes)
    const int soff = (ks >> 2) * 512;
    const uint4 cw = make_uint4(code[0], code[1], code[2], code[3]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (cbase[j] < 0) continue;
      *reinterpret_cast<uint4*>(a.codes + (uint32_t)(cbase[j] + (col >> 1))) = cw;
      if (sf_lane) *reinterpret_cast<uint32_t*>(a.sf + (uint32_t)(sbase[j] + soff)) = sfw;
    }
  }
}

// ---------------------------------------------------------------------------
// Gate/up scale fold (set-up): the half of each expert's W1 with the smaller global
// scale g gets its block scales multiplied by g / max(gate, up) and re-rounded to UE4M3.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) fold_gate_up_kernel(uint8_t* __restrict__ sf, const float* __restrict__ gg,
                                                           const float* __restrict__ gu, float* __restrict__ common,
                                                           int E, int64_t half_bytes) {
  const int64_t n = (int64_t)E * 2 * half_bytes;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t e = i / (2 * half_bytes);
    const bool up = ((i / half_bytes) & 1) != 0;
    const float g_gate = __ldg(gg + e), g_up = __ldg(gu + e);
    const float c = fmaxf(g_gate, g_up);
    const float g = up ? g_up : g_gate;
    if (g == c || c == 0.0f) continue;
    const float ratio = __fdiv_rn(g, c);
    sf[i] = (uint8_t)e4m3_byte(__fmul_rn(e4m3_value(sf[i]), ratio));
  }
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride)
    common[e] = fmaxf(__ldg(gg + e), __ldg(gu + e));
}

cudaError_t launch_fold_gate_up(uint8_t* sf, const float* gg, const float* gu, float* common, int E, int I, int K,
                                cudaStream_t st) {
  const int64_t half_bytes = (int64_t)I * (K / 16);
  const int64_t n = (int64_t)E * 2 * half_bytes;
  const int blocks = (int)std::min<int64_t>(std::max<int64_t>((n + 255) / 256, 1), 4096);
  fold_gate_up_kernel<<<blocks, 256, 0, st>>>(sf, gg, gu, common, E, half_bytes);
  return cudaGetLastError();
}

cudaError_t launch_quantize(int dst, const QuantArgs& a, int blocks, cudaStream_t st, bool pdl) {
  // the run kernel stores 16 code bytes at a time: it needs a 16-byte aligned code buffer
  // (the API asks for 4); 32-bit offsets need capacity * K / 2 < 2^31
  if (dst == kDstSlots && a.topk <= 8 && a.capacity * (int64_t)(a.K / 2) < (int64_t(1) << 31) &&
      (reinterpret_cast<uintptr_t>(a.codes) & 15) == 0) {
    // tasks of kRunElems elements; four 256-thread blocks fit per SM
    const int64_t tasks = a.rows * (int64_t)((a.K + kRunElems - 1) / kRunElems);
    const int sms = sm_count_of_current_device();
    const int b = (int)std::min<int64_t>(std::max<int64_t>((tasks + 7) / 8, 1), (int64_t)sms * 4);
    (void)blocks;
    return launch_ex(quantize_slots_kernel, b, 256, 0, st, pdl, a);
  }
  switch (dst) {
    case kDstRowMajorSf: return launch_ex(quantize_kernel<kDstRowMajorSf>, blocks, 256, 0, st, pdl, a);
    case kDstSwizzledSf: return launch_ex(quantize_kernel<kDstSwizzledSf>, blocks, 256, 0, st, pdl, a);
    case kDstSlots: return launch_ex(quantize_kernel<kDstSlots>, blocks, 256, 0, st, pdl, a);
    default: return launch_ex(quantize_kernel<kDstMasked>, blocks, 256, 0, st, pdl, a);
  }
}

cudaError_t launch_amax(const void* x, int64_t rows, int K, int64_t ld_x, uint32_t* amax_bits, int blocks,
                        cudaStream_t st, uint32_t* partials, bool pdl) {
  return launch_ex(amax_bf16_kernel, blocks, 256, 0, st, pdl, reinterpret_cast<const uint4*>(x), rows, K / 8, ld_x / 8,
                   amax_bits, partials);
}

// ---------------------------------------------------------------------------
// out_bf16 = bf16(out32), 8 elements per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cast_f32_bf16_kernel(const float4* __restrict__ in,
                                                            uint4* __restrict__ out, int64_t n8) {
  griddep_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const float4 a = __ldcs(in + 2 * i), b = __ldcs(in + 2 * i + 1);
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    __stcs(out + i, o);
  }
}

// ---------------------------------------------------------------------------
// Weight scales [E, N, K_sf] row-major -> the GEMM's layout (setup only).
// gateup: logical row r of W1 (gate 0..I-1, up I..2I-1) goes to row
// 128*(r'/64) + (r'%64) (+64 for up), r' = r mod I, so each 128-row atom
// holds 64 gate rows then the matching 64 up rows.
// ---------------------------------------------------------------------------
__global__ void prepare_weight_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                         int E, int N, int k_sf, int gateup) {
  const int64_t per = (int64_t)N * k_sf;
  const int64_t total = (int64_t)E * per;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int I = N / 2;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t e = i / per;
    const int64_t rem = i - e * per;
    const int r = (int)(rem / k_sf);
    const int k = (int)(rem - (int64_t)r * k_sf);
    int m = r;
    if (gateup) {
      const int up = r >= I;
      const int rr = up ? r - I : r;
      m = (rr >> 6) * 128 + up * 64 + (rr & 63);
    }
    dst[e * per + sf_swizzle_offset(m, k, k_sf)] = src[i];
  }
}

// ---------------------------------------------------------------------------
// out[t] = bf16(sum_j w[t, j] * y[pair_slot[t, j]]) over j ascending, in fp32 (each
// product and each sum rounded), pairs with slot -1 skipped; 8 columns per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_rows_kernel(const uint4* __restrict__ y, int64_t ld_vec,
                                                           const int32_t* __restrict__ pair_slot,
                                                           const float* __restrict__ w, int topk, int64_t T,
                                                           int vec_per_row, int64_t capacity, uint4* __restrict__ out,
                                                           int32_t* status, bool discard_rows) {
  griddep_wait();
  const int64_t total = T * vec_per_row;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int64_t t = i / vec_per_row;
    const int64_t v = i - t * vec_per_row;
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
    auto add = [&](float wj, const uint4& q) {
      const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[2 * c] = __fadd_rn(acc[2 * c], __fmul_rn(wj, bf16lo(qw[c])));
        acc[2 * c + 1] = __fadd_rn(acc[2 * c + 1], __fmul_rn(wj, bf16hi(qw[c])));
      }
    };
    if (topk <= 8) {
      // the token's slots, then all its rows' loads in flight together; summed in pair order
      int32_t sj[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) sj[j] = j < topk ? __ldg(pair_slot + t * topk + j) : -1;
      float wj[8];
      uint4 q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (sj[j] >= capacity) {
          set_status(status, MOE_ERR_DEVICE_INDEX);
          sj[j] = -1;
        }
        wj[j] = sj[j] >= 0 ? __ldg(w + t * topk + j) : 0.0f;
        q[j] = sj[j] >= 0 ? __ldcs(y + (int64_t)sj[j] * ld_vec + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (sj[j] >= 0) add(wj[j], q[j]);
      // rows that are dead once read (the layer's own): drop their lines from L2 without
      // writing them back (the last rows the down GEMM wrote are still dirty there); one
      // lane per 128 bytes (the launcher asks for it only with 128-byte aligned rows)
      if (discard_rows && (v & 7) == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (sj[j] >= 0)
            asm volatile("discard.global.L2 [%0], 128;" ::"l"(y + (int64_t)sj[j] * ld_vec + v) : "memory");
      }
    } else {
      for (int j = 0; j < topk; ++j) {
        const int32_t s = __ldg(pair_slot + t * topk + j);
        if (s < 0) continue;
        if (s >= capacity) {
          set_status(status, MOE_ERR_DEVICE_INDEX);
          continue;
        }
        add(__ldg(w + t * topk + j), __ldg(y + (int64_t)s * ld_vec + v));
      }
    }
    __stcs(out + i, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
  }
}

cudaError_t launch_combine(const void* y, int64_t ld_y, const int32_t* pair_slot, const float* w, int topk, int64_t T,
                           int K, int64_t capacity, void* out, int32_t* status, int blocks, cudaStream_t st,
                           bool pdl, bool discard_rows) {
  // no more blocks than are resident at once: a second wave of blocks would start only
  // as the first ones leave (the loop inside is grid-strided)
  static PerDeviceInt resident;
  const int max_blocks = resident.get([] {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_rows_kernel, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    return per_sm * sm_count_of_current_device();
  });
  blocks = std::max(1, std::min(blocks, max_blocks));
  return launch_ex(combine_rows_kernel, blocks, 256, 0, st, pdl, reinterpret_cast<const uint4*>(y), ld_y / 8,
                   pair_slot, w, topk, T, K / 8, capacity, reinterpret_cast<uint4*>(out), status,
                   discard_rows && ld_y % 64 == 0 && (reinterpret_cast<uintptr_t>(y) & 127) == 0);
}

cudaError_t launch_cast(const float* in, void* out, int64_t n8, int blocks, cudaStream_t st, bool pdl) {
  return launch_ex(cast_f32_bf16_kernel, blocks, 256, 0, st, pdl, reinterpret_cast<const float4*>(in),
                   reinterpret_cast<uint4*>(out), n8);
}

cudaError_t launch_prepare_weight_sf(const uint8_t* src, uint8_t* dst, int E, int N, int k_sf, int gateup,
                                     int blocks, cudaStream_t st) {
  prepare_weight_sf_kernel<<<blocks, 256, 0, st>>>(src, dst, E, N, k_sf, gateup);
  return cudaGetLastError();
}

}  // namespace moe
