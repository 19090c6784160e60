// Parts shared by the two tiled grouped-GEMM kernels (gemm.cu: one CTA per 128-row
// tile; gemm_pair.cu: a CTA pair per 256-row tile): parameters, the on-device tile
// table, and the accumulator epilogue (alpha, BF16 rounding, SiLU * up, requantise,
// BF16 rows or weighted scatter).
//
// Method: nvfp4-megamoe-kernel commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py
// ("global scale as alpha"), of vllm/nvfp4_cutedsl.py ("intermediate_size": gate | up
// split at I) and of tests ("complete pipeline": SiLU(gate)*up in BF16, requantise,
// weighted scatter).
#pragma once

#include "tcgen05.cuh"

namespace moe {

constexpr int kBM = 128;
constexpr int kBKBytes = 128;               // 256 fp4 per row per stage
constexpr int kGemmThreads = 384;
constexpr int kEpiWarps = 8;
constexpr int kTmemCols = 512;

enum GemmKind : int { kL1GateUp = 0, kL1Silu = 1, kL1Requant = 2, kL2Rows = 3, kL2Scatter = 4 };

struct GemmParams {
  const uint8_t* a_sf;              // swizzled [cap/128][Kred/64][512]
  const uint8_t* b_sf;              // prepared [E][rows_per_expert/128][Kred/64][512]
  const int32_t* offsets;           // [E+1]
  const int32_t* padded_offsets;    // [E+1]
  int E;
  int Kred;                         // contraction length in elements
  int n_tiles;                      // output tiles per expert
  int b_rows;                       // weight rows per expert
  int I;                            // L1: columns of gate (= of up)
  const float* gs_a;
  const float* gs_b0;               // L1 gate / L2 down
  const float* gs_b1;               // L1 up
  void* out_bf16;
  int64_t out_ld;                   // elements per output row
  float* h_amax;
  uint8_t* h_fp4;
  uint8_t* h_sf;
  const float* gs_h;
  const int32_t* slot_token;
  const float* slot_weight;
  float* out32;
  int64_t T;
  int out_cols;                     // L2: K
  int64_t cap;                      // slot rows of A (bound for the offsets)
  int32_t* status;
};

// Tile table in shared memory (fields poff[E+1], cnt[E], cum[E+1], bad_offsets of S):
// padded offsets and counts of every expert, checked once (monotone, 128-aligned,
// counts within their padded ranges, inside the slot capacity), and the exclusive scan
// of tiles per expert = ceil(m-tiles / rows_per_tile) * n-tiles.  Called by every
// thread of the block; ends with the table visible to all of them.
template <class S>
MOE_DEV void build_tile_table(S& s, const GemmParams& p, int m_tiles_per_tile) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) s.bad_offsets = 0;
  __syncthreads();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s.poff[i] = p.padded_offsets[i];
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) s.cnt[i] = p.offsets[i + 1] - p.offsets[i];
  __syncthreads();
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) {
    const int lo = s.poff[i], hi = s.poff[i + 1], c = s.cnt[i];
    if (lo < 0 || hi < lo || (lo & 127) || (hi & 127) || c < 0 || c > hi - lo || hi > p.cap)
      s.bad_offsets = 1;
  }
  if (warp == 0) {
    int run = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      const int mt = e < p.E ? max(s.poff[e + 1] - s.poff[e], 0) >> 7 : 0;
      const int v = (mt + m_tiles_per_tile - 1) / m_tiles_per_tile * p.n_tiles;
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += t;
      }
      if (e < p.E) s.cum[e] = run + incl - v;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) s.cum[p.E] = run;
  }
  __syncthreads();
}

// Tile t -> (expert, n-tile, m-tile group); e advances monotonically with t.  A tile
// covers m_tiles_per_tile consecutive 128-row m-tiles of one expert, m fastest.
struct TileCursor {
  int e = 0;
  template <class S>
  MOE_DEV bool locate(const S& s, int E, int m_tiles_per_tile, int t, int& n, int& m) {
    while (e < E && t >= s.cum[e + 1]) ++e;
    if (e >= E) return false;
    const int local = t - s.cum[e];
    const int mt = (((s.poff[e + 1] - s.poff[e]) >> 7) + m_tiles_per_tile - 1) / m_tiles_per_tile;
    n = local / mt;
    m = local - n * mt;
    return true;
  }
};

// This warp's half of a 128 x BN accumulator tile into registers (TMEM lane quarter
// of taddr).  L1: the gate values then the matching up values of BN/4 h columns;
// L2: BN/2 consecutive output columns.
template <int KIND, int BN>
MOE_DEV void epilogue_load(uint32_t taddr, int half, float (&v)[BN / 2]) {
  constexpr bool kL1 = KIND <= kL1Requant;
  constexpr int kCols = BN / 2;
  if constexpr (kL1) {
    // BN 256: half h = prepared block h (gate at 128h, up at 128h + 64), 64 columns each;
    // BN 128: half h = gate columns 32h.., up columns 64 + 32h..
    constexpr int G = kCols / 2;
    const uint32_t g0 = BN == 256 ? 128 * half : 32 * half;
    if constexpr (G == 64) {  // gate columns g0.. then up columns g0 + 64..: one 128-column load
      tmem_ld128(taddr + g0, *reinterpret_cast<float(*)[128]>(&v[0]));
    } else {
#pragma unroll
      for (int j = 0; j < G; j += 16) {
        tmem_ld16(taddr + g0 + j, *reinterpret_cast<float(*)[16]>(&v[j]));
        tmem_ld16(taddr + g0 + 64 + j, *reinterpret_cast<float(*)[16]>(&v[G + j]));
      }
    }
  } else {
    if constexpr (kCols == 128) {
      tmem_ld128(taddr + half * kCols, *reinterpret_cast<float(*)[128]>(&v[0]));
    } else if constexpr (kCols % 64 == 0) {
#pragma unroll
      for (int j = 0; j < kCols; j += 64)
        tmem_ld64(taddr + half * kCols + j, *reinterpret_cast<float(*)[64]>(&v[j]));
    } else {
#pragma unroll
      for (int j = 0; j < kCols; j += 16)
        tmem_ld16(taddr + half * kCols + j, *reinterpret_cast<float(*)[16]>(&v[j]));
    }
  }
}

// The epilogue math of this thread's row (slot row prow of expert e, n-tile n) for the
// accumulator half in v.  valid = the row holds a routed pair (padding rows compute but
// store nothing).  amax collects max |h| of valid rows (L1 SiLU with a dynamic scale).
// The accumulator is already released when this runs, so it overlaps the next tile's
// MMAs; gap_ns > 0 spreads the work over that time (a sleep between 16-column chunks):
// issued in one burst, the epilogue's instructions and stores slow the MMA thread, the
// producer and the copiers that share the SM's sub-partitions (measured on prefill: L2
// 4 % faster with 360 ns gaps, L1 2 % with 300 ns; gaps that make the epilogue longer
// than a tile cost far more).
template <int KIND, int BN>
MOE_DEV void epilogue_store(const GemmParams& p, const float (&v)[BN / 2], int e, int n, int half, bool valid,
                            int64_t prow, float& amax, unsigned gap_ns = 0) {
  constexpr bool kL1 = KIND <= kL1Requant;
  constexpr int kCols = BN / 2;
  if constexpr (kL1) {
    constexpr int G = kCols / 2;           // h columns of this warp
    const int hcol0 = n * (BN / 2) + (BN == 256 ? 64 * half : 32 * half);
    const float gs_a = __ldg(p.gs_a);
    const float ag = __fmul_rn(gs_a, __ldg(p.gs_b0 + e));
    const float au = __fmul_rn(gs_a, __ldg(p.gs_b1 + e));
    float rg = 0.0f;
    if (KIND == kL1Requant) rg = recip_global_scale(__ldg(p.gs_h));
    uint32_t sfw = 0;
#pragma unroll
    for (int c = 0; c < G / 16; ++c) {
      if (gap_ns && c) __nanosleep(gap_ns);
      float g[16], u[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        g[i] = round_bf16(__fmul_rn(ag, v[16 * c + i]));
        u[i] = round_bf16(__fmul_rn(au, v[G + 16 * c + i]));
      }
      const int col = hcol0 + 16 * c;  // h column (gate/up column) of element 0
      if (KIND == kL1GateUp) {
        if (valid) {
          uint4* dg = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + col);
          uint4* du =
              reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + p.I + col);
          dg[0] = make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]),
                             pack_bf16x2(g[6], g[7]));
          dg[1] = make_uint4(pack_bf16x2(g[8], g[9]), pack_bf16x2(g[10], g[11]), pack_bf16x2(g[12], g[13]),
                             pack_bf16x2(g[14], g[15]));
          du[0] = make_uint4(pack_bf16x2(u[0], u[1]), pack_bf16x2(u[2], u[3]), pack_bf16x2(u[4], u[5]),
                             pack_bf16x2(u[6], u[7]));
          du[1] = make_uint4(pack_bf16x2(u[8], u[9]), pack_bf16x2(u[10], u[11]), pack_bf16x2(u[12], u[13]),
                             pack_bf16x2(u[14], u[15]));
        }
      } else {
        float h[16];
        float bm = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          h[i] = silu_mul(g[i], u[i]);
          bm = fmaxf(bm, fabsf(h[i]));
        }
        if (valid) {
          if (p.out_bf16) {
            uint4* dh = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + col);
            dh[0] = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                               pack_bf16x2(h[6], h[7]));
            dh[1] = make_uint4(pack_bf16x2(h[8], h[9]), pack_bf16x2(h[10], h[11]), pack_bf16x2(h[12], h[13]),
                               pack_bf16x2(h[14], h[15]));
          }
          amax = fmaxf(amax, bm);
        }
        if (KIND == kL1Requant) {
          float rb;
          const uint32_t sb = block_scale(bm, rg, rb);
          uint32_t w0 = 0, w1 = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // signed (h*rg)*rb: the conversion keeps the sign, also of a zero code
            uint32_t b0 = e2m1x2(code_mag(h[2 * i], rg, rb), code_mag(h[2 * i + 1], rg, rb));
            uint32_t b1 = e2m1x2(code_mag(h[8 + 2 * i], rg, rb), code_mag(h[8 + 2 * i + 1], rg, rb));
            w0 |= b0 << (8 * i);
            w1 |= b1 << (8 * i);
          }
          sfw |= sb << (8 * c);
          if (valid) *reinterpret_cast<uint2*>(p.h_fp4 + prow * (p.I >> 1) + (col >> 1)) = make_uint2(w0, w1);
        }
      }
    }
    if (KIND == kL1Requant && valid) {
      // G/16 consecutive scale columns starting at a multiple of 2 (BN 128) or 4 (BN 256)
      uint8_t* sp = p.h_sf + sf_swizzle_offset(prow, hcol0 >> 4, p.I >> 4);
      if constexpr (G == 64)
        *reinterpret_cast<uint32_t*>(sp) = sfw;
      else
        *reinterpret_cast<uint16_t*>(sp) = (uint16_t)sfw;
    }
  } else {
    const float alpha = __fmul_rn(__ldg(p.gs_a), __ldg(p.gs_b0 + e));
    int32_t tok = -1;
    float wgt = 0.0f;
    if (KIND == kL2Scatter && valid) {
      tok = __ldg(p.slot_token + prow);
      wgt = __ldg(p.slot_weight + prow);
      if (tok >= p.T) {
        set_status(p.status, MOE_ERR_DEVICE_INDEX);
        tok = -1;
      }
    }
#pragma unroll
    for (int c = 0; c < kCols / 16; ++c) {
      if (KIND == kL2Rows && gap_ns && c) __nanosleep(gap_ns);
      float y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) y[i] = round_bf16(__fmul_rn(alpha, v[16 * c + i]));
      const int col = n * BN + half * kCols + c * 16;
      if (KIND == kL2Rows) {
        if (valid) {
          uint4* dy = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + col);
          // streaming stores: the rows are read once, by the combine after this kernel;
          // left as ordinary lines, the last ~100 MB of them would still sit dirty in L2
          // and be written back while the combine reads
          __stcs(dy, make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                pack_bf16x2(y[6], y[7])));
          __stcs(dy + 1, make_uint4(pack_bf16x2(y[8], y[9]), pack_bf16x2(y[10], y[11]), pack_bf16x2(y[12], y[13]),
                                    pack_bf16x2(y[14], y[15])));
        }
      } else if (tok >= 0) {
        float4* dst = reinterpret_cast<float4*>(p.out32 + (int64_t)tok * p.out_cols + col);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          atomicAdd(dst + j, make_float4(__fmul_rn(wgt, y[4 * j]), __fmul_rn(wgt, y[4 * j + 1]),
                                         __fmul_rn(wgt, y[4 * j + 2]), __fmul_rn(wgt, y[4 * j + 3])));
      }
    }
  }
}

// End of the epilogue loop: the warp's max |h| into the dynamic-scale accumulator.
template <int KIND>
MOE_DEV void epilogue_finish(const GemmParams& p, float amax) {
  if (KIND == kL1Silu && p.h_amax) {
    // non-negative floats order like their bit patterns
    const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax));
    if ((threadIdx.x & 31) == 0 && mb) atomicMax(reinterpret_cast<uint32_t*>(p.h_amax), mb);
  }
}

// The CTA-pair kernel (host): ta = slot rows [cap, Kred/2] in boxes of 128 rows, tb =
// weight rows (L1: make_tmap_w1_blocks with one block per box; L2: boxes of 128 rows),
// kind a GemmKind.
moe_status launch_pair_gemm(int kind, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                            cudaStream_t st, bool pdl);
bool pair_gemm_enabled(bool l1);

// Gap between an epilogue warp's 16-column chunks: a tile's MMAs take about 0.45 us per
// 256-deep k-block, and the chunks with their gaps must end well within that (prefill L2:
// 12 k-blocks, seven 360 ns gaps, 2.5 us of a 5.5 us tile; L1: 16 k-blocks, three 300 ns
// gaps beside ~3.4 us of math in a 7.5 us tile).
template <int KIND>
MOE_DEV unsigned epilogue_gap_ns(int nkb) {
  return KIND == kL2Rows ? (unsigned)min(30 * nkb, 400) : KIND == kL1Requant ? (unsigned)min(19 * nkb, 300) : 0u;
}

}  // namespace moe
