// Persistent grouped NVFP4 x NVFP4 GEMM on tcgen05 block-scaled MMA (sm_103a), for
// experts that own many slots (prefill): the tensor-bound case.
//
// Method: nvfp4-megamoe-kernel commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py
// ("global scale as alpha": D = alpha * A @ B per expert, alpha = product of the
// global scales), of src ("grouped GEMM over 1-D slot ranges"; the scale-factor
// atom layout m = f0 + 32 f1 + 128 f2, k_sf = f4 + 4 f5), of vllm/nvfp4_cutedsl.py
// ("intermediate_size": gate | up split at I; int32 expert offsets) and of tests
// ("complete pipeline": SiLU(gate)*up in BF16, requantise, weighted scatter).
//
// Tile: 128 slot rows (M) x BN weight rows (N = 256, or 128 where the shape needs
// it), K staged 256 elements at a time.  For L1 a 256-row tile is two prepared
// 128-row blocks, each 64 gate rows then the matching 64 up rows (128 h columns).
// One CTA per SM, 12 warps:
//   warp 0      TMA producer: A (slot rows), B (weight rows) and their scale atoms
//               into a shared-memory ring (full/empty mbarriers), four loads per stage.
//   warp 1      MMA issuer and TMEM owner: only tcgen05.mma (M=128, N=BN, K=64),
//               four per stage, into one TMEM accumulator of BN columns.
//   warps 2, 3  scale copiers: once a stage's scale atoms have landed, tcgen05.cp of
//               them into TMEM (each warp two of the four k-steps), then a commit that
//               arrives on the stage's full barrier, so the MMA warp waits on a single
//               barrier per stage.  Issued from other warps than the MMAs: one thread
//               issuing both spends about twice as long per stage (measured), and the
//               MMA warp's own per-stage work (wait, fence, commit) already costs as
//               much as a third of its four MMAs.
//   warps 4-11  epilogue: two warps per TMEM lane quarter, each taking half of the
//               accumulator columns into registers; the accumulator is released as
//               soon as all eight have loaded, before the epilogue math, so the next
//               tile's MMAs wait only for the TMEM reads.
// Tiles are (expert, n-tile, m-tile), m fastest, dealt round-robin over the CTAs, so
// CTAs running at the same time share weight tiles through L2; the expert of a tile
// comes from the padded offsets on the device (no host sync).
#include "gemm_tiled.cuh"
#include "pipeline.cuh"

namespace moe {

template <int BN>
struct TiledCfg {
  static constexpr int kBlocks = BN / 128;                  // 128-row weight blocks per tile
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kAStage = kBM * kBKBytes;            // 16 KB
  static constexpr int kBStage = BN * kBKBytes;             // 32 / 16 KB
  static constexpr int kSfaStage = 4 * 512;
  static constexpr int kSfbStage = kBlocks * 4 * 512;
  static constexpr int kSfbPerStep = 4 * kBlocks;           // TMEM columns of B scales per k-step
  static constexpr int kSfCols = 16 + 4 * kSfbPerStep;      // TMEM columns of one stage's scales
  static constexpr int kSfBase = BN;                        // accumulator first
  static constexpr uint32_t kIdesc =
      (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
  static_assert(kSfBase + kStages * kSfCols <= kTmemCols, "tensor memory budget");
};

template <int BN>
struct __align__(1024) GemmSmem {
  using C = TiledCfg<BN>;
  uint8_t a[C::kStages][C::kAStage];
  uint8_t b[C::kStages][C::kBStage];
  uint8_t sfa[C::kStages][C::kSfaStage];
  uint8_t sfb[C::kStages][C::kSfbStage];
  uint64_t full[C::kStages];
  uint64_t empty[C::kStages];
  uint64_t sf_full[C::kStages];     // the stage's scale atoms have landed (copiers wait on it)
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int bad_offsets;
  int poff[257];
  int cnt[256];
  int cum[257];                     // tiles before expert e
};

template <int KIND, int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_sfb, const GemmParams p) {
  using C = TiledCfg<BN>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  GemmSmem<BN>& s =
      *reinterpret_cast<GemmSmem<BN>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kL1 = KIND <= kL1Requant;
  int* abort_flag = &s.abort_flag;

  griddep_wait();
  griddep_launch_dependents();
  build_tile_table(s, p, 1);
  if (threadIdx.x == 32) {
    for (int i = 0; i < kStages; ++i) {
      // full: operand bytes + the producer's arrival + both copiers' commits (their
      // scale copies are done), so the MMA warp waits on one barrier per stage
      mbar_init(&s.full[i], 3);
      mbar_init(&s.empty[i], 1);
      mbar_init(&s.sf_full[i], 1);
    }
    mbar_init(&s.tfull, 1);
    mbar_init(&s.tempty, kEpiWarps);
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  const bool bad = s.bad_offsets != 0;
  if (bad && threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE_INDEX);
  const int total_tiles = bad ? 0 : s.cum[p.E];
  const int nkb = (p.Kred + 255) >> 8;
  const int ksf4 = p.Kred >> 6;  // scale atoms per 128 rows

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t n_issued = 0;  // stages issued (the teardown derives each entry's last phase)
      bool ok = true;
      TileCursor cur;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        int n, m;
        if (!cur.locate(s, p.E, 1, t, n, m)) break;
        const int e = cur.e;
        const int row_a = s.poff[e] + m * kBM;
        const uint8_t* sfa_src = p.a_sf + ((int64_t)(row_a >> 7) * ksf4) * 512;
        // prepared weight row blocks n*kBlocks .. n*kBlocks + kBlocks - 1 of expert e
        const int sfb_block = e * (p.b_rows >> 7) + n * C::kBlocks;
        // four loads per stage (the producer's issue time, not the bytes, bounds how fast
        // stages arrive): the weight scale atoms of all kBlocks blocks in one 3-D box (a short
        // last stage reads zeros past the row end); the A scale atoms; A rows; the tile's
        // weight rows in one box (L1: kBlocks blocks of 64 gate then 64 up rows, a 5-D box).
        // The scales go first (the weight scales' 3-D box before the activation scales' bulk
        // copy, which lands sooner): their copies into tensor memory are on the path from a
        // stage's release to its MMAs, and they then land ahead of the operand bytes.
        for (int kb = 0; kb < nkb; ++kb) {
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.sf_full[stage], natoms * 512 + C::kSfbStage);
          mbar_arrive_expect_tx(&s.full[stage], C::kAStage + C::kBStage);
          const int x = kb * kBKBytes;
          tma_load_3d(s.sfb[stage], &tmap_sfb, &s.sf_full[stage], 0, 8 * kb, sfb_block);
          bulk_load(s.sfa[stage], sfa_src + kb * 4 * 512, natoms * 512, &s.sf_full[stage]);
          tma_load_2d(s.a[stage], &tmap_a, &s.full[stage], x, row_a);
          if (kL1)
            tma_load_5d(s.b[stage], &tmap_b, &s.full[stage], x, 0, 0, n * C::kBlocks, e);
          else
            tma_load_2d(s.b[stage], &tmap_b, &s.full[stage], x, e * p.b_rows + n * BN);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok || *(volatile int*)abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        for (int i = 0; i < kStages; ++i)
          if (n_issued > (uint32_t)i) wait_bar_drain(&s.full[i], sched::ring_last_phase(n_issued, i, kStages));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      const uint64_t da0 = sdesc_sw128(s.a[0]), db0 = sdesc_sw128(s.b[0]);
      // this stage's scale columns and operand descriptors, advanced with the ring position
      // (register updates after each commit, not a multiply before each stage's first MMA)
      uint32_t sf = tmem + C::kSfBase;
      uint64_t da = da0, db = db0;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++it) {
        if (!wait_bar_bounded(&s.tempty, (it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (natoms == 4) {  // every k-block but a short last one: no loop overhead between MMAs
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_fp4(tmem, da + 2 * kk, db + 2 * kk, C::kIdesc, sf + 4 * kk, sf + 16 + C::kSfbPerStep * kk,
                         (kb | kk) != 0);
          } else {
            for (int kk = 0; kk < natoms; ++kk)
              tc_mma_fp4(tmem, da + 2 * kk, db + 2 * kk, C::kIdesc, sf + 4 * kk, sf + 16 + C::kSfbPerStep * kk,
                         (kb | kk) != 0);
          }
          tc_commit(&s.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
            sf = tmem + C::kSfBase;
            da = da0;
            db = db0;
          } else {
            sf += C::kSfCols;
            da += (uint64_t)(C::kAStage >> 4);
            db += (uint64_t)(C::kBStage >> 4);
          }
        }
        if (!ok) break;
        tc_commit(&s.tfull);
      }
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit(&s.drain);
      wait_bar_drain(&s.drain, 0);
    }
  } else if (warp <= 3) {
    // ------------------------------------------------------------ scale copiers
    // copier c copies k-steps 2c, 2c+1 of every stage: the A atom and the kBlocks B
    // atoms of each (B atom j of k-step kk at column 16 + kSfbPerStep*kk + 4j).
    if (lane == 0) {
      const int c = warp - 2;
      int stage = 0;
      uint32_t phase = 0;
      const uint64_t dsa0 = sdesc_sf(s.sfa[0]), dsb0 = sdesc_sf(s.sfb[0]);
      for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.sf_full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sf = tmem + C::kSfBase + stage * C::kSfCols;
          const uint64_t dsa = dsa0 + (uint64_t)((stage * C::kSfaStage) >> 4);
          const uint64_t dsb = dsb0 + (uint64_t)((stage * C::kSfbStage) >> 4);
          if (natoms == 4) {  // every k-block but a short last one: the copies back to back
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int kk = 2 * c + h;
              tc_cp_sf(sf + 4 * kk, dsa + 32 * kk);
#pragma unroll
              for (int j = 0; j < C::kBlocks; ++j)
                tc_cp_sf(sf + 16 + C::kSfbPerStep * kk + 4 * j, dsb + 128 * j + 32 * kk);
            }
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int kk = 2 * c + h;
              if (kk < natoms) {
                tc_cp_sf(sf + 4 * kk, dsa + 32 * kk);
#pragma unroll
                for (int j = 0; j < C::kBlocks; ++j)
                  tc_cp_sf(sf + 16 + C::kSfbPerStep * kk + 4 * j, dsb + 128 * j + 32 * kk);
              }
            }
          }
          tc_commit(&s.full[stage]);  // arrives once this warp's copies are done
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int half = (warp - 4) >> 2;          // which half of the accumulator columns
    const int row = q * 32 + lane;
    constexpr int kCols = BN / 2;              // accumulator columns per epilogue warp
    int it = 0;
    TileCursor cur;
    float amax = 0.0f;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++it) {
      int n, m;
      if (!cur.locate(s, p.E, 1, t, n, m)) break;
      const int e = cur.e;
      const bool valid = m * kBM + row < s.cnt[e];
      const int64_t prow = (int64_t)s.poff[e] + m * kBM + row;
      if (!wait_bar_bounded(&s.tfull, it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
      float v[kCols];
      epilogue_load<KIND, BN>(taddr, half, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty);  // accumulator free: values are in registers
      epilogue_store<KIND, BN>(p, v, e, n, half, valid, prow, amax, epilogue_gap_ns<KIND>(nkb));
    }
    epilogue_finish<KIND>(p, amax);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int KIND, int BN>
static moe_status launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsb, const GemmParams& p,
                            cudaStream_t st, bool pdl) {
  constexpr size_t kSmemBytes = sizeof(GemmSmem<BN>) + 1024;
  static PerDeviceOnce configured;
  if (configured.run([] {
        return cudaFuncSetAttribute(grouped_gemm_kernel<KIND, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
      }) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_ex(grouped_gemm_kernel<KIND, BN>, num_sms(), kGemmThreads, kSmemBytes, st, pdl, ta, tb, tsb, p) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// ta: slot rows (boxes of 128 rows); tb: weight rows (L1: make_tmap_w1_blocks with bn/128
// blocks per box; L2: boxes of bn rows); tsb: the prepared weight scales (bn/128 blocks).
template <int KIND>
static moe_status launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsb,
                              const GemmParams& p, int bn, cudaStream_t st, bool pdl) {
  return bn == 256 ? launch_bn<KIND, 256>(ta, tb, tsb, p, st, pdl) : launch_bn<KIND, 128>(ta, tb, tsb, p, st, pdl);
}

static int g_policy = MOE_GEMM_AUTO;

int gemm_policy() { return __atomic_load_n(&g_policy, __ATOMIC_RELAXED); }

int set_gemm_policy(int policy) { return __atomic_exchange_n(&g_policy, policy, __ATOMIC_RELAXED); }

// Which GEMM runs its 256-wide tiles on CTA pairs: L2 unless single-CTA tiles are
// forced (prefill L2 0.38 ms against 0.41 ms); L1 only when forced (0.69 ms against
// 0.68: the pair computes the empty half of every expert's odd last m-tile).
bool pair_gemm_enabled(bool l1) {
  const int pol = gemm_policy();
  return l1 ? pol == MOE_GEMM_TILED_PAIR : pol != MOE_GEMM_TILED_1CTA;
}

// Small per-expert slot counts (at most 64 slots per local expert on average even if
// every pair were local): stream the weights with the slot chunk on the MMA's N side.
bool use_stream_gemm(int64_t cap, int E, int Kred) {
  const int pol = gemm_policy();
  if (pol == MOE_GEMM_TILED || pol == MOE_GEMM_TILED_1CTA || pol == MOE_GEMM_TILED_PAIR ||
      !stream_gemm_supported(Kred))
    return false;
  if (pol != MOE_GEMM_AUTO) return true;
  return cap - (int64_t)(kTileM - 1) * E <= (int64_t)64 * E;
}

// Slot chunk of the streaming kernel: 32 (more pipeline stages fit; heavier experts
// take several chunks) unless the policy forces 64.
int stream_chunk(int64_t, int) { return gemm_policy() == MOE_GEMM_STREAMING_N64 ? 64 : 32; }

// L1: A = slot activations [cap, K/2]; B = W1 [E*2I, K/2]; a tile covers BN/2 h columns.
moe_status launch_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a, const int32_t* offsets,
                          const int32_t* padded_offsets, int E, int64_t cap, int K, int I, const uint8_t* w1_fp4,
                          const uint8_t* w1_sf, const float* gs_g, const float* gs_u, int epilogue, void* out_bf16,
                          float* h_amax, uint8_t* h_fp4, uint8_t* h_sf, const float* gs_h, int32_t* status,
                          cudaStream_t st, bool pdl, int32_t* tile_claim) {
  if (use_stream_gemm(cap, E, K))
    return launch_stream_gemm_l1(a_fp4, a_sf, gs_a, offsets, padded_offsets, E, cap, K, I, w1_fp4, w1_sf, gs_g, gs_u,
                                 epilogue, out_bf16, h_amax, h_fp4, h_sf, gs_h, status, st, pdl, tile_claim);
  const int bn = I % 128 == 0 ? 256 : 128;
  CUtensorMap ta, tb, tsb;
  if (!make_tmap(&ta, a_fp4, (uint64_t)K / 2, (uint64_t)cap, kBM)) return MOE_ERR_CUDA;
  GemmParams p{};
  p.a_sf = a_sf;
  p.b_sf = w1_sf;
  p.offsets = offsets;
  p.padded_offsets = padded_offsets;
  p.E = E;
  p.Kred = K;
  p.n_tiles = I / (bn / 2);
  p.b_rows = 2 * I;
  p.I = I;
  p.cap = cap;
  p.gs_a = gs_a;
  p.gs_b0 = gs_g;
  p.gs_b1 = gs_u;
  p.out_bf16 = out_bf16;
  p.out_ld = epilogue == MOE_L1_GATEUP_BF16 ? 2 * (int64_t)I : I;
  p.h_amax = h_amax;
  p.h_fp4 = h_fp4;
  p.h_sf = h_sf;
  p.gs_h = gs_h;
  p.status = status;
  if (epilogue == MOE_L1_SILU_BF16 && h_amax) {
    if (cudaMemsetAsync(h_amax, 0, sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
    pdl = false;  // the predecessor is now the memset, not a kernel
  }
  if (bn == 256 && pair_gemm_enabled(true)) {
    const int kind = epilogue == MOE_L1_GATEUP_BF16 ? kL1GateUp : epilogue == MOE_L1_SILU_BF16 ? kL1Silu : kL1Requant;
    if (epilogue != MOE_L1_GATEUP_BF16 && epilogue != MOE_L1_SILU_BF16 && epilogue != MOE_L1_SILU_REQUANT)
      return MOE_ERR_INVALID_ARG;
    // each CTA of a pair loads one 64 gate + 64 up row block
    if (!make_tmap_w1_blocks(&tb, w1_fp4, (uint64_t)K / 2, I, E, 1)) return MOE_ERR_CUDA;
    return launch_pair_gemm(kind, ta, tb, p, st, pdl);
  }
  if (!make_tmap_w1_blocks(&tb, w1_fp4, (uint64_t)K / 2, I, E, bn / 128) ||
      !make_tmap_sf_blocks(&tsb, w1_sf, K / 64, (uint64_t)E * (2 * I / 128), bn / 128))
    return MOE_ERR_CUDA;
  switch (epilogue) {
    case MOE_L1_GATEUP_BF16: return launch_kind<kL1GateUp>(ta, tb, tsb, p, bn, st, pdl);
    case MOE_L1_SILU_BF16: return launch_kind<kL1Silu>(ta, tb, tsb, p, bn, st, pdl);
    case MOE_L1_SILU_REQUANT: return launch_kind<kL1Requant>(ta, tb, tsb, p, bn, st, pdl);
  }
  return MOE_ERR_INVALID_ARG;
}

// L2: A = h codes [cap, I/2]; B = W2 [E*K, I/2]; a tile covers BN output columns.
moe_status launch_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h, const int32_t* offsets,
                          const int32_t* padded_offsets, int E, int64_t cap, int I, int K, const uint8_t* w2_fp4,
                          const uint8_t* w2_sf, const float* gs_w2, int epilogue, void* y_rows,
                          const int32_t* slot_token, const float* slot_weight, float* out32, int64_t T,
                          int32_t* status, cudaStream_t st, bool pdl, int32_t* tile_claim) {
  if (use_stream_gemm(cap, E, I))
    return launch_stream_gemm_l2(h_fp4, h_sf, gs_h, offsets, padded_offsets, E, cap, I, K, w2_fp4, w2_sf, gs_w2,
                                 epilogue, y_rows, slot_token, slot_weight, out32, T, status, st, pdl, tile_claim);
  const int bn = K % 256 == 0 ? 256 : 128;
  const bool pair = bn == 256 && pair_gemm_enabled(false);
  CUtensorMap ta, tb, tsb;
  if (!make_tmap(&ta, h_fp4, (uint64_t)I / 2, (uint64_t)cap, kBM)) return MOE_ERR_CUDA;
  // boxes of one tile's weight rows (a CTA pair: each CTA 128 of them)
  if (!make_tmap(&tb, w2_fp4, (uint64_t)I / 2, (uint64_t)E * K, pair ? 128 : bn)) return MOE_ERR_CUDA;
  GemmParams p{};
  p.a_sf = h_sf;
  p.b_sf = w2_sf;
  p.offsets = offsets;
  p.padded_offsets = padded_offsets;
  p.E = E;
  p.Kred = I;
  p.n_tiles = K / bn;
  p.b_rows = K;
  p.I = I;
  p.gs_a = gs_h;
  p.gs_b0 = gs_w2;
  p.out_bf16 = y_rows;
  p.out_ld = K;
  p.slot_token = slot_token;
  p.slot_weight = slot_weight;
  p.out32 = out32;
  p.T = T;
  p.out_cols = K;
  p.cap = cap;
  p.status = status;
  if (pair) {
    if (epilogue != MOE_L2_ROWS_BF16 && epilogue != MOE_L2_SCATTER) return MOE_ERR_INVALID_ARG;
    return launch_pair_gemm(epilogue == MOE_L2_ROWS_BF16 ? kL2Rows : kL2Scatter, ta, tb, p, st, pdl);
  }
  if (!make_tmap_sf_blocks(&tsb, w2_sf, I / 64, (uint64_t)E * (K / 128), bn / 128)) return MOE_ERR_CUDA;
  switch (epilogue) {
    case MOE_L2_ROWS_BF16: return launch_kind<kL2Rows>(ta, tb, tsb, p, bn, st, pdl);
    case MOE_L2_SCATTER: return launch_kind<kL2Scatter>(ta, tb, tsb, p, bn, st, pdl);
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace moe
