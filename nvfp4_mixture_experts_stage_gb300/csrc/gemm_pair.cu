// Persistent grouped NVFP4 x NVFP4 GEMM for the tensor-bound case (prefill, skewed
// routing) on CTA pairs: one tcgen05.mma of M = 256 (cta_group::2) computes a tile of
// 256 slot rows x 256 weight rows on two SMs.
//
// Method: as the single-CTA tiled kernel (nvfp4-megamoe-kernel commits of
// src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py, "global scale as alpha"; of src,
// "grouped GEMM over 1-D slot ranges" and the scale-factor atom layout; of
// vllm/nvfp4_cutedsl.py, gate | up split at I; of tests, "complete pipeline").
//
// Why pairs: a single SM running M=128 x N=256 MMAs must stream 12 KB of operands
// per 64-deep k-step into its shared memory and issue 3 scale copies and one MMA per
// k-step from its own threads.  In a pair each SM stages its own 128 slot rows and
// only half of the 256 weight rows (the MMA reads the other half from the peer's
// shared memory), so each SM receives 8 KB per k-step, a stage takes 38 KB of shared
// memory instead of 54 KB (five stages fit instead of four), and one thread issues
// the MMA and the scale copies of both SMs.
//
// Cluster of two CTAs, 12 warps each, one CTA per SM.  Rank 0 leads; every barrier
// the pipeline runs on lives in the leader except each CTA's empty[s] and tfull.
//   warp 0 (both)      TMA producer: this CTA's scale atoms first (the B atoms of all 256
//                      weight rows, since the MMA reads every B scale from the local TMEM,
//                      then the A atoms of its rows), then its A rows and its 128 weight rows, into
//                      a five-stage ring.  The loads use the CTA-pair form of TMA, so the
//                      peer's bytes count directly on the leader's sf_full[c][s] (scales) and
//                      full[s] (operands); the leader's producer arms both with the bytes
//                      of the two CTAs.
//   warp 1, leader     MMA issuer: four M=256 N=256 K=64 MMAs per stage once full[s]
//                      completes (operand bytes of both CTAs + the copier's commit); a
//                      multicast commit frees the stage in both CTAs; a multicast commit
//                      on tfull hands the accumulator to both epilogues.
//   warps 2, 3, leader scale copiers, alternating stages (copier c takes the stages g
//                      with g % 2 == c): once sf_full[c][s] completes, the stage's 12 scale
//                      atoms into both TMEMs (one cta_group::2 copy each), then a commit on
//                      full[s].  Each copier has its own sf_full barriers: a barrier whose
//                      consecutive phases were waited on by different warps could let one
//                      of them, two uses ahead, pass on the parity of an older phase.
//   warps 4-11 (both)  epilogue of this CTA's 128 rows (shared with the single-CTA
//                      kernel); after reading the accumulator every warp arrives on the
//                      leader's tempty (16 arrivals), which the next tile's MMAs wait for.
// Tiles are (expert, n-tile, pair of 128-row m-tiles), m fastest, dealt round-robin
// over the pairs.  An expert with an odd number of m-tiles leaves the peer's half of
// its last tile empty: the peer loads no A rows there and stores nothing.
// Teardown: a CTA leaves only after every arrival aimed at its barriers has landed,
// including the ones nobody consumes in the pipeline (the multicast release of each
// stage's last use, the last tile's remote tempty arrivals): its producer and the
// leader's MMA thread wait for those phases before the final cluster barrier.
#include <algorithm>

#include "gemm_tiled.cuh"
#include "pipeline.cuh"

namespace moe {

namespace {

constexpr int kPStages = 5;
constexpr int kPAStage = kBM * kBKBytes;   // 16 KB: this CTA's 128 slot rows
constexpr int kPBStage = 128 * kBKBytes;   // 16 KB: this CTA's 128 of the tile's 256 weight rows
constexpr int kPSfaStage = 4 * 512;        // A scale atoms of this CTA's rows, one per k-step
constexpr int kPSfbStage = 2 * 4 * 512;    // B scale atoms of both weight blocks: [block][k-step]
constexpr int kPSfCols = 16 + 4 * 8;       // TMEM columns of one stage's scales (A 4, B 8 per k-step)
constexpr int kPSfBase = 256;              // accumulator first
// kind::mxf4nvf4, E2M1 A and B, K-major, UE4M3 scales, N = 256, M = 256 (the pair)
constexpr uint32_t kPIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
static_assert(kPSfBase + kPStages * kPSfCols <= kTmemCols, "tensor memory budget");

struct __align__(1024) PairSmem {
  uint8_t a[kPStages][kPAStage];
  uint8_t b[kPStages][kPBStage];
  uint8_t sfa[kPStages][kPSfaStage];
  uint8_t sfb[kPStages][kPSfbStage];
  uint64_t sf_full[2][kPStages];  // leader, per copier: both CTAs' scale atoms of the stage have landed
  uint64_t full[kPStages];     // leader: both CTAs' operands landed and the scales are in TMEM
  uint64_t empty[kPStages];    // the pair's MMAs of the stage are done (multicast commit)
  uint64_t tfull;            // accumulator complete (multicast commit)
  uint64_t tempty;           // leader: all epilogue warps of the pair have read it
  uint64_t drain;            // leader: every MMA it issued is complete
  uint32_t tmem_base;
  int abort_flag;
  int bad_offsets;
  int poff[257];
  int cnt[256];
  int cum[257];
};

MOE_DEV int pair_tiles(int total_tiles, int pair, int npairs) {
  return pair < total_tiles ? (total_tiles - pair + npairs - 1) / npairs : 0;
}

}  // namespace

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ CUtensorMap tmap_sfa, const __grid_constant__ CUtensorMap tmap_sfb,
                             const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  PairSmem& s = *reinterpret_cast<PairSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kL1 = KIND <= kL1Requant;
  const uint32_t rank = cluster_ctarank();  // 0: leader, 1: peer
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  int* abort_flag = &s.abort_flag;

  griddep_wait();
  griddep_launch_dependents();
  build_tile_table(s, p, 2);
  if (threadIdx.x == 32) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&s.sf_full[0][i], 1);
      mbar_init(&s.sf_full[1][i], 1);
      mbar_init(&s.full[i], 2);  // the producer's arming + the copier's commit (+ the bytes)
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(&s.tfull, 1);
    mbar_init(&s.tempty, 2 * kEpiWarps);
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    // one warp of each CTA allocates the same columns in both TMEMs
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrival or multicast commit
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  const bool bad = s.bad_offsets != 0;
  if (bad && threadIdx.x == 0 && rank == 0) set_status(p.status, MOE_ERR_DEVICE_INDEX);
  const int total_tiles = bad ? 0 : s.cum[p.E];
  const int nkb = (p.Kred + 255) >> 8;
  const int ksf4 = p.Kred >> 6;  // scale atoms per 128 rows
  const int my_stages = pair_tiles(total_tiles, pair, npairs) * nkb;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      TileCursor cur;
      // leader addresses of the two copiers' sf_full rings (scalars: a runtime-indexed
      // array would live in local memory and cost a load on every stage)
      const uint32_t sf_full_c0 = mapa_shared(smem_u32(&s.sf_full[0][0]), 0);
      const uint32_t sf_full_c1 = mapa_shared(smem_u32(&s.sf_full[1][0]), 0);
      uint32_t g = 0;  // stages issued so far; stage g's scales go to copier sched::pair_copier(g)
      const uint32_t full0 = mapa_shared(smem_u32(&s.full[0]), 0);
      for (int t = pair; t < total_tiles && ok; t += npairs) {
        int n, mp;
        if (!cur.locate(s, p.E, 2, t, n, mp)) break;
        const int e = cur.e;
        const int mt = (s.poff[e + 1] - s.poff[e]) >> 7;
        const int m = 2 * mp + (int)rank;  // this CTA's 128-row m-tile
        const bool has_rows = m < mt;
        const bool peer_rows = 2 * mp + 1 < mt;
        const int row_a = s.poff[e] + m * kBM;
        // scale atoms as rows of 256 B: a stage's four atoms are eight rows; the weight
        // scales of prepared blocks 2n and 2n + 1 come in one 3-D box
        const int sfa_row = ((row_a >> 7) * ksf4) * 2;
        const int sfb_block = e * (p.b_rows >> 7) + n * 2;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!wait_bar_bounded(&s.empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (rank == 0) {
            // both CTAs' bytes: SFA 2 KB + SFB 4 KB each (A rows only where the CTA has rows);
            // A 16 KB + B 16 KB each
            mbar_arrive_expect_tx(&s.sf_full[sched::pair_copier(g)][stage],
                                  2 * 4096 + 2048 * (1 + (peer_rows ? 1 : 0)));
            mbar_arrive_expect_tx(&s.full[stage], 2 * kPBStage + kPAStage * (1 + (peer_rows ? 1 : 0)));
          }
          const uint32_t sfb = (sched::pair_copier(g) ? sf_full_c1 : sf_full_c0) + 8 * stage,
                         fb = full0 + 8 * stage;
          const int x = kb * kBKBytes;
          tma_load_3d_pair(s.sfb[stage], &tmap_sfb, sfb, 0, 8 * kb, sfb_block);
          if (has_rows) tma_load_2d_pair(s.sfa[stage], &tmap_sfa, sfb, 0, sfa_row + 8 * kb);
          if (has_rows) tma_load_2d_pair(s.a[stage], &tmap_a, fb, x, row_a);
          if (kL1) {
            // prepared block 2n + rank: 64 gate rows then the matching 64 up rows (one 5-D box)
            tma_load_5d_pair(s.b[stage], &tmap_b, fb, x, 0, 0, 2 * n + (int)rank, e);
          } else {
            tma_load_2d_pair(s.b[stage], &tmap_b, fb, x, e * p.b_rows + n * 256 + 128 * (int)rank);
          }
          ++g;
          if (++stage == kPStages) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok || *(volatile int*)abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away: the
        // leader sees its barriers complete; every load lands within microseconds
        if (rank == 0)
          for (int i = 0; i < kPStages; ++i)
            if (g > (uint32_t)i) wait_bar_drain(&s.full[i], sched::ring_last_phase(g, i, kPStages));
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      } else {
        // The release of each stage's last use is a multicast commit from the leader's
        // MMA thread that nobody else waits for; it must land in this CTA's empty[i]
        // before the CTA (and its shared memory) is gone.
        for (int i = 0; i < kPStages; ++i)
          if (g > (uint32_t)i &&
              !wait_bar_bounded(&s.empty[i], sched::ring_last_phase(g, i, kPStages), abort_flag, p.status))
            break;
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      const uint64_t da0 = sdesc_sw128(s.a[0]), db0 = sdesc_sw128(s.b[0]);
      // this stage's scale columns and operand descriptors, advanced with the ring position
      uint32_t sf = tmem + kPSfBase;
      uint64_t da = da0, db = db0;
      for (int t = pair; t < total_tiles && ok; t += npairs, ++it) {
        if (!wait_bar_bounded(&s.tempty, (it & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          if (natoms == 4) {  // every k-block but a short last one: no loop overhead between MMAs
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_fp4_pair(tmem, da + 2 * kk, db + 2 * kk, kPIdesc, sf + 4 * kk, sf + 16 + 8 * kk,
                              (kb | kk) != 0);
          } else {
            for (int kk = 0; kk < natoms; ++kk)
              tc_mma_fp4_pair(tmem, da + 2 * kk, db + 2 * kk, kPIdesc, sf + 4 * kk, sf + 16 + 8 * kk,
                              (kb | kk) != 0);
          }
          tc_commit_pair_mc(&s.empty[stage], 0x3);
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1;
            sf = tmem + kPSfBase;
            da = da0;
            db = db0;
          } else {
            sf += kPSfCols;
            da += (uint64_t)(kPAStage >> 4);
            db += (uint64_t)(kPBStage >> 4);
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(&s.tfull, 0x3);
      }
      // the last tile's 16 epilogue arrivals (8 of them remote, from the peer) land here
      // before this CTA can leave
      if (ok && it > 0) wait_bar_bounded(&s.tempty, (it & 1) ^ 1, abort_flag, p.status);
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit_pair_mc(&s.drain, 0x1);
      wait_bar_drain(&s.drain, 0);
    }
  } else if (warp <= 3) {
    // ------------------------------------------------------------ scale copiers (leader)
    // copier c takes stages c, c + 2, ...: the A atom (column 4 kk) and the two B atoms
    // (columns 16 + 8 kk and 16 + 8 kk + 4) of every k-step kk.  kPStages is odd, so
    // these are the uses of sf_full[c][s] in order, one phase each.
    if (rank == 0 && lane == 0) {
      const uint64_t dsa0 = sdesc_sf(s.sfa[0]), dsb0 = sdesc_sf(s.sfb[0]);
      const int c = warp - 2;
      int kb = c % nkb;  // g % nkb, advanced by 2 per stage
      for (int g = c; g < my_stages; g += 2) {  // the stages with sched::pair_copier(g) == c
        const int natoms = min(4, ksf4 - 4 * kb);
        const int stage = (int)sched::pair_stage((uint32_t)g, kPStages);
        const uint32_t phase = sched::pair_sf_use((uint32_t)g, kPStages) & 1;
        if (!wait_bar_bounded(&s.sf_full[c][stage], phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t sf = tmem + kPSfBase + stage * kPSfCols;
        const uint64_t dsa = dsa0 + (uint64_t)((stage * kPSfaStage) >> 4);
        const uint64_t dsb = dsb0 + (uint64_t)((stage * kPSfbStage) >> 4);
        if (natoms == 4) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_cp_sf_pair(sf + 4 * kk, dsa + 32 * kk);
            tc_cp_sf_pair(sf + 16 + 8 * kk, dsb + 32 * kk);
            tc_cp_sf_pair(sf + 16 + 8 * kk + 4, dsb + 128 + 32 * kk);
          }
        } else {
          for (int kk = 0; kk < natoms; ++kk) {
            tc_cp_sf_pair(sf + 4 * kk, dsa + 32 * kk);
            tc_cp_sf_pair(sf + 16 + 8 * kk, dsb + 32 * kk);
            tc_cp_sf_pair(sf + 16 + 8 * kk + 4, dsb + 128 + 32 * kk);
          }
        }
        tc_commit_pair_mc(&s.full[stage], 0x1);  // the leader's barrier, once the copies are done
        kb += 2;
        while (kb >= nkb) kb -= nkb;  // nkb may be 1
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 4) >> 2;  // which half of the accumulator columns
    const int row = q * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&s.tempty), 0);
    int it = 0;
    TileCursor cur;
    float amax = 0.0f;
    for (int t = pair; t < total_tiles; t += npairs, ++it) {
      int n, mp;
      if (!cur.locate(s, p.E, 2, t, n, mp)) break;
      const int e = cur.e;
      const int m = 2 * mp + (int)rank;
      const bool valid = m * kBM + row < s.cnt[e];
      const int64_t prow = (int64_t)s.poff[e] + m * kBM + row;
      if (!wait_bar_bounded(&s.tfull, it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      float v[128];
      epilogue_load<KIND, 256>(tmem + ((uint32_t)(q * 32) << 16), half, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {  // accumulator free: values are in registers
        if (rank == 0)
          mbar_arrive(&s.tempty);
        else
          mbar_arrive_remote(tempty_leader);
      }
      epilogue_store<KIND, 256>(p, v, e, n, half, valid, prow, amax, epilogue_gap_ns<KIND>(nkb));
    }
    epilogue_finish<KIND>(p, amax);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int KIND>
static moe_status launch_pair_kind(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                                   const CUtensorMap& tsb, const GemmParams& p, cudaStream_t st, bool pdl) {
  constexpr size_t kSmemBytes = sizeof(PairSmem) + 1024;
  // as many pairs as can be resident at once (pairs sit in one GPC each); 0 on failure
  static PerDeviceInt grids;
  const int grid = grids.get([] {
    if (cudaFuncSetAttribute(grouped_gemm_pair_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_pair_kernel<KIND>, &cfg) != cudaSuccess ||
        clusters < 1)
      return 0;
    return 2 * std::min(clusters, num_sms() / 2);
  });
  if (grid <= 0) return MOE_ERR_CUDA;
  return launch_ex(grouped_gemm_pair_kernel<KIND>, dim3((unsigned)grid), dim3(kGemmThreads), kSmemBytes, st, pdl, ta,
                   tb, tsa, tsb, p) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status launch_pair_gemm(int kind, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                            cudaStream_t st, bool pdl) {
  // scale atoms seen as rows of 256 B, a stage's four atoms per box (a partial last stage
  // reads the following atoms, or zeros past the end, which no MMA uses)
  CUtensorMap tsa, tsb;
  const uint64_t sfa_rows = (uint64_t)p.cap * (uint64_t)p.Kred / 16 / 256;
  if (!make_tmap_plain(&tsa, p.a_sf, 256, sfa_rows, 8) ||
      !make_tmap_sf_blocks(&tsb, p.b_sf, p.Kred / 64, (uint64_t)p.E * (uint64_t)(p.b_rows / 128), 2))
    return MOE_ERR_CUDA;
  switch (kind) {
    case kL1GateUp: return launch_pair_kind<kL1GateUp>(ta, tb, tsa, tsb, p, st, pdl);
    case kL1Silu: return launch_pair_kind<kL1Silu>(ta, tb, tsa, tsb, p, st, pdl);
    case kL1Requant: return launch_pair_kind<kL1Requant>(ta, tb, tsa, tsb, p, st, pdl);
    case kL2Rows: return launch_pair_kind<kL2Rows>(ta, tb, tsa, tsb, p, st, pdl);
    case kL2Scatter: return launch_pair_kind<kL2Scatter>(ta, tb, tsa, tsb, p, st, pdl);
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace moe
