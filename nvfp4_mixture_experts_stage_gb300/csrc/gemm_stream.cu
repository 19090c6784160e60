// Weight-streaming grouped NVFP4 GEMM for small per-expert slot counts (decode).
//
// Same layer arithmetic as the tiled kernel in gemm.cu (nvfp4-megamoe-kernel commits
// of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py: D = alpha * A @ B per expert; of
// vllm/nvfp4_cutedsl.py: gate | up split at I; of tests: SiLU(gate)*up, requantise,
// weighted scatter), organised for the case where every expert owns only a few
// slots and the weights must simply stream from HBM:
//
//   * operands are swapped: the MMA's M=128 side is a block of weight rows and
//     its N=64 side is a chunk of up to 64 slot rows of one expert, so D^T sits in
//     TMEM with one weight row per lane;
//   * the chunk's activation scales are copied into TMEM once per chunk and stay
//     there for the whole contraction, so each pipeline stage copies only the four
//     weight-scale atoms it brings (the tiled kernel copies eight);
//   * each CTA walks a contiguous range of (expert, chunk, weight-block) tiles, so
//     consecutive tiles reuse the resident activation scales;
//   * when the launch is given a claim counter (zeroed by an earlier kernel of the
//     layer), the last tiles (three per CTA) are not in any range: every CTA claims
//     them one at a time once its range is done, so CTAs that started late (behind
//     the previous GEMM's slowest CTA) or stream slower take fewer of them.  The
//     producer claims and passes each tile to the other roles through a small queue
//     in shared memory;
//   * warp 6 builds the TMEM images of the next chunk's activation scales in shared
//     memory while the current chunk runs;
//   * two MMA-issuing warps split every tile's k-blocks by parity into two
//     accumulators (the epilogue adds them), since the tensor pipe serves each
//     issuing thread at about one instruction per ~130 cycles.  Only when a tile
//     has an even number of k-blocks: then every ring stage always belongs to the
//     same issuer.  With an odd count the stages would alternate between the two,
//     and a barrier whose consecutive phases are waited on by different threads can
//     let one of them, two uses ahead, pass on the parity of an older phase; one
//     issuer then takes all k-blocks.
//
// Scale-factor placement read by kind::mxf4nvf4.block_scale.scale_vec::4X (M=128):
// operand A row m at TMEM lane m, column base + m/32; operand B row n at lane n%32,
// column base + n/32; bases 4-column aligned.  A 512-byte atom copied with
// tcgen05.cp.32x128b.warpx4 satisfies the A placement directly; the B images put
// the chunk's rows i and 32+i in bytes 0..3 and 4..7 of image row i.
#include "tcgen05.cuh"
#include "pipeline.cuh"

namespace moe {
namespace stream {

// CHUNK = slots per chunk (the MMA's N): 32 or 64.  A 32-slot chunk halves the
// activation tile and leaves room for 8 pipeline stages instead of 6.
template <int CHUNK>
struct Cfg {
  static constexpr int kStages = CHUNK == 32 ? 8 : 6;
  static constexpr int kBStage = CHUNK * 128;            // CHUNK slot rows x 256 fp4
  // Accumulators first: one per issuer, double-buffered when they fit (32-slot chunks
  // fill the 512 columns exactly), so the issuers start a tile while the epilogue is
  // still reading the previous one.
  static constexpr int kAccBufs = CHUNK == 32 ? 2 : 1;
  static constexpr int kSfbBase = 2 * CHUNK * kAccBufs;
  static constexpr int kSfwBase = kSfbBase + 4 * 64;     // resident activation scales: 4 columns per k-step
  static constexpr uint32_t kIdesc =
      (1u << 7) | (1u << 10) | ((uint32_t)(CHUNK >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  static_assert(kSfwBase + 16 * kStages <= 512, "tensor memory budget");
};
constexpr int kWStage = 128 * 128;            // 16 KB: 128 weight rows x 256 fp4
constexpr int kSfwStage = 4 * 512;            // 4 weight-scale atoms
constexpr int kThreads = 256;                 // 8 warps
constexpr int kTmemCols = 512;
constexpr int kMaxKSteps = 64;                // contraction <= 4096
constexpr int kStageLd = 72;                  // padded row of the L1 exchange buffers (bf16)

enum Kind : int { kL1GateUp = 0, kL1Silu = 1, kL1Requant = 2, kL2Rows = 3, kL2Scatter = 4 };

struct Params {
  const uint8_t* a_sf;              // slot-row scales, 512-byte atoms [cap/128][Kred/64]
  const uint8_t* w_sf;              // prepared weight scales [E][w_rows/128][Kred/64]
  const int32_t* offsets;
  const int32_t* padded_offsets;
  int E;
  int Kred;
  int n_tiles;                      // weight blocks per expert
  int w_rows;                       // weight rows per expert
  int I;
  const float* gs_a;
  const float* gs_w0;               // L1 gate / L2 down
  const float* gs_w1;               // L1 up
  void* out_bf16;
  int64_t out_ld;
  float* h_amax;
  uint8_t* h_fp4;
  uint8_t* h_sf;
  const float* gs_h;
  const int32_t* slot_token;
  const float* slot_weight;
  float* out32;
  int64_t T;
  int out_cols;
  int64_t cap;
  int32_t* status;
  int early_weights;                // request weights before griddep_wait (see the producer)
  int32_t* claim;                   // pool claim counter, zero at launch; NULL: static ranges only
};

constexpr int kTileQ = 8;            // queue of claimed tiles (the producer leads the epilogue by <= 4)
constexpr int kPoolPerCta = 3;       // pool size in tiles per CTA

template <int CHUNK>
struct __align__(1024) Smem {
  static constexpr int kStages = Cfg<CHUNK>::kStages;
  uint8_t w[kStages][kWStage];
  uint8_t b[kStages][Cfg<CHUNK>::kBStage];
  uint8_t sfw[kStages][kSfwStage];
  uint8_t img[kMaxKSteps][512];
  uint16_t xg[CHUNK][kStageLd];     // L1 exchange: gate values [slot][h col] (bf16 bits)
  uint16_t xu[CHUNK][kStageLd];     //              up values
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];                // per accumulator buffer: both issuers' MMAs of a tile done (2 arrivals)
  uint64_t tempty[2];               // per buffer: epilogue has the accumulators in registers (4 warps)
  uint64_t drain[2];                // issuer r's MMAs so far done (one arrival per chunk switch)
  uint64_t fin[2];
  uint64_t img_full;
  uint64_t img_free;
  uint64_t dep;                     // the producer's griddep_wait() has returned
  uint64_t tq_full[kTileQ];         // entry written (the producer)
  uint64_t tq_empty[kTileQ];        // entry read by the four consumer roles
  int tq[kTileQ];                   // claimed tiles in claim order; -1 ends the walk
  int epi_tile;                     // the epilogue warps' copy of the entry being read
  uint32_t tmem_base;
  int abort_flag;
  int bad_offsets;
  int poff[257];
  int cnt[256];
  int cum[257];                     // tiles before expert e
};

// Tile t -> (expert, chunk, weight block); e advances monotonically with t.  Within
// an expert the chunk varies fastest, so an expert split into several chunks reads
// each weight block again right after the first read (from L2).
template <int CHUNK>
struct Cursor {
  int e = 0;
  template <class S>
  MOE_DEV void locate(const S& s, int n_tiles, int t, int& c, int& n) {
    while (t >= s.cum[e + 1]) ++e;
    const int local = t - s.cum[e];
    const int nch = (s.cnt[e] + CHUNK - 1) / CHUNK;
    n = local / nch;
    c = local - n * nch;
  }
};

MOE_DEV void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier of the four epilogue warps that also returns whether any of them passed true,
// so that all of them take the same branch.
MOE_DEV bool epi_bar_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// The tiles of one CTA: its static range [t, hi), then (dyn) the tiles it claims from
// the pool.  The producer claims each pool tile and writes it into queue entry d % kTileQ;
// the issuers, the scale-image builder and the epilogue each read every entry in order
// (one thread per role waits and arrives).  An entry of -1 ends the walk.
struct TileWalk {
  int t, hi;
  int d = 0;
  bool dyn;
};

template <class S>
MOE_DEV int claim_tile(TileWalk& w, S& s, const Params& p, int n_static, int total, int* abort_flag, bool& ok) {
  if (w.t < w.hi) return w.t++;
  if (!w.dyn) return -1;
  const int q = w.d % kTileQ;
  if (!wait_bar_bounded(&s.tq_empty[q], ((uint32_t)(w.d / kTileQ) & 1) ^ 1, abort_flag, p.status)) {
    ok = false;
    return -1;
  }
  int v = n_static + atomicAdd(p.claim, 1);
  if (v >= total) {
    v = -1;
    w.dyn = false;
  }
  s.tq[q] = v;
  mbar_arrive(&s.tq_full[q]);
  ++w.d;
  return v;
}

// One thread of a consumer role: the next tile, or -1 (walk over, or aborted).
template <class S>
MOE_DEV int next_tile(TileWalk& w, S& s, int* abort_flag, int32_t* status) {
  if (w.t < w.hi) return w.t++;
  if (!w.dyn) return -1;
  const int q = w.d % kTileQ;
  if (!wait_bar_bounded(&s.tq_full[q], (uint32_t)(w.d / kTileQ) & 1, abort_flag, status)) {
    w.dyn = false;
    return -1;
  }
  const int v = *reinterpret_cast<volatile int*>(&s.tq[q]);
  mbar_arrive(&s.tq_empty[q]);
  ++w.d;
  if (v < 0) w.dyn = false;
  return v;
}

template <int KIND, int CHUNK>
__global__ void __launch_bounds__(kThreads, 1)
    stream_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x,
                       const Params p) {
  using C = Cfg<CHUNK>;
  constexpr int kChunk = CHUNK;
  constexpr int kStages = C::kStages;
  constexpr int kBStage = C::kBStage;
  constexpr int kAccBufs = C::kAccBufs;
  constexpr int kSfbBase = C::kSfbBase;
  constexpr int kSfwBase = C::kSfwBase;
  constexpr uint32_t kIdesc = C::kIdesc;
  extern __shared__ uint8_t smem_raw[];
  Smem<CHUNK>& s =
      *reinterpret_cast<Smem<CHUNK>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kL1 = KIND <= kL1Requant;

  if (threadIdx.x == 0) s.bad_offsets = 0;
  __syncthreads();
  // The routing tables were written before the previous kernel of the layer started
  // (see the producer below), so they are read before griddep_wait(), from L2.
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s.poff[i] = __ldcg(p.padded_offsets + i);
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) s.cnt[i] = __ldcg(p.offsets + i + 1) - __ldcg(p.offsets + i);
  __syncthreads();
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) {
    const int lo = s.poff[i], hi = s.poff[i + 1], c = s.cnt[i];
    if (lo < 0 || hi < lo || (lo & 127) || (hi & 127) || c < 0 || c > hi - lo || hi > p.cap) s.bad_offsets = 1;
  }
  if (warp == 0) {
    // tiles per expert = chunks * weight blocks; exclusive scan over experts
    int run = 0;
    for (int e0 = 0; e0 < p.E; e0 += 32) {
      const int e = e0 + lane;
      const int v = e < p.E ? ((max(s.cnt[e], 0) + kChunk - 1) / kChunk) * p.n_tiles : 0;
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
  if (threadIdx.x == 32) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 2);
      mbar_init(&s.tempty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.drain[i], 1);
      mbar_init(&s.fin[i], 1);
    }
    mbar_init(&s.img_full, 1);
    mbar_init(&s.img_free, 2);
    mbar_init(&s.dep, 1);
    for (int i = 0; i < kTileQ; ++i) {
      mbar_init(&s.tq_full[i], 1);
      mbar_init(&s.tq_empty[i], 4);
    }
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
  griddep_launch_dependents();
  const uint32_t tmem = s.tmem_base;

  const bool bad = s.bad_offsets != 0;
  if (bad && threadIdx.x == 0) set_status(p.status, MOE_ERR_DEVICE_INDEX);
  const int total = bad ? 0 : s.cum[p.E];
  const int n_static = p.claim ? max(0, total - kPoolPerCta * (int)gridDim.x) : total;
  const int t_lo = (int)(((int64_t)n_static * blockIdx.x) / gridDim.x);
  const int t_hi = (int)(((int64_t)n_static * (blockIdx.x + 1)) / gridDim.x);
  const bool dyn = p.claim != nullptr && n_static < total;
  const int nkb = (p.Kred + 255) >> 8;
  const int ksf4 = p.Kred >> 6;  // k-steps (scale atoms per 128 rows)
  // both issuers take k-blocks only when a tile has an even number of them (with the
  // even ring length, each stage then always has the same issuer)
  const bool two_issuers = sched::stream_two_issuers(nkb);
  static_assert(Cfg<CHUNK>::kStages % 2 == 0, "stages alternate between issuers");
  int* abort_flag = &s.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Under programmatic dependent launch this kernel may start while the previous
    // kernel of the layer is still running.  Only the operand B rows (activations)
    // and their scales come from that kernel.  With early_weights the first ring's
    // worth of weight tiles is requested before griddep_wait(), and their B tiles
    // right after it; the tile walk itself depends on the routing tables, which are
    // complete by then (moe_forward launches this kernel only behind a kernel that
    // waited for them).  L2 does this (it overlaps the tail of L1, which is also
    // streaming weights); L1 does not, since the quantiser before it is a chain of
    // short dependent memory round trips that queueing behind a burst of weight
    // requests would slow down several-fold.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // the first n_pre k-blocks: weights now, B rows once the previous kernel is done
      const int n_pre = p.early_weights ? min(kStages, (t_hi - t_lo) * nkb) : 0;
      int pre_row[kStages];
      int j = 0;  // k-blocks issued
      bool waited = false;
      // One thread per CTA waits for the previous grid; the builder waits on s.dep.
      if (n_pre == 0) {
        griddep_wait();
        mbar_arrive(&s.dep);
        waited = true;
      }
      auto wait_then_issue_pre_b = [&]() {
        griddep_wait();
        mbar_arrive(&s.dep);
        waited = true;
        for (int i = 0; i < j; ++i) tma_load_2d(s.b[i], &tmap_x, &s.full[i], (i % nkb) * 128, pre_row[i]);
      };
      Cursor<CHUNK> cur;
      TileWalk walk{t_lo, t_hi, 0, dyn};
      for (int t; ok && (t = claim_tile(walk, s, p, n_static, total, abort_flag, ok)) >= 0;) {
        int c, n;
        cur.locate(s, p.n_tiles, t, c, n);
        const int e = cur.e;
        const int row_x = s.poff[e] + c * kChunk;
        const uint8_t* sfw_src = p.w_sf + ((int64_t)e * (p.w_rows >> 7) + n) * (int64_t)ksf4 * 512;
        const int yw = kL1 ? e * p.w_rows + n * 64 : e * p.w_rows + n * 128;
        for (int kb = 0; kb < nkb; ++kb) {
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.full[stage], kWStage + kBStage + natoms * 512);
          const int x = kb * 128;
          tma_load_2d(s.w[stage], &tmap_w, &s.full[stage], x, yw);
          if (kL1) tma_load_2d(s.w[stage] + kWStage / 2, &tmap_w, &s.full[stage], x, yw + p.I);
          if (waited)
            tma_load_2d(s.b[stage], &tmap_x, &s.full[stage], x, row_x);
          else
            pre_row[j] = row_x;
          bulk_load(s.sfw[stage], sfw_src + kb * 4 * 512, natoms * 512, &s.full[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          if (++j == n_pre) wait_then_issue_pre_b();
        }
      }
      if (!waited) wait_then_issue_pre_b();  // no k-blocks, or stopped early
      if (!ok || *(volatile int*)abort_flag)
        for (int i = 0; i < kStages; ++i)
          if (j > i) wait_bar_drain(&s.full[i], sched::ring_last_phase((uint32_t)j, i, kStages));
    }
  } else if (warp == 1 || warp == 7) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads issue concurrently (the tensor pipe serves each issuing thread at
    // roughly one instruction per ~130 cycles): issuer r takes the k-blocks with
    // kb % 2 == r of every tile and accumulates into its own 64 columns; the
    // epilogue adds the two partial sums.  With an odd number of k-blocks per tile
    // issuer 0 takes them all and issuer 1 only keeps the per-tile and per-chunk
    // commits.  Each issuer copies the resident activation scales of its own
    // k-blocks during the first tile of a chunk.
    if (lane == 0) {
      const int r = warp == 1 ? 0 : 1;
      bool ok = true;
      int it = 0, ch = -1, last_e = -1, last_c = -1;
      uint32_t g = 0;  // k-blocks of earlier tiles (ring position)
      // shared-memory descriptors of stage 0 / image 0; others are fixed offsets (the
      // start-address field holds address/16 and every address here is below 256 KB)
      const uint64_t dw0 = sdesc_sw128(s.w[0]), db0 = sdesc_sw128(s.b[0]);
      const uint64_t dsf0 = sdesc_sf(s.sfw[0]), dimg0 = sdesc_sf(s.img[0]);
      Cursor<CHUNK> cur;
      TileWalk walk{t_lo, t_hi, 0, dyn};
      for (int t; ok && (t = next_tile(walk, s, abort_flag, p.status)) >= 0; ++it, g += nkb) {
        int c, n;
        cur.locate(s, p.n_tiles, t, c, n);
        bool fresh = false;  // first tile of a chunk: copy this issuer's activation scales
        if (cur.e != last_e || c != last_c) {
          ++ch;
          last_e = cur.e;
          last_c = c;
          fresh = true;
          // this issuer's MMAs reading its old scale columns must finish first; the
          // other issuer never reads them (k-blocks are split by parity)
          if (ch > 0) {
            tc_commit(&s.drain[r]);
            if (!wait_bar_bounded(&s.drain[r], (ch - 1) & 1, abort_flag, p.status)) { ok = false; break; }
          }
          if (!wait_bar_bounded(&s.img_full, ch & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
        }
        const int buf = it % kAccBufs;
        const uint32_t use = (uint32_t)(it / kAccBufs);  // earlier tiles in this buffer
        if (!wait_bar_bounded(&s.tempty[buf], (use & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (2 * buf + r) * kChunk;
        bool first = true;
        for (int kb = sched::stream_first_kb(r, nkb); kb < nkb; kb += sched::stream_kb_step(nkb)) {
          const uint32_t gs = g + kb;
          const int stage = gs % kStages;
          const uint32_t phase = (gs / kStages) & 1;
          const int natoms = min(4, ksf4 - 4 * kb);
          if (!wait_bar_bounded(&s.full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sfw_col = tmem + kSfwBase + 16 * stage;
          const uint32_t sfb_col = tmem + kSfbBase + 16 * kb;
          const uint64_t dsf = dsf0 + (uint64_t)(stage * (kSfwStage >> 4));
          const uint64_t dw = dw0 + (uint64_t)(stage * (kWStage >> 4));
          const uint64_t db = db0 + (uint64_t)(stage * (kBStage >> 4));
          const uint64_t dimg = dimg0 + (uint64_t)(kb * (4 * 512 >> 4));
          if (natoms == 4) {
#pragma unroll
            for (int a = 0; a < 4; ++a) tc_cp_sf(sfw_col + 4 * a, dsf + 32 * a);
            if (fresh) {
#pragma unroll
              for (int a = 0; a < 4; ++a) tc_cp_sf(sfb_col + 4 * a, dimg + 32 * a);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_fp4(d, dw + 2 * kk, db + 2 * kk, kIdesc, sfw_col + 4 * kk, sfb_col + 4 * kk,
                         (!first || kk > 0) ? 1u : 0u);
          } else {
            for (int a = 0; a < natoms; ++a) tc_cp_sf(sfw_col + 4 * a, dsf + 32 * a);
            if (fresh)
              for (int a = 0; a < natoms; ++a) tc_cp_sf(sfb_col + 4 * a, dimg + 32 * a);
            for (int kk = 0; kk < natoms; ++kk)
              tc_mma_fp4(d, dw + 2 * kk, db + 2 * kk, kIdesc, sfw_col + 4 * kk, sfb_col + 4 * kk,
                         (!first || kk > 0) ? 1u : 0u);
          }
          tc_commit(&s.empty[stage]);
          first = false;
        }
        if (!ok) break;
        if (fresh) tc_commit(&s.img_free);  // images may be rebuilt once both issuers' copies are done
        tc_commit(&s.tfull[buf]);  // arrives once this issuer's MMAs of the tile are done
      }
      tc_commit(&s.fin[r]);
      wait_bar_drain(&s.fin[r], 0);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ activation-scale images
    wait_bar_bounded(&s.dep, 0, abort_flag, p.status);  // the scales come from the previous kernel
    // Image row i (16 B) of k-step k: bytes 0..3 the scales of chunk row i, bytes 4..7
    // those of row 32+i (64-slot chunks), the rest zero.  The zeros are written once;
    // every chunk then gathers its 4-byte words with asynchronous copies, all in
    // flight at once (one memory round trip per chunk, not one per k-step batch).
    for (int k = 0; k < ksf4; ++k) *reinterpret_cast<uint4*>(&s.img[k][lane * 16]) = make_uint4(0u, 0u, 0u, 0u);
    int ch = -1, last_e = -1, last_c = -1;
    Cursor<CHUNK> cur;
    TileWalk walk{t_lo, t_hi, 0, dyn};
    for (;;) {
      int t = 0;
      if (lane == 0) t = next_tile(walk, s, abort_flag, p.status);
      t = __shfl_sync(0xFFFFFFFFu, t, 0);
      if (t < 0) break;
      int c, n;
      cur.locate(s, p.n_tiles, t, c, n);
      if (cur.e == last_e && c == last_c) continue;
      ++ch;
      last_e = cur.e;
      last_c = c;
      if (!wait_bar_bounded(&s.img_free, (ch & 1) ^ 1, abort_flag, p.status)) break;
      const int64_t r0 = (int64_t)s.poff[cur.e] + c * kChunk + lane;
      const uint8_t* base0 = p.a_sf + (r0 >> 7) * (int64_t)ksf4 * 512 + (r0 & 31) * 16 + ((r0 >> 5) & 3) * 4;
      for (int k = 0; k < ksf4; ++k) cp_async4(&s.img[k][lane * 16], base0 + k * 512);
      if (kChunk == 64) {
        const int64_t r1 = r0 + 32;
        const uint8_t* base1 = p.a_sf + (r1 >> 7) * (int64_t)ksf4 * 512 + (r1 & 31) * 16 + ((r1 >> 5) & 3) * 4;
        for (int k = 0; k < ksf4; ++k) cp_async4(&s.img[k][lane * 16 + 4], base1 + k * 512);
      }
      cp_async_wait_all();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.img_full);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    // Everything this role reads that the previous kernel wrote (the activation
    // global scale) is read after a tile's accumulators are complete, hence after
    // the producer's griddep_wait(); the routing tables are older than that kernel.
    const int q = warp & 3;           // TMEM lane quarter = weight rows 32q..32q+31
    const int tid = threadIdx.x - 64; // 0..127 over the four epilogue warps
    int it = 0;
    Cursor<CHUNK> cur;
    float amax = 0.0f;
    TileWalk walk{t_lo, t_hi, 0, dyn};
    for (;; ++it) {
      int t;
      if (walk.t < walk.hi) {
        t = walk.t++;
      } else if (!walk.dyn) {
        t = -1;
      } else {  // one thread reads the queue entry for the four warps
        if (tid == 0) s.epi_tile = next_tile(walk, s, abort_flag, p.status);
        epi_bar();
        t = *reinterpret_cast<volatile int*>(&s.epi_tile);
        if (t < 0) walk.dyn = false;
      }
      if (t < 0) break;
      int c, n;
      cur.locate(s, p.n_tiles, t, c, n);
      const int e = cur.e;
      const int cnt_c = min(kChunk, s.cnt[e] - c * kChunk);  // valid slots of this chunk
      const int64_t row0 = (int64_t)s.poff[e] + c * kChunk;
      // per-slot scatter targets, fetched while the MMAs run: lane i holds slot i (+32)
      int32_t tok_l[kChunk / 32];
      float w_l[kChunk / 32];
      if (KIND == kL2Scatter) {
#pragma unroll
        for (int h = 0; h < kChunk / 32; ++h) {
          const bool v = 32 * h + lane < cnt_c;
          tok_l[h] = v ? __ldg(p.slot_token + row0 + 32 * h + lane) : -1;
          w_l[h] = v ? __ldg(p.slot_weight + row0 + 32 * h + lane) : 0.0f;
        }
      }
      const int buf = it % kAccBufs;
      wait_bar_bounded(&s.tfull[buf], (uint32_t)(it / kAccBufs) & 1, abort_flag, p.status);
      // every epilogue warp has arrived; all of them leave if any of them saw an abort
      if (epi_bar_any(*(volatile int*)abort_flag != 0)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + 2 * buf * kChunk;
      float v[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; j += 16) tmem_ld16(taddr + j, *reinterpret_cast<float(*)[16]>(&v[j]));
      if (two_issuers) {  // partial sum of the odd k-blocks
#pragma unroll
        for (int j = 0; j < kChunk; j += 16) {
          float y[16];
          tmem_ld16(taddr + kChunk + j, y);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[j + i] = __fadd_rn(v[j + i], y[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.tempty[buf]);  // accumulators free: values are in registers

      if (kL1) {
        const float gs_a = __ldg(p.gs_a);
        const bool up = q >= 2;
        const float alpha = __fmul_rn(gs_a, __ldg((up ? p.gs_w1 : p.gs_w0) + e));
        const int col = (q & 1) * 32 + lane;  // h column within the 64-column block
        uint16_t (*x)[kStageLd] = up ? s.xu : s.xg;
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          if (j < cnt_c) x[j][col] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(alpha, v[j])));
        epi_bar();  // exchange complete
        // thread -> (slot, part): 128 threads over CHUNK slots x 64 columns; each part is
        // NB 16-column blocks
        constexpr int kParts = 128 / kChunk;      // 2 (64-slot chunk) or 4 (32-slot chunk)
        constexpr int NB = 4 / kParts;            // 2 or 1 blocks per thread
        constexpr int NC = 16 * NB;               // 32 or 16 columns per thread
        const int sl = tid / kParts, hb = tid % kParts;
        if (sl < cnt_c) {
          const int64_t prow = row0 + sl;
          const int hcol = n * 64 + hb * NC;
          float g[NC], u[NC];
#pragma unroll
          for (int i = 0; i < NC; i += 2) {
            const uint32_t gw = *reinterpret_cast<const uint32_t*>(&s.xg[sl][hb * NC + i]);
            const uint32_t uw = *reinterpret_cast<const uint32_t*>(&s.xu[sl][hb * NC + i]);
            g[i] = bf16lo(gw); g[i + 1] = bf16hi(gw);
            u[i] = bf16lo(uw); u[i + 1] = bf16hi(uw);
          }
          if (KIND == kL1GateUp) {
            uint4* dg = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + hcol);
            uint4* du = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + p.I + hcol);
#pragma unroll
            for (int i = 0; i < NC / 8; ++i) {
              dg[i] = make_uint4(pack_bf16x2(g[8 * i], g[8 * i + 1]), pack_bf16x2(g[8 * i + 2], g[8 * i + 3]),
                                 pack_bf16x2(g[8 * i + 4], g[8 * i + 5]), pack_bf16x2(g[8 * i + 6], g[8 * i + 7]));
              du[i] = make_uint4(pack_bf16x2(u[8 * i], u[8 * i + 1]), pack_bf16x2(u[8 * i + 2], u[8 * i + 3]),
                                 pack_bf16x2(u[8 * i + 4], u[8 * i + 5]), pack_bf16x2(u[8 * i + 6], u[8 * i + 7]));
            }
          } else {
            float h[NC];
#pragma unroll
            for (int i = 0; i < NC; ++i) h[i] = silu_mul(g[i], u[i]);
            if (KIND == kL1Silu) {
              uint4* dh = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_bf16) + prow * p.out_ld + hcol);
#pragma unroll
              for (int i = 0; i < NC / 8; ++i)
                dh[i] = make_uint4(pack_bf16x2(h[8 * i], h[8 * i + 1]), pack_bf16x2(h[8 * i + 2], h[8 * i + 3]),
                                   pack_bf16x2(h[8 * i + 4], h[8 * i + 5]), pack_bf16x2(h[8 * i + 6], h[8 * i + 7]));
#pragma unroll
              for (int i = 0; i < NC; ++i) amax = fmaxf(amax, fabsf(h[i]));
            } else {
              const float rg = recip_global_scale(__ldg(p.gs_h));
              uint32_t sfw = 0, cw[2 * NB];
#pragma unroll
              for (int b = 0; b < NB; ++b) {  // 16-element blocks
                float bm = 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(h[16 * b + i]));
                float rb;
                sfw |= block_scale(bm, rg, rb) << (8 * b);
#pragma unroll
                for (int w4 = 0; w4 < 2; ++w4) {
                  uint32_t word = 0;
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float lo = h[16 * b + 8 * w4 + 2 * i], hi = h[16 * b + 8 * w4 + 2 * i + 1];
                    const uint32_t byte =
                        e2m1x2(code_mag(lo, rg, rb), code_mag(hi, rg, rb));  // signed: sign kept
                    word |= byte << (8 * i);
                  }
                  cw[2 * b + w4] = word;
                }
              }
              uint8_t* hp = p.h_fp4 + prow * (p.I >> 1) + (hcol >> 1);
              uint8_t* sp = p.h_sf + sf_swizzle_offset(prow, hcol >> 4, p.I >> 4);
              if (NB == 2) {
                *reinterpret_cast<uint4*>(hp) = make_uint4(cw[0], cw[1], cw[2 % (2 * NB)], cw[3 % (2 * NB)]);
                *reinterpret_cast<uint16_t*>(sp) = (uint16_t)sfw;
              } else {
                *reinterpret_cast<uint2*>(hp) = make_uint2(cw[0], cw[1]);
                *sp = (uint8_t)sfw;
              }
            }
          }
        }
        epi_bar();  // exchange buffers may be overwritten by the next tile
      } else {
        const float alpha = __fmul_rn(__ldg(p.gs_a), __ldg(p.gs_w0 + e));
        const int col = n * 128 + q * 32 + lane;  // output column
        if (KIND == kL2Rows) {
#pragma unroll
          for (int j = 0; j < kChunk; ++j) {
            if (j < cnt_c) {  // uniform across the warp
              const float y = round_bf16(__fmul_rn(alpha, v[j]));
              reinterpret_cast<__nv_bfloat16*>(p.out_bf16)[(row0 + j) * p.out_ld + col] = __float2bfloat16_rn(y);
            }
          }
        } else {
          // Weighted scatter, four slots at a time: lane l holds column col of every slot;
          // the products are exchanged so that lane l adds columns 4(l%8)..4(l%8)+3 of
          // slot j0 + l/8 with one vector reduction (a quarter of the atomic operations).
          const int sub = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll
          for (int j0 = 0; j0 < kChunk; j0 += 4) {
            if (j0 < cnt_c) {  // uniform across the warp
              float pr[4];
              int32_t tk[4];
#pragma unroll
              for (int s4 = 0; s4 < 4; ++s4) {
                const int j = j0 + s4;
                tk[s4] = __shfl_sync(0xFFFFFFFFu, tok_l[j >> 5], j & 31);
                const float wt = __shfl_sync(0xFFFFFFFFu, w_l[j >> 5], j & 31);
                pr[s4] = __fmul_rn(wt, round_bf16(__fmul_rn(alpha, v[j])));
              }
              float a[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float x0 = __shfl_sync(0xFFFFFFFFu, pr[0], c4 + i);
                const float x1 = __shfl_sync(0xFFFFFFFFu, pr[1], c4 + i);
                const float x2 = __shfl_sync(0xFFFFFFFFu, pr[2], c4 + i);
                const float x3 = __shfl_sync(0xFFFFFFFFu, pr[3], c4 + i);
                a[i] = sub == 0 ? x0 : sub == 1 ? x1 : sub == 2 ? x2 : x3;
              }
              const int32_t tok = sub == 0 ? tk[0] : sub == 1 ? tk[1] : sub == 2 ? tk[2] : tk[3];
              if (j0 + sub < cnt_c) {
                if (tok >= p.T) {
                  set_status(p.status, MOE_ERR_DEVICE_INDEX);
                } else if (tok >= 0) {
                  atomicAdd(reinterpret_cast<float4*>(p.out32 + (int64_t)tok * p.out_cols + n * 128 + q * 32 + c4),
                            make_float4(a[0], a[1], a[2], a[3]));
                }
              }
            }
          }
        }
      }
    }
    if (KIND == kL1Silu && p.h_amax) {
      const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax));
      if (lane == 0 && mb) atomicMax(reinterpret_cast<uint32_t*>(p.h_amax), mb);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int KIND, int CHUNK>
static moe_status launch_chunk(const CUtensorMap& tw, const CUtensorMap& tx, const Params& p, cudaStream_t st,
                               bool pdl) {
  constexpr size_t kSmemBytes = sizeof(Smem<CHUNK>) + 1024;
  static PerDeviceOnce configured;
  if (configured.run([] {
        return cudaFuncSetAttribute(stream_gemm_kernel<KIND, CHUNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
      }) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_ex(stream_gemm_kernel<KIND, CHUNK>, num_sms(), kThreads, kSmemBytes, st, pdl, tw, tx, p) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

template <int KIND>
static moe_status launch_kind(const CUtensorMap& tw, const CUtensorMap& tx, const Params& p, int chunk,
                              cudaStream_t st, bool pdl) {
  return chunk == 32 ? launch_chunk<KIND, 32>(tw, tx, p, st, pdl) : launch_chunk<KIND, 64>(tw, tx, p, st, pdl);
}

}  // namespace stream

bool stream_gemm_supported(int Kred) { return Kred <= 64 * stream::kMaxKSteps; }

moe_status launch_stream_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a, const int32_t* offsets,
                                 const int32_t* padded_offsets, int E, int64_t cap, int K, int I,
                                 const uint8_t* w1_fp4, const uint8_t* w1_sf, const float* gs_g, const float* gs_u,
                                 int epilogue, void* out_bf16, float* h_amax, uint8_t* h_fp4, uint8_t* h_sf,
                                 const float* gs_h, int32_t* status, cudaStream_t st, bool pdl,
                                 int32_t* tile_claim) {
  using namespace stream;
  const int chunk = stream_chunk(cap, E);
  CUtensorMap tw, tx;
  if (!make_tmap(&tw, w1_fp4, (uint64_t)K / 2, (uint64_t)E * 2 * I, 64)) return MOE_ERR_CUDA;
  if (!make_tmap(&tx, a_fp4, (uint64_t)K / 2, (uint64_t)cap, chunk)) return MOE_ERR_CUDA;
  Params p{};
  p.a_sf = a_sf;
  p.w_sf = w1_sf;
  p.offsets = offsets;
  p.padded_offsets = padded_offsets;
  p.E = E;
  p.Kred = K;
  p.n_tiles = I / 64;
  p.w_rows = 2 * I;
  p.I = I;
  p.gs_a = gs_a;
  p.gs_w0 = gs_g;
  p.gs_w1 = gs_u;
  p.out_bf16 = out_bf16;
  p.out_ld = epilogue == MOE_L1_GATEUP_BF16 ? 2 * (int64_t)I : I;
  p.h_amax = h_amax;
  p.h_fp4 = h_fp4;
  p.h_sf = h_sf;
  p.gs_h = gs_h;
  p.cap = cap;
  p.status = status;
  p.claim = tile_claim;
  if (epilogue == MOE_L1_SILU_BF16 && h_amax) {
    if (cudaMemsetAsync(h_amax, 0, sizeof(float), st) != cudaSuccess) return MOE_ERR_CUDA;
    pdl = false;  // the predecessor is now the memset, not a kernel
  }
  switch (epilogue) {
    case MOE_L1_GATEUP_BF16: return launch_kind<kL1GateUp>(tw, tx, p, chunk, st, pdl);
    case MOE_L1_SILU_BF16: return launch_kind<kL1Silu>(tw, tx, p, chunk, st, pdl);
    case MOE_L1_SILU_REQUANT: return launch_kind<kL1Requant>(tw, tx, p, chunk, st, pdl);
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status launch_stream_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h, const int32_t* offsets,
                                 const int32_t* padded_offsets, int E, int64_t cap, int I, int K,
                                 const uint8_t* w2_fp4, const uint8_t* w2_sf, const float* gs_w2, int epilogue,
                                 void* y_rows, const int32_t* slot_token, const float* slot_weight, float* out32,
                                 int64_t T, int32_t* status, cudaStream_t st, bool pdl, int32_t* tile_claim) {
  using namespace stream;
  const int chunk = stream_chunk(cap, E);
  CUtensorMap tw, tx;
  if (!make_tmap(&tw, w2_fp4, (uint64_t)I / 2, (uint64_t)E * K, 128)) return MOE_ERR_CUDA;
  if (!make_tmap(&tx, h_fp4, (uint64_t)I / 2, (uint64_t)cap, chunk)) return MOE_ERR_CUDA;
  Params p{};
  p.a_sf = h_sf;
  p.w_sf = w2_sf;
  p.offsets = offsets;
  p.padded_offsets = padded_offsets;
  p.E = E;
  p.Kred = I;
  p.early_weights = 1;
  p.n_tiles = K / 128;
  p.w_rows = K;
  p.I = I;
  p.gs_a = gs_h;
  p.gs_w0 = gs_w2;
  p.out_bf16 = y_rows;
  p.out_ld = K;
  p.slot_token = slot_token;
  p.slot_weight = slot_weight;
  p.out32 = out32;
  p.T = T;
  p.out_cols = K;
  p.cap = cap;
  p.status = status;
  p.claim = tile_claim;
  switch (epilogue) {
    case MOE_L2_ROWS_BF16: return launch_kind<kL2Rows>(tw, tx, p, chunk, st, pdl);
    case MOE_L2_SCATTER: return launch_kind<kL2Scatter>(tw, tx, p, chunk, st, pdl);
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace moe
