/*
 * moe_stage.h -- C ABI of the NVFP4 routed-expert MoE stage for GB300 (sm_103a).
 *
 * The layer this library computes is the one described on the nvfp4-megamoe-kernel
 * commit pages (commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py, of src, of
 * vllm/nvfp4_cutedsl.py and of tests):
 *
 *   x (BF16) --global scale amax/2688--> NVFP4 (E2M1 codes + UE4M3 block scales, 16/block)
 *     --route (token,k) pairs to experts--> slot rows grouped by expert
 *     --L1 grouped GEMM [gate|up], alpha = gs_x * gs_w--> BF16 g, u
 *     --SiLU(g) * u--> BF16 h --requantise--> NVFP4
 *     --L2 grouped GEMM (down), alpha = gs_h * gs_w2--> BF16 y
 *     --scatter-add weighted by the routing weights--> rank-local output (BF16).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Memory: every pointer argument is DEVICE memory owned by the caller, unless
 *    the argument says otherwise.  The library never allocates, frees or caches
 *    device memory; scratch space is the caller's `ws` buffer, sized by the
 *    *_workspace_size queries.  All buffers must be 256-byte aligned except where
 *    noted (BF16 tensors: 16 bytes).
 *  - Work is enqueued on the caller's stream, never synchronises the host, and
 *    can be captured into a CUDA graph (no host reads of device data).
 *  - Devices: every call runs on the current device.  Launch settings (the SM
 *    count, the kernels' shared-memory opt-ins, the CTA-pair kernel's grid) are
 *    looked up on the first call on each device and kept per device (thread-safe),
 *    so one process may drive several devices, from several host threads.  Make the
 *    first call of each entry point on a device outside stream capture.
 *  - Return value: MOE_OK, or an error found on the host before anything was
 *    enqueued (MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_WORKSPACE),
 *    or MOE_ERR_CUDA if a launch failed.
 *  - Device-side errors (a bounded wait that gave up, an index that failed its
 *    bounds check) are written to the optional `dev_status` word (int32, device
 *    memory; first error wins, never cleared by the library) and the kernel
 *    returns early.  Read it after synchronising.
 *  - Byte formats: NVFP4 codes are sign-magnitude E2M1 nibbles, two per byte,
 *    the even-K element in the low nibble.  Block scales are UE4M3 (float8 e4m3fn,
 *    sign 0) bytes, one per 16 consecutive elements along the contraction axis.
 *    "Swizzled" scales use the block-scaled MMA layout: 512-byte atoms of 128 rows
 *    x 4 scale columns, offset in atom = 16*(m%32) + 4*((m/32)%4) + (k%4), atom
 *    index = (m/128)*(K/64) + k/4.
 */
#ifndef MOE_STAGE_H
#define MOE_STAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* moe_stream_t;

typedef int moe_status;
#define MOE_OK                    0
#define MOE_ERR_INVALID_ARG       1  /* null pointer, bad enum, misalignment, negative size */
#define MOE_ERR_UNSUPPORTED_SHAPE 2  /* K % 128, I % 64, E > 256, topk > 32, ... */
#define MOE_ERR_WORKSPACE         3  /* ws_bytes smaller than the size query's answer */
#define MOE_ERR_CUDA              4  /* a CUDA launch or tensor-map encode failed */
#define MOE_ERR_TIMEOUT           5  /* device: a bounded wait gave up (dev_status only) */
#define MOE_ERR_DEVICE_INDEX      6  /* device: an index failed its bounds check (dev_status only) */

/* Text for a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Rows of one MMA tile: each expert's slot range is padded to a multiple of it. */
#define MOE_TILE_M 128

/* Scale layouts for moe_stage_activation. */
#define MOE_SF_ROWMAJOR 0  /* [rows, K/16] bytes */
#define MOE_SF_SWIZZLED 1  /* MMA layout, rows padded to 128 */

/* Weight kinds for moe_prepare_weights. */
#define MOE_PREP_W1 0      /* gate|up projection, [E, 2I, K]  */
#define MOE_PREP_W2 1      /* down projection,    [E, K, I]   */

/* L1 epilogues. */
#define MOE_L1_GATEUP_BF16   0  /* store g | u as BF16 [slots, 2I] */
#define MOE_L1_SILU_BF16     1  /* store h = bf16(silu(g)*u) [slots, I] and max|h| */
#define MOE_L1_SILU_REQUANT  2  /* quantise h with a fixed global scale to NVFP4 */

/* L2 epilogues. */
#define MOE_L2_ROWS_BF16 0      /* store y as BF16 [slots, K] */
#define MOE_L2_SCATTER   1      /* out32[token] += weight * y (fp32 atomics) */

/* Global-scale modes for the requantised activation h in moe_forward. */
#define MOE_GS_DYNAMIC 0        /* gs_h = max|h| / 2688 over this call's slots */
#define MOE_GS_FIXED   1        /* gs_h supplied by the caller (calibrated) */

/* ------------------------------------------------------------------------- */
/* Size queries (host only, no device work).                                  */
/* ------------------------------------------------------------------------- */

/* Slot capacity for T tokens, top-k and E local experts: an upper bound on the
 * padded slot count, T*topk + 127*E rounded up to a multiple of 128.  Every
 * slot-indexed buffer (slot_token, slot_weight, activation/h codes and scales)
 * holds this many rows.  Returns -1 on bad arguments. */
int64_t moe_slot_capacity(int64_t T, int topk, int E);

/* Scratch bytes moe_route needs. */
size_t moe_route_workspace_size(int64_t T, int topk, int E);

/* Scratch bytes moe_stage_activation / moe_stage_activation_to_slots need. */
size_t moe_stage_workspace_size(void);

/* Scratch bytes moe_forward needs for up to T_max tokens. */
size_t moe_workspace_size(int64_t T_max, int K, int I, int E, int topk);

/* ------------------------------------------------------------------------- */
/* Setup (not on the per-call path)                                          */
/* ------------------------------------------------------------------------- */

/* Rearrange weight block scales into the layout the grouped GEMMs read.
 * Source: the tests-page "scale transpose" commit -- checkpoint weight scales
 * are (N, K_sf) row-major per expert.
 *   sf_rowmajor: [E, N, K/16] UE4M3 bytes (N = 2I for MOE_PREP_W1, rows 0..I-1
 *                gate and I..2I-1 up; N = K_out for MOE_PREP_W2).
 *   sf_prepared: E*N*K/16 bytes, written.  For MOE_PREP_W2 it is the swizzled
 *                layout of each expert's [N, K/16] matrix.  For MOE_PREP_W1 the
 *                rows are first regrouped so that every 128-row atom holds 64
 *                gate rows followed by the 64 matching up rows (the L1 tile
 *                computes 64 h columns from both halves).
 *   N % 128 == 0, K % 64 == 0.  Buffers may be any alignment. */
moe_status moe_prepare_weights(const uint8_t* sf_rowmajor, uint8_t* sf_prepared,
                               int E, int N, int K, int kind, moe_stream_t stream);

/* Quantise a rank's BF16 expert weights to the form the layer consumes, on the device
 * (the pages' finalize_weights / weight_transform step, for BF16 inputs): per expert,
 * the gate rows, the up rows and the down projection each get their own global scale
 * (amax / 2688) and are block-quantised as moe_stage_activation does; the scales are
 * then rearranged as moe_prepare_weights does.
 *   w1: [E, 2I, K] BF16 (gate rows 0..I-1, up rows I..2I-1), w2: [E, K, I] BF16,
 *       16-byte aligned (device).
 *   w1_fp4 [E, 2I, K/2], w2_fp4 [E, K, I/2]: codes; w1_sf, w2_sf: E*2I*K/16 and
 *       E*K*I/16 bytes in the GEMMs' layouts; gs_w1_gate, gs_w1_up, gs_w2: [E] fp32.
 *   ws: moe_quantize_weights_workspace_size(E, I, K) bytes of scratch (the row-major
 *       scales pass through it).
 *   I % 64 == 0, K % 128 == 0.  Stream-ordered, no host sync; set-up, not timed. */
size_t moe_quantize_weights_workspace_size(int E, int I, int K);
moe_status moe_quantize_weights(const void* w1, const void* w2, int E, int I, int K,
                                uint8_t* w1_fp4, uint8_t* w1_sf, float* gs_w1_gate, float* gs_w1_up,
                                uint8_t* w2_fp4, uint8_t* w2_sf, float* gs_w2,
                                void* ws, size_t ws_bytes, moe_stream_t stream);

/* The pages' one-alpha handling of W1's two global scales (commits of
 * vllm/nvfp4_cutedsl.py, "dual global scale"): per expert e, with c = max(gs_gate[e],
 * gs_up[e]), every block scale s of the half whose global scale g is smaller becomes
 * the UE4M3 value nearest to s * (g / c) (fp32 division, fp32 multiply, round to
 * nearest even, saturating); gs_common[e] = c.  The L1 GEMM then takes gs_common as
 * both its gate and up weight scales.  The layer's own path keeps two exact alphas;
 * this is the compatibility form, for the accuracy comparison.
 *   w1_sf:      [E, 2I, K/16] UE4M3 bytes, row-major (before moe_prepare_weights),
 *               gate rows 0..I-1, up rows I..2I-1; folded in place (device).
 *   gs_gate, gs_up: [E] fp32 (device); gs_common: [E] fp32 (device), written.
 *   Experts whose two scales are equal or both zero are unchanged.  I > 0,
 *   K % 16 == 0; MOE_ERR_INVALID_ARG for NULL pointers or non-positive sizes. */
moe_status moe_fold_gate_up_scales(uint8_t* w1_sf, const float* gs_gate, const float* gs_up,
                                   float* gs_common, int E, int I, int K, moe_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Per-call path                                                              */
/* ------------------------------------------------------------------------- */

/* Quantise a BF16 tensor to NVFP4 (stage_activation of the nvfp4_mega_moe.py
 * commits: returns codes, scales and the global scale).
 *   x:        [T, K] BF16, row stride ld_x elements (ld_x >= K, ld_x % 8 == 0).
 *   x_fp4:    [T, K/2] codes, written.
 *   x_sf:     MOE_SF_ROWMAJOR: [T, K/16]; MOE_SF_SWIZZLED: ceil(T/128)*128*K/16.
 *   gs_out:   one fp32, written with the global scale used.
 *   gs_fixed: NULL -> gs = max|x| / 2688 (two passes over x); else one fp32
 *             holding a fixed global scale (one pass; the calibrated mode of the
 *             vllm/nvfp4_cutedsl.py commits).
 *   Arithmetic (fp32, round-to-nearest-even): rg = 1/gs (saturated to FLT_MAX);
 *   per 16-block s = (max|x|*rg)/6 -> UE4M3 (RNE, saturating at 448); each
 *   element (|x|*rg) * (1/decode(s)) -> nearest E2M1 (ties to even, saturating
 *   at 6); bit 3 = sign bit of x; a zero scale gives sign-only nibbles.
 *   K % 64 == 0.  ws: moe_stage_workspace_size() bytes. */
moe_status moe_stage_activation(const void* x, int64_t T, int K, int64_t ld_x,
                                uint8_t* x_fp4, uint8_t* x_sf, int sf_layout,
                                float* gs_out, const float* gs_fixed,
                                void* ws, size_t ws_bytes, int32_t* dev_status,
                                moe_stream_t stream);

/* The same quantisation, written straight into the slot rows the router chose
 * (the activation gather of the src commits fused into the quantiser):
 * token t's codes go to every slot pair_slot[t*topk + j] >= 0.
 *   a_fp4: [capacity, K/2]; a_sf: capacity*K/16 bytes, swizzled.
 *   Padding slot rows are not written (the GEMMs never read them into valid
 *   outputs). */
moe_status moe_stage_activation_to_slots(const void* x, int64_t T, int K, int64_t ld_x,
                                         const int32_t* pair_slot, int topk, int64_t capacity,
                                         uint8_t* a_fp4, uint8_t* a_sf,
                                         float* gs_out, const float* gs_fixed,
                                         void* ws, size_t ws_bytes, int32_t* dev_status,
                                         moe_stream_t stream);

/* Route (token, k) pairs to expert-grouped slots (the slot routing of the src and
 * vllm/nvfp4_cutedsl.py commits: local ids, bincount + cumsum offsets in int32,
 * stable grouping by expert, zero-weight padding).
 *   topk_ids [T, topk] int32 GLOBAL expert ids; local = id - expert_offset; pairs
 *   with local outside [0, E) are dropped.  topk_w [T, topk] fp32.
 *   Outputs (all written): counts [E], offsets [E+1] (exclusive cumsum of counts),
 *   padded_offsets [E+1] (cumsum of counts rounded up to 128), slot_token
 *   [capacity] (token of each slot, -1 for padding), slot_weight [capacity] (0 for
 *   padding), pair_slot [T*topk] (slot of each pair, -1 if dropped).  Within an
 *   expert, slots follow ascending t*topk + j.
 *   capacity >= moe_slot_capacity(T, topk, E).  E <= 256, topk <= 32.
 *   ws: moe_route_workspace_size(T, topk, E) bytes. */
moe_status moe_route(const int32_t* topk_ids, const float* topk_w, int64_t T, int topk,
                     int E, int expert_offset,
                     int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                     int32_t* slot_token, float* slot_weight, int32_t* pair_slot,
                     int64_t capacity, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route for callers that cannot allocate (the commit pages have no
 * counterpart: this is an addition of this library).  Some callers have no
 * allocator at hand when they route: a plugin whose host runtime owns all
 * device memory and passes in only the call's tensors, or a serving loop that
 * must never allocate on its hot path.  This entry point takes the same
 * arguments as moe_route minus ws/ws_bytes, writes the same outputs (bit for
 * bit), and allocates nothing: its two scratch tables live in a fixed array in
 * the library's own device memory, 2 * MOE_ROUTE_STATIC_TABLE_INTS int32
 * (2 MiB), held by every GPU that loads the library until the process exits.
 *   Limit: ceil(T*topk/256) * E <= MOE_ROUTE_STATIC_TABLE_INTS (for E = 48 about
 *   1.39 million (token, k) pairs); larger calls return MOE_ERR_UNSUPPORTED_SHAPE
 *   without enqueuing anything.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before capturing a
 *   stream.  The address is kept for the life of the process: a device or primary
 *   context reset (cudaDeviceReset) after that first call is not supported, since
 *   the library's module may be reloaded at another address.
 *   Every call shares the one array.  Calls ordered on one stream are safe; calls
 *   that can overlap on the GPU (other streams, other host threads) race on it and
 *   corrupt each other's routing.  Nothing needs clearing between calls: both
 *   tables are rewritten in full before they are read. */
#define MOE_ROUTE_STATIC_TABLE_INTS 262144
moe_status moe_route_static_scratch(const int32_t* topk_ids, const float* topk_w, int64_t T, int topk,
                                    int E, int expert_offset,
                                    int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                                    int32_t* slot_token, float* slot_weight, int32_t* pair_slot,
                                    int64_t capacity, moe_stream_t stream);

/* L1 grouped GEMM, gate|up (nvfp4_mega_moe_l1 of the nvfp4_mega_moe.py commits;
 * split at I per the vllm/nvfp4_cutedsl.py "intermediate_size" commit).
 * For every expert e and slot row p in [padded_offsets[e], padded_offsets[e] +
 * offsets[e+1] - offsets[e]):
 *   acc[p, n] = sum_k deq(A)[p, k] * deq(W1[e])[n, k]     (fp32 accumulate)
 *   g = bf16(gs_a * gs_w1_gate[e] * acc[:, 0:I]),  u = bf16(gs_a * gs_w1_up[e] * acc[:, I:2I])
 *   a_fp4 [capacity, K/2], a_sf swizzled (capacity*K/16); gs_a one fp32.
 *   w1_fp4 [E, 2I, K/2]; w1_sf prepared by moe_prepare_weights(MOE_PREP_W1).
 *   epilogue:
 *     MOE_L1_GATEUP_BF16: out_bf16 [capacity, 2I] gets g | u.
 *     MOE_L1_SILU_BF16:   out_bf16 [capacity, I] gets h = bf16(silu(g)*u),
 *                         silu(g) = g/(1+exp(-g)) in fp32; if h_amax != NULL it is
 *                         set to max|h| over valid rows (fp32, zeroed by this call).
 *     MOE_L1_SILU_REQUANT: h is quantised with the fixed global scale *gs_h (as in
 *                         moe_stage_activation) into h_fp4 [capacity, I/2] and
 *                         h_sf (swizzled, capacity*I/16); out_bf16 may be NULL or
 *                         receive h as well.
 *   Rows of padding are never written.  K % 128 == 0, I % 64 == 0, E <= 256:
 *   moe_stage_activation quantises any K % 64 == 0, but the layer's hidden size K is
 *   also the L2 GEMM's output width, which that GEMM covers in tiles of 128 or 256
 *   columns, so the layer entry points (L1, L2, moe_forward) take K % 128 == 0. */
moe_status moe_grouped_gemm_l1(const uint8_t* a_fp4, const uint8_t* a_sf, const float* gs_a,
                               const int32_t* offsets, const int32_t* padded_offsets,
                               int E, int64_t capacity, int K, int I,
                               const uint8_t* w1_fp4, const uint8_t* w1_sf,
                               const float* gs_w1_gate, const float* gs_w1_up,
                               int epilogue, void* out_bf16, float* h_amax,
                               uint8_t* h_fp4, uint8_t* h_sf, const float* gs_h,
                               int32_t* dev_status, moe_stream_t stream);

/* Requantise h [capacity, I] BF16 rows to NVFP4 with gs_h = h_amax[0]/2688
 * (written to gs_h_out), skipping padding rows (slot_token < 0): the
 * stage_activation of h of the nvfp4_mega_moe.py "global scale" commit.
 * h_fp4 [capacity, I/2]; h_sf swizzled.  I % 64 == 0. */
moe_status moe_requant(const void* h, int64_t capacity, int I, const int32_t* slot_token,
                       const float* h_amax, float* gs_h_out, uint8_t* h_fp4, uint8_t* h_sf,
                       int32_t* dev_status, moe_stream_t stream);

/* L2 grouped GEMM, down projection (nvfp4_mega_moe_l2), same slot order as L1:
 *   y[p, n] = bf16(gs_h * gs_w2[e] * sum_i deq(H)[p, i] * deq(W2[e])[n, i])
 *   h_fp4 [capacity, I/2], h_sf swizzled; w2_fp4 [E, K, I/2]; w2_sf prepared
 *   (MOE_PREP_W2).
 *   epilogue MOE_L2_ROWS_BF16: y_rows [capacity, K] BF16.
 *   epilogue MOE_L2_SCATTER: out32[slot_token[p], :] += slot_weight[p] * y[p, :]
 *   (fp32 atomic adds; out32 [T, K] is NOT cleared by this call).
 *   K % 128 == 0, I % 64 == 0. */
moe_status moe_grouped_gemm_l2(const uint8_t* h_fp4, const uint8_t* h_sf, const float* gs_h,
                               const int32_t* offsets, const int32_t* padded_offsets,
                               int E, int64_t capacity, int I, int K,
                               const uint8_t* w2_fp4, const uint8_t* w2_sf, const float* gs_w2,
                               int epilogue, void* y_rows,
                               const int32_t* slot_token, const float* slot_weight,
                               float* out32, int64_t T,
                               int32_t* dev_status, moe_stream_t stream);

/* Which grouped-GEMM kernel moe_grouped_gemm_l1/l2 and moe_forward launch
 * (process-wide setting; returns the previous one; not synchronised with work in
 * flight, so set it between calls):
 *   MOE_GEMM_AUTO      (default) the weight-streaming kernel when the slot capacity
 *                      implies at most 64 slots per local expert on average
 *                      (capacity - 127*E <= 64*E) and the contraction is <= 4096,
 *                      the tiled kernels otherwise (as MOE_GEMM_TILED: L1 on single
 *                      SMs, L2's 256-wide tiles on SM pairs);
 *   MOE_GEMM_TILED     always a tiled kernel, slots on the MMA's M side: L1 in tiles
 *                      of 128 slot rows x 256 weight rows on single SMs; L2 in tiles
 *                      of 256 slot rows x 256 weight rows on pairs of SMs (a cluster
 *                      of two CTAs sharing one M=256 MMA: each SM stages its own 128
 *                      slot rows and half of the weight rows); 128 x 128 tiles on
 *                      single SMs where I % 128 or, for L2, K % 256 leaves no choice;
 *   MOE_GEMM_TILED_1CTA the tiled kernels on single SMs only;
 *   MOE_GEMM_TILED_PAIR the tiled kernels with 256-wide tiles on SM pairs for both
 *                      GEMMs;
 *   MOE_GEMM_STREAMING the weight-streaming kernel whenever the contraction is
 *                      <= 4096: weight rows on the MMA's M side, chunks of slots on
 *                      its N side, the chunk's activation scales resident in tensor
 *                      memory.  Experts with more slots than a chunk are split
 *                      into several chunks; an expert's chunks are processed back to
 *                      back for each weight block, so the repeated weight reads come
 *                      from L2.  The chunk is 32 slots (8 pipeline stages fit);
 *   MOE_GEMM_STREAMING_N32 / _N64  the streaming kernel with the chunk forced.
 * All kernels compute the same arithmetic (results may differ in the fp32
 * summation order only). */
#define MOE_GEMM_AUTO           0
#define MOE_GEMM_TILED          1
#define MOE_GEMM_STREAMING      2
#define MOE_GEMM_STREAMING_N32  3
#define MOE_GEMM_STREAMING_N64  4
#define MOE_GEMM_TILED_1CTA     5
#define MOE_GEMM_TILED_PAIR     6
int moe_set_gemm_policy(int policy);

/* out_bf16[i] = bf16(out32[i]) for i < T*K (round to nearest even). */
moe_status moe_cast_output(const float* out32, void* out_bf16, int64_t T, int K,
                           moe_stream_t stream);

/* Weighted combine of per-slot L2 rows (the scatter_add of the nvfp4-megamoe-kernel
 * pages done per token instead of with atomics):
 *   out_bf16[t, :] = bf16( sum_j w[t, j] * y_rows[pair_slot[t*topk + j], :] )
 * over j = 0 .. topk-1 in that order, in fp32 with each product and each sum
 * rounded (the oracle's combine bit for bit); pairs with slot -1 are skipped, so a
 * token with no local expert gets 0.
 *   y_rows [capacity, ld_y] BF16 (the MOE_L2_ROWS_BF16 output), ld_y >= K, ld_y % 8 == 0;
 *   pair_slot [T*topk] from moe_route; topk_w [T, topk] fp32; out_bf16 [T, K].
 *   K % 8 == 0; y_rows and out_bf16 16-byte aligned.  A slot >= capacity is skipped
 *   and reported as MOE_ERR_DEVICE_INDEX in *dev_status (if not NULL). */
moe_status moe_combine_rows(const void* y_rows, int64_t ld_y, const int32_t* pair_slot,
                            const float* topk_w, int64_t T, int topk, int K, int64_t capacity,
                            void* out_bf16, int32_t* dev_status, moe_stream_t stream);

/* Expert weights of one rank, all device memory. */
typedef struct moe_weights {
    const uint8_t* w1_fp4;      /* [E, 2I, K/2]                          */
    const uint8_t* w1_sf;       /* prepared, MOE_PREP_W1                 */
    const float*   gs_w1_gate;  /* [E]                                   */
    const float*   gs_w1_up;    /* [E]                                   */
    const uint8_t* w2_fp4;      /* [E, K, I/2]                           */
    const uint8_t* w2_sf;       /* prepared, MOE_PREP_W2                 */
    const float*   gs_w2;       /* [E]                                   */
} moe_weights;

/* The whole rank-local layer (nvfp4_moe_full / the CuTeDSL runner's forward):
 * route -> quantise x into slots -> L1 (+SiLU*up, +requant) -> L2 (+weighted
 * scatter) -> BF16 output.  The caller sums outputs across ranks.  While the fp32
 * output accumulator (T*K*4 bytes) is at most 32 MiB the weighted scatter is fused
 * into the L2 epilogue (fp32 atomics, then a cast); above that the L2 GEMM writes
 * BF16 rows and moe_combine_rows' arithmetic produces the output.
 *   x [T, K] BF16 (row stride K); topk_ids/topk_w [T, topk]; out [T, K] BF16.
 *   gs_x_fixed: NULL -> amax of x; else a fixed fp32 global scale.
 *   gs_h_mode MOE_GS_DYNAMIC: gs_h (device fp32) receives max|h|/2688;
 *   MOE_GS_FIXED: gs_h holds the scale to use (h quantised in the L1 epilogue).
 *   ws: moe_workspace_size(T, K, I, E, topk) bytes (T <= the T_max it was sized for).
 *   Tokens none of whose experts are local get 0. */
moe_status moe_forward(const void* x, int64_t T, int K, int I, int E,
                       const int32_t* topk_ids, const float* topk_w, int topk,
                       int expert_offset, const moe_weights* w,
                       const float* gs_x_fixed, int gs_h_mode, float* gs_h,
                       void* out, int32_t* dev_status,
                       void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_forward with stage timestamps, for tracing and roofline measurement.
 * stage_events: NULL, or MOE_TRACE_EVENTS cudaEvent_t handles (created by the
 * caller, with timing enabled) recorded on `stream` at: [0] start, [1] after
 * routing, [2] after quantising x into the slots, [3] after the L1 GEMM,
 * [4] after requantising h (equal to [3] in MOE_GS_FIXED mode), [5] after the
 * L2 GEMM, [6] after the output cast or combine.  While the stream is being captured into
 * a CUDA graph the records become event-record nodes of the graph.  All other
 * arguments and behaviour are those of moe_forward. */
#define MOE_TRACE_EVENTS 7
moe_status moe_forward_traced(const void* x, int64_t T, int K, int I, int E,
                              const int32_t* topk_ids, const float* topk_w, int topk,
                              int expert_offset, const moe_weights* w,
                              const float* gs_x_fixed, int gs_h_mode, float* gs_h,
                              void* out, int32_t* dev_status,
                              void* ws, size_t ws_bytes, void* const* stage_events,
                              moe_stream_t stream);

/* Self-test of the failure reporting the kernels rely on (no counterpart on the commit
 * pages).  Launches one block on `stream` in which thread 0 waits, with the library's
 * bounded mbarrier wait, on a barrier that nothing arrives on, and thread 32 waits on a
 * second such barrier starting half a limit later.  Thread 0 gives up after the wait
 * limit (1 s), sets the block's abort flag and writes MOE_ERR_TIMEOUT to *dev_status
 * (first error wins); thread 32 must then return through the abort flag before its own
 * limit.  dev_result (2 int32, device): [0] = 1 if thread 0 gave up on its limit,
 * [1] = 1 if thread 32 returned through the abort flag.  Nothing waits forever and the
 * context stays usable.  Returns MOE_ERR_INVALID_ARG for NULL pointers, MOE_ERR_CUDA if
 * the launch fails; takes about one second of device time. */
moe_status moe_selftest_bounded_wait(int32_t* dev_status, int32_t* dev_result, moe_stream_t stream);

/* Self-test of the two code encoders (no counterpart on the commit pages; the encodings
 * are those of the pages' "NVFP4 quantisation" commits: E2M1 codes round to the nearest
 * of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with the sign in bit 3, UE4M3 block scales round to
 * nearest and saturate at 448).  For i < n the fp32 value v with bit pattern
 * first_pattern + i is encoded exactly as the quantisers, the requantiser and the L1
 * requant epilogue encode a scaled value and a block scale:
 *   e2m1_codes[i] = E2M1 code of v (round to nearest, ties to the even magnitude index,
 *                   saturating at 6; bit 3 = sign bit of v, also when v rounds to zero);
 *   e4m3_bytes[i] = UE4M3 byte of v (round to nearest even, saturating at 448 = 0x7E;
 *                   defined for v >= 0, the only values the library encodes).
 * NaN patterns give unspecified bytes.  Both outputs are device buffers of n bytes owned
 * by the caller.  Returns MOE_ERR_INVALID_ARG for n < 0, NULL outputs with n > 0, or a
 * range past pattern 0xFFFFFFFF; MOE_ERR_CUDA if the launch fails. */
moe_status moe_selftest_codecs(uint32_t first_pattern, int64_t n, uint8_t* e2m1_codes, uint8_t* e4m3_bytes,
                               moe_stream_t stream);

/* Self-test of the SiLU the L1 epilogues apply (the "complete pipeline" commit of the
 * tests page: h = SiLU(gate) * up in BF16; SiLU(g) = g / (1 + exp(-g))).  For i < n:
 *   silu_out[i] = the fp32 value the epilogue computes for gate value g[i] before it
 *                 multiplies by up and rounds h to BF16 (the fast exp and division
 *                 intrinsics; a few fp32 ulp from the exact value, see the tests).
 * g, silu_out: device fp32 arrays of n elements owned by the caller.  Returns
 * MOE_ERR_INVALID_ARG for n < 0 or NULL arrays with n > 0, MOE_ERR_CUDA if the launch
 * fails. */
moe_status moe_selftest_silu(const float* g, int64_t n, float* silu_out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_STAGE_H */
