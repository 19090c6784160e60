// Which thread of a grouped-GEMM kernel waits on which pipeline barrier, and on which
// use of it.  Kept apart from the kernels so that a host program can enumerate the
// schedules: an mbarrier wait tests only the parity of a phase, so every barrier is
// waited on by one thread that passes each of its phases in order (or by threads that
// each pass every phase).  A waiter that skipped phases -- alternate uses of one
// barrier shared by two threads -- could pass two uses early once loads complete out
// of order.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {
namespace sched {

// CTA-pair kernel.  g counts the k-blocks (ring stages) the pair has issued; the ring
// has `stages` entries (an odd number).  Stage g's scale atoms are copied by copier
// pair_copier(g), which waits on its own sf_full barrier of ring entry
// pair_stage(g); g is that barrier's use pair_sf_use(g) (phase parity = use & 1).
MOE_HD int pair_copier(uint32_t g) { return (int)(g & 1u); }
MOE_HD uint32_t pair_stage(uint32_t g, int stages) { return g % (uint32_t)stages; }
MOE_HD uint32_t pair_sf_use(uint32_t g, int stages) { return g / (2u * (uint32_t)stages); }

// Streaming kernel.  A tile has nkb k-blocks; issuer r (0 or 1) takes k-blocks
// stream_first_kb(r, nkb), + stream_kb_step(nkb), ... below nkb.  Both issuers take
// k-blocks only for an even nkb: then, with an even ring, each ring entry always has
// the same issuer.  For an odd nkb issuer 0 takes them all.
MOE_HD bool stream_two_issuers(int nkb) { return nkb % 2 == 0; }
MOE_HD int stream_first_kb(int r, int nkb) { return stream_two_issuers(nkb) ? r : (r == 0 ? 0 : nkb); }
MOE_HD int stream_kb_step(int nkb) { return stream_two_issuers(nkb) ? 2 : 1; }

// Producers issue ring stages in order: the k-th stage (k = 0, 1, ...) goes to entry
// k % stages with phase parity (k / stages) & 1.  After n stages, the parity of entry i's
// last use (for n > i) -- what a teardown waits for -- is ring_last_phase(n, i, stages),
// so the producer keeps a count instead of a per-entry record.
MOE_HD uint32_t ring_last_phase(uint32_t n, int i, int stages) {
  return ((n - 1u - (uint32_t)i) / (uint32_t)stages) & 1u;
}

}  // namespace sched
}  // namespace moe
