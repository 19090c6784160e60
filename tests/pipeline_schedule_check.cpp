// Host check of the grouped-GEMM kernels' barrier schedules, compiled against the same
// schedule functions the kernels call (csrc/pipeline.cuh).  For every waiter and every
// barrier it waits on, the uses it waits for must be 0, 1, 2, ... in order: a wait
// tests only the parity of a phase, so a waiter that skipped a use could pass on an
// older phase of the same parity.  The schedules the kernels had before (one scale
// barrier per ring entry shared by two alternating copiers; two streaming issuers for
// any k-block count) are checked the same way and must show violations, which shows
// the check would have caught them.
//
// Prints one line "violations <schedule> <count>" per schedule.
#include <cstdio>
#include <map>
#include <utility>

#include "../nvfp4_mixture_experts_stage_gb300/csrc/pipeline.cuh"

using moe::sched::pair_copier;
using moe::sched::pair_sf_use;
using moe::sched::pair_stage;
using moe::sched::ring_last_phase;
using moe::sched::stream_first_kb;
using moe::sched::stream_kb_step;

namespace {

// Per (waiter, barrier): the next use the waiter must see.
struct Uses {
  std::map<std::pair<int, long>, long> next;
  long violations = 0;
  void see(int waiter, long barrier, long use) {
    long& n = next[{waiter, barrier}];
    if (use != n) ++violations;
    n = use + 1;
  }
};

// CTA-pair kernel: stages g = 0 .. n-1 of one pair, ring of `stages` entries.
long pair_current(int stages, int n) {
  Uses u;
  for (int c = 0; c < 2; ++c)
    for (int g = c; g < n; g += 2) {  // the copier loop: g = c, c + 2, ...
      if (pair_copier((uint32_t)g) != c) ++u.violations;
      const long barrier = (long)c * stages + pair_stage((uint32_t)g, stages);
      u.see(c, barrier, pair_sf_use((uint32_t)g, stages));
    }
  // the producer arms the barriers in stage order with the same mapping
  for (int g = 0; g < n; ++g)
    u.see(2, (long)pair_copier((uint32_t)g) * stages + pair_stage((uint32_t)g, stages),
          pair_sf_use((uint32_t)g, stages));
  return u.violations;
}

long pair_shared_barrier(int stages, int n) {
  Uses u;
  for (int c = 0; c < 2; ++c)
    for (int g = c; g < n; g += 2) u.see(c, g % stages, g / stages);
  return u.violations;
}

// Streaming kernel: `tiles` tiles of nkb k-blocks, ring of `stages` entries; issuer r
// waits on entry (g + kb) % stages, use (g + kb) / stages, g = tile * nkb.  Also checks
// that the issuers' k-blocks cover each tile exactly once.
long stream_current(int stages, int nkb, int tiles) {
  Uses u;
  for (int t = 0; t < tiles; ++t) {
    int covered[64] = {0};
    for (int r = 0; r < 2; ++r)
      for (int kb = stream_first_kb(r, nkb); kb < nkb; kb += stream_kb_step(nkb)) {
        ++covered[kb];
        const long pos = (long)t * nkb + kb;
        u.see(r, pos % stages, pos / stages);
      }
    for (int kb = 0; kb < nkb; ++kb)
      if (covered[kb] != 1) ++u.violations;
  }
  return u.violations;
}

long stream_always_two(int stages, int nkb, int tiles) {
  Uses u;
  for (int t = 0; t < tiles; ++t)
    for (int r = 0; r < 2; ++r)
      for (int kb = r; kb < nkb; kb += 2) {
        const long pos = (long)t * nkb + kb;
        u.see(r, pos % stages, pos / stages);
      }
  return u.violations;
}

// Producer teardown: after n stages issued in order, the parity of each entry's last use
// from ring_last_phase against a record kept while issuing (also flags a formula that
// forgets the wrap: parity = last stage index & 1 instead of its use & 1).
long ring_teardown(int stages, int n, bool naive) {
  long bad = 0;
  long last[16];
  for (int i = 0; i < stages; ++i) last[i] = -1;
  int stage = 0;
  unsigned phase = 0;
  for (int k = 0; k < n; ++k) {
    last[stage] = phase;
    if (++stage == stages) { stage = 0; phase ^= 1u; }
  }
  for (int i = 0; i < stages; ++i) {
    if (n <= i) continue;
    const unsigned got = naive ? (unsigned)((n - 1 - i) & 1) : ring_last_phase((uint32_t)n, i, stages);
    if ((long)got != last[i]) ++bad;
  }
  return bad;
}

}  // namespace

int main() {
  long cur = 0, old = 0;
  for (int stages : {3, 5, 7})
    for (int n = 0; n <= 400; ++n) {
      cur += pair_current(stages, n);
      old += pair_shared_barrier(stages, n);
    }
  std::printf("violations pair %ld\n", cur);
  std::printf("violations pair_shared_barrier %ld\n", old);
  long scur = 0, sold_odd = 0, sold_even = 0;
  for (int stages : {6, 8})
    for (int nkb = 1; nkb <= 32; ++nkb)
      for (int tiles = 1; tiles <= 12; ++tiles) {
        scur += stream_current(stages, nkb, tiles);
        (nkb % 2 ? sold_odd : sold_even) += stream_always_two(stages, nkb, tiles);
      }
  std::printf("violations stream %ld\n", scur);
  std::printf("violations stream_always_two_odd %ld\n", sold_odd);
  std::printf("violations stream_always_two_even %ld\n", sold_even);
  long rcur = 0, rnaive = 0;
  for (int stages : {4, 5, 6, 8})
    for (int n = 0; n <= 200; ++n) {
      rcur += ring_teardown(stages, n, false);
      rnaive += ring_teardown(stages, n, true);
    }
  std::printf("violations ring_teardown %ld\n", rcur);
  std::printf("violations ring_teardown_naive %ld\n", rnaive);
  return 0;
}
