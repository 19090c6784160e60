"""Token -> slot routing, restated on the CPU (oracle; test infrastructure only).

Sources on the nvfp4-megamoe-kernel commit pages:

* commits of ``src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py``, the
  "global expert ids" commit: top-k ids are global (0..383 for 384 experts);
  rank r owns the 48 experts starting at 48*r and subtracts that offset to get
  local ids; ids of other ranks' experts are not this rank's work.
* commits of ``src``, the "1-D slot_expert_ids and slot_token" commits: the
  grouped GEMM consumes slots (token, k) pairs, grouped by expert, with a
  slot -> token map; with top-1 and tokens already ordered by expert that map
  is the identity.
* commits of ``vllm/nvfp4_cutedsl.py``: the "CUDA graph" commits -- slots are
  ordered by sorting (token, k) pairs by expert, per-expert counts come from a
  bincount and offsets from a cumulative sum kept in int32 on the device, and
  padding slots carry zero routing weight so a combine over all slots is
  harmless.
* commits of ``tests``, the "token layout" commit: the grouped GEMM wants the
  rows laid out as [expert 0 slots | expert 1 slots | ...].

Readings where the pages are silent:

* order within an expert: ascending flat pair index t * topk + j (a stable
  sort; the pages' argsort does not fix the order of equal keys);
* padding: each expert's slot range is padded to a multiple of 128 rows (one
  MMA tile), padded offsets are the cumulative sum of the padded counts;
  padding slots and every slot past the last expert hold token -1 and weight
  0, up to the caller's slot capacity;
* ids outside [offset, offset + E) -- other ranks' experts or invalid ids such
  as -1 -- are dropped and their pair_slot is -1.
"""

import numpy as np

TILE_M = 128


def slot_capacity(T, topk, E):
    """Upper bound on the padded slot count for T tokens, top-k and E experts:
    sum over experts of ceil(count/128)*128 <= T*topk + 127*E, rounded up to a
    whole 128-row tile."""
    n = T * topk + (TILE_M - 1) * E
    return -(-n // TILE_M) * TILE_M


def route(topk_ids, topk_w, E, expert_offset, capacity=None):
    """Route (token, k) pairs to expert-grouped slots.

    topk_ids: [T, topk] int32 global expert ids; topk_w: [T, topk] float32.
    Returns a dict of int32/float32 arrays:
      counts [E], offsets [E+1], padded_offsets [E+1],
      slot_token [capacity], slot_weight [capacity], pair_slot [T*topk].
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    w = np.asarray(topk_w, dtype=np.float32)
    T, k = ids.shape
    if capacity is None:
        capacity = slot_capacity(T, k, E)
    local = (ids - expert_offset).reshape(-1)
    flat = np.arange(T * k)
    valid = (local >= 0) & (local < E)
    counts = np.bincount(local[valid], minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    padded = -(-counts // TILE_M) * TILE_M
    poff = np.concatenate([[0], np.cumsum(padded)])
    if poff[-1] > capacity:
        raise ValueError("slot capacity too small")

    slot_token = np.full(capacity, -1, dtype=np.int32)
    slot_weight = np.zeros(capacity, dtype=np.float32)
    pair_slot = np.full(T * k, -1, dtype=np.int32)

    vflat = flat[valid]
    vlocal = local[valid]
    order = np.lexsort((vflat, vlocal))  # primary key: local expert; then flat index
    sorted_flat = vflat[order]
    sorted_local = vlocal[order]
    rank = np.arange(sorted_flat.size) - offsets[sorted_local]
    slots = poff[sorted_local] + rank
    slot_token[slots] = sorted_flat // k
    slot_weight[slots] = w.reshape(-1)[sorted_flat]
    pair_slot[sorted_flat] = slots
    return {
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "padded_offsets": poff.astype(np.int32),
        "slot_token": slot_token,
        "slot_weight": slot_weight,
        "pair_slot": pair_slot,
    }
