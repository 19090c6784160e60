"""Pins for the oracle's routing (CPU only): brute-force loops on tiny inputs
and the invariants the commit pages state."""

import numpy as np
import pytest

import workloads
from oracle.route import route, slot_capacity


def _brute(ids, w, E, off):
    """Python loops: for each expert in order, walk the pairs in (t, j) order
    and append; pad each expert to a multiple of 128 slots."""
    T, k = ids.shape
    cap = slot_capacity(T, k, E)
    st = [-1] * cap
    sw = [0.0] * cap
    ps = [-1] * (T * k)
    counts, offs, poff = [], [0], [0]
    slot = 0
    for e in range(E):
        c = 0
        for t in range(T):
            for j in range(k):
                if int(ids[t, j]) - off == e:
                    st[slot + c] = t
                    sw[slot + c] = float(w[t, j])
                    ps[t * k + j] = slot + c
                    c += 1
        counts.append(c)
        offs.append(offs[-1] + c)
        padded = ((c + 127) // 128) * 128
        slot += padded
        poff.append(slot)
    return counts, offs, poff, st, sw, ps


@pytest.mark.parametrize("seed", range(6))
def test_route_matches_brute_force(seed):
    r = np.random.default_rng(seed)
    T, k, E = int(r.integers(1, 40)), int(r.integers(1, 5)), int(r.integers(1, 9))
    off = int(r.integers(0, 3)) * E
    ids = r.integers(-2, 4 * E, (T, k)).astype(np.int32)   # includes invalid / foreign ids
    w = r.random((T, k)).astype(np.float32)
    got = route(ids, w, E, off)
    counts, offs, poff, st, sw, ps = _brute(ids, w, E, off)
    assert list(got["counts"]) == counts
    assert list(got["offsets"]) == offs
    assert list(got["padded_offsets"]) == poff
    assert list(got["slot_token"]) == st
    assert np.array_equal(got["slot_weight"], np.array(sw, np.float32))
    assert list(got["pair_slot"]) == ps


def test_offsets_are_bincount_cumsum_and_int32():
    ids, w = workloads.routing(workloads.WORKLOADS["decode"])
    rt = route(ids, w, 48, 144)
    local = ids.reshape(-1).astype(np.int64) - 144
    local = local[(local >= 0) & (local < 48)]
    assert np.array_equal(rt["counts"], np.bincount(local, minlength=48))
    assert np.array_equal(rt["offsets"][1:], np.cumsum(rt["counts"]))
    assert rt["offsets"].dtype == np.int32 and rt["padded_offsets"].dtype == np.int32
    assert np.all(rt["padded_offsets"] % 128 == 0)
    assert rt["offsets"][-1] == local.size


def test_pair_slot_inverts_slot_token():
    ids, w = workloads.routing(workloads.WORKLOADS["skew_top8"])
    T, k = ids.shape
    rt = route(ids, w, 48, 0)
    ps = rt["pair_slot"]
    ok = ps >= 0
    assert np.array_equal(rt["slot_token"][ps[ok]], np.nonzero(ok)[0] // k)
    assert np.array_equal(rt["slot_weight"][ps[ok]], w.reshape(-1)[ok])
    # every non-padding slot is hit exactly once
    assert np.array_equal(np.sort(ps[ok]), np.nonzero(rt["slot_token"] >= 0)[0])
    # padding slots: token -1, weight 0
    assert np.all(rt["slot_weight"][rt["slot_token"] < 0] == 0)


def test_empty_experts_have_equal_offsets():
    ids, w = workloads.routing(workloads.WORKLOADS["skew_top1"])
    rt = route(ids, w, 48, 0)
    empty = rt["counts"] == 0
    assert empty.sum() == 8      # 8 experts get no token by construction
    e = np.nonzero(empty)[0]
    assert np.all(rt["offsets"][e] == rt["offsets"][e + 1])
    assert np.all(rt["padded_offsets"][e] == rt["padded_offsets"][e + 1])
    assert rt["counts"].max() > 0.30 * ids.shape[0]   # one expert > 30%


def test_top1_sorted_by_expert_is_the_identity_slot_map():
    """The "identity slot map" commit (commits of src): with top-1 and tokens
    already ordered by expert, slot order is token order."""
    ids, w = workloads.routing(workloads.WORKLOADS["skew_top1"])
    rt = route(ids, w, 48, 0)
    compact = rt["slot_token"][rt["slot_token"] >= 0]
    assert np.array_equal(compact, np.arange(ids.shape[0]))
    # the unsorted twin gives a permutation, not the identity
    ids2, w2 = workloads.shuffled_twin(ids, w)
    rt2 = route(ids2, w2, 48, 0)
    c2 = rt2["slot_token"][rt2["slot_token"] >= 0]
    assert np.array_equal(np.sort(c2), np.arange(ids.shape[0]))
    assert not np.array_equal(c2, np.arange(ids.shape[0]))


def test_foreign_and_invalid_ids_are_dropped():
    """The "global expert ids" commit: rank r owns [48 r, 48 r + 48); other ids
    are not its work."""
    ids = np.array([[-1, 143, 144], [191, 192, 400]], np.int32)
    w = np.ones((2, 3), np.float32)
    rt = route(ids, w, 48, 144)
    assert list(rt["pair_slot"]) == [-1, -1, 0, 128, -1, -1]
    assert rt["counts"][0] == 1 and rt["counts"][47] == 1 and rt["counts"].sum() == 2
