"""moe_route_static_scratch: routing for callers that cannot allocate.

Plugins whose host runtime owns all device memory, or serving loops that must
not allocate on their hot path, cannot pass moe_route a workspace.  The
workspace-free entry point keeps its scratch tables in a fixed device array
inside the library.  These tests call it through the C ABI and check that it
routes exactly like moe_route (routing is integer work: bit-exact), on two
calls in a row with different inputs (the array keeps the previous call's
contents), and that calls past its fixed size are refused up front.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from nvfp4_mixture_experts_stage_gb300 import binding
    return binding


def _buffers(B, T, k, E):
    cap = B.moe_slot_capacity(T, k, E)
    d = lambda n, dt=torch.int32: torch.full((n,), -7, dtype=dt, device="cuda")
    return {"counts": d(E), "offsets": d(E + 1), "padded_offsets": d(E + 1), "slot_token": d(cap),
            "slot_weight": d(cap, torch.float32), "pair_slot": d(T * k)}


def _with_workspace(B, ids, w, E, off):
    T, k = ids.shape
    o = _buffers(B, T, k, E)
    ws = torch.empty(B.moe_route_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    B.moe_route(ids, w, E, off, o["counts"], o["offsets"], o["padded_offsets"], o["slot_token"],
                o["slot_weight"], o["pair_slot"], ws)
    return o


def _without_workspace(B, ids, w, E, off):
    T, k = ids.shape
    o = _buffers(B, T, k, E)
    B.moe_route_static_scratch(ids, w, E, off, o["counts"], o["offsets"], o["padded_offsets"], o["slot_token"],
                               o["slot_weight"], o["pair_slot"])
    return o


def _same(a, b):
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_static_scratch_route_matches_moe_route_twice_in_a_row(B):
    cases = [workloads.WORKLOADS["decode"], workloads.WORKLOADS["skew_top8"]]
    for wl in cases:   # two calls in a row; the second finds the first call's tables in the array
        ids, w = workloads.routing(wl)
        ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
        _same(_without_workspace(B, ids_d, w_d, wl.E, wl.expert_offset),
              _with_workspace(B, ids_d, w_d, wl.E, wl.expert_offset))


def test_static_scratch_two_table_calls_in_a_row(B):
    """Two calls in a row that both use the fixed tables (above 4096 (token, k) pairs
    routing goes through the chunk tables; below, one block routes without them), with
    different routings and expert counts, so the second call runs over the first call's
    table contents."""
    skew = workloads.WORKLOADS["skew_top8"]             # 32768 pairs, 48 experts
    ids1, w1 = workloads.routing(skew)
    r = np.random.default_rng(11)
    ids2 = r.integers(-3, 110, (2000, 8)).astype(np.int32)   # 16000 pairs, 100 experts at offset 5
    w2 = r.random((2000, 8)).astype(np.float32)
    assert ids1.size > 4096 and ids2.size > 4096
    d = lambda a: torch.from_numpy(a).cuda()
    o1 = _without_workspace(B, d(ids1), d(w1), skew.E, 0)
    torch.cuda.synchronize()
    o2 = _without_workspace(B, d(ids2), d(w2), 100, 5)
    _same(o1, _with_workspace(B, d(ids1), d(w1), skew.E, 0))
    _same(o2, _with_workspace(B, d(ids2), d(w2), 100, 5))


def test_static_scratch_route_back_to_back_on_one_stream(B):
    # a large call then a small one, enqueued without a host sync in between
    big = workloads.WORKLOADS["prefill"]
    ids1, w1 = workloads.routing(big)
    r = np.random.default_rng(9)
    ids2 = r.integers(-1, 40, (37, 3)).astype(np.int32)
    w2 = r.random((37, 3)).astype(np.float32)
    d = lambda a: torch.from_numpy(a).cuda()
    o1 = _without_workspace(B, d(ids1), d(w1), big.E, 0)
    o2 = _without_workspace(B, d(ids2), d(w2), 7, 2)
    _same(o1, _with_workspace(B, d(ids1), d(w1), big.E, 0))
    _same(o2, _with_workspace(B, d(ids2), d(w2), 7, 2))


def test_static_scratch_refuses_calls_beyond_its_size(B):
    E = 256
    T = (B.MOE_ROUTE_STATIC_TABLE_INTS // E + 1) * 256 // 8   # one chunk too many at top-8
    ids = torch.zeros((T, 8), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, 8), dtype=torch.float32, device="cuda")
    o = _buffers(B, T, 8, E)
    with pytest.raises(B.MoeError) as err:
        B.moe_route_static_scratch(ids, w, E, 0, o["counts"], o["offsets"], o["padded_offsets"], o["slot_token"],
                                   o["slot_weight"], o["pair_slot"])
    assert err.value.status == B.MOE_ERR_UNSUPPORTED_SHAPE
