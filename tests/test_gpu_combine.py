"""GPU parity of the per-token weighted combine (moe_combine_rows) against the
oracle's combine: bit for bit, since both sum w[t, j] * y[slot(t, j)] in pair
order in fp32 and round once to BF16.  moe_forward takes this path for large
batches (the full-size prefill and skewed-routing tests); here it is checked
alone on routing with foreign ids (slot -1), empty tokens and a ragged K."""

import numpy as np
import pytest
import torch

import workloads
from oracle import moe as omoe, nvfp4 as q, route as oroute

pytestmark = pytest.mark.gpu

B = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B
    from nvfp4_mixture_experts_stage_gb300 import binding
    B = binding


def _case(T, K, E, topk, offset, n_global, seed, y_scale=1.0):
    r = np.random.default_rng(seed)
    ids = np.stack([r.choice(n_global, topk, replace=False) for _ in range(T)]).astype(np.int32)
    w = r.random((T, topk)).astype(np.float32)
    rt = oroute.route(ids, w, E, offset)
    cap = B.moe_slot_capacity(T, topk, E)
    y = q.bf16_round((r.standard_normal((cap, K)) * y_scale).astype(np.float32))
    ref = omoe.combine(y, rt, T, topk, w)
    y_dev = torch.from_numpy(y).to(torch.bfloat16).cuda()
    out = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_combine_rows(y_dev, torch.from_numpy(rt["pair_slot"].astype(np.int32)).cuda(),
                       torch.from_numpy(w).cuda(), out, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return out.float().cpu().numpy(), ref, rt


@pytest.mark.parametrize("T,K,E,topk,offset,n_global", [(37, 256, 8, 2, 0, 8), (64, 4096, 48, 8, 144, 384),
                                                         (300, 7168, 48, 8, 0, 48), (5, 8, 4, 3, 4, 12),
                                                         (20, 256, 32, 12, 0, 32)])
def test_combine_bit_exact(T, K, E, topk, offset, n_global):
    got, ref, rt = _case(T, K, E, topk, offset, n_global, seed=T + K)
    assert np.array_equal(got, ref)


def test_combine_tokens_without_local_expert_are_zero():
    got, ref, rt = _case(50, 64, 4, 2, 8, 16, seed=5)   # experts 8..11 local of 16
    ps = rt["pair_slot"].reshape(50, 2)
    none = (ps < 0).all(axis=1)
    assert none.any()
    assert not np.any(got[none])
    assert np.array_equal(got, ref)


def test_combine_large_magnitudes_round_like_the_oracle():
    got, ref, _ = _case(16, 512, 8, 4, 0, 8, seed=9, y_scale=3e4)
    assert np.array_equal(got, ref)
