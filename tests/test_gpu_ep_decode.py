"""Expert parallelism simulated on one GPU at the decode shape.

A 384-expert layer (K=4096, I=3072, top-8 over global ids) split over 8 ranks of
48 experts each (expert offsets 0, 48, ..., 336).  Rank r's layer holds global
experts 48r .. 48r+47 and drops the pairs routed elsewhere; the ranks run one
after another on the same decode batch, and the sum of their outputs is checked
against the oracle's layer over all 384 experts on sampled tokens.  The pages
define the split this way: global expert ids with a rank-local range, each rank
writing only its own experts' contributions, and the cross-rank sum done by the
caller (nvfp4-megamoe-kernel, commits of src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py:
"global expert IDs" and "cross-rank all-reduce happens in the parent").

The h scale is held fixed (the calibrated mode): with scales derived from the data
each rank would scale its own h, which a single 384-expert layer cannot reproduce.
The weights of global expert g come from the seeded generator's expert g; the GPU
quantises them with the library's quantiser, the oracle with its own.
"""

import concurrent.futures as cf
import dataclasses

import numpy as np
import pytest
import torch

import workloads
from oracle import moe as omoe, nvfp4 as q
from tests.helpers import assert_layer_close

pytestmark = pytest.mark.gpu

N_RANKS, E_LOCAL, E_GLOBAL = 8, 48, 384


def _oracle_expert(wl, g):
    I = wl.I
    w1 = workloads.expert_w1(wl, g).float().numpy()
    w2 = workloads.expert_w2(wl, g).float().numpy()
    return g, q.quantize(w1[:I]), q.quantize(w1[I:]), q.quantize(w2)


def test_eight_ranks_of_384_experts_sum_to_the_full_layer():
    from nvfp4_mixture_experts_stage_gb300 import binding as B, runtime as R

    wl = workloads.WORKLOADS["decode"]
    assert (wl.n_global, wl.E, wl.topk) == (E_GLOBAL, E_LOCAL, 8)
    # the weight streams of all 384 global experts (the first 48 are the decode layer's own)
    wg = dataclasses.replace(wl, E=E_GLOBAL)
    x = workloads.activations(wl)
    ids, w = workloads.routing(wl)
    assert ids.min() >= 0 and ids.max() < E_GLOBAL
    gs_h = workloads.fixed_gs_h(wl)

    # sampled tokens: the first and last, and random ones, so that every rank has pairs
    # among them
    tokens = np.unique(np.concatenate([np.random.default_rng(5).choice(wl.T, 10, replace=False), [0, wl.T - 1]]))
    assert set(np.unique(ids[tokens] // E_LOCAL)) == set(range(N_RANKS))

    total = np.zeros((wl.T, wl.K), np.float64)
    x_dev = x.cuda()
    ids_dev = torch.from_numpy(ids).cuda()
    w_dev = torch.from_numpy(w).cuda()
    with cf.ThreadPoolExecutor(16) as ex:
        for r in range(N_RANKS):
            g0 = E_LOCAL * r
            w1 = list(ex.map(lambda e: workloads.expert_w1(wg, g0 + e), range(E_LOCAL)))
            w2 = list(ex.map(lambda e: workloads.expert_w2(wg, g0 + e), range(E_LOCAL)))
            layer = R.quantize_weights_on_device(wl, lambda e: w1[e], lambda e: w2[e])
            del w1, w2
            layer.expert_offset = g0
            fw = R.Forward(layer, wl.T, B.MOE_GS_FIXED)
            fw.gs_h.fill_(float(gs_h))
            out = fw(x_dev, ids_dev, w_dev)
            torch.cuda.synchronize()
            assert int(fw.status.item()) == 0, r
            total += out.float().cpu().numpy()
            del fw, layer, out
            torch.cuda.empty_cache()

    # the oracle's 384-expert layer for the sampled tokens: only their experts are
    # quantised, numbered compactly; other pairs are foreign to it and dropped, which
    # leaves the sampled tokens' outputs unchanged (x's scale still comes from all of x)
    used = np.unique(ids[tokens])
    compact = np.full(E_GLOBAL, -1, np.int64)
    compact[used] = np.arange(len(used))
    U, I, K = len(used), wl.I, wl.K
    W = {"w1_codes": np.empty((U, 2 * I, K // 2), np.uint8), "w1_sf": np.empty((U, 2 * I, K // 16), np.uint8),
         "gs_w1_gate": np.empty(U, np.float32), "gs_w1_up": np.empty(U, np.float32),
         "w2_codes": np.empty((U, K, I // 2), np.uint8), "w2_sf": np.empty((U, K, I // 16), np.uint8),
         "gs_w2": np.empty(U, np.float32)}
    with cf.ThreadPoolExecutor(16) as ex:
        for g, gq, uq, dq in ex.map(lambda g: _oracle_expert(wg, int(g)), used):
            i = compact[g]
            W["w1_codes"][i, :I], W["w1_sf"][i, :I], W["gs_w1_gate"][i] = gq
            W["w1_codes"][i, I:], W["w1_sf"][i, I:], W["gs_w1_up"][i] = uq
            W["w2_codes"][i], W["w2_sf"][i], W["gs_w2"][i] = dq
    ids_c = compact[ids].astype(np.int32)          # -1: an expert no sampled token uses
    ref = omoe.forward(x.float().numpy(), ids_c, w, U, 0, W, gs_h=gs_h, tokens=tokens)
    # each rank rounds its partial output to BF16 before the sum; the oracle rounds once
    assert_layer_close(total[tokens], ref["out"], "8-rank sum vs the 384-expert layer")
    # tokens outside the sample: finite, and zero only where no expert is routed (never here)
    assert np.isfinite(total).all()
