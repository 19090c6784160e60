"""GPU parity of the whole layer (moe_forward through the C ABI) against the
oracle, on the seeded workloads, plus CUDA-graph capture and replay."""

import numpy as np
import pytest
import torch

import workloads
from oracle import moe as omoe
from tests.helpers import assert_layer_close, oracle_weights

pytestmark = pytest.mark.gpu

B = R = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B, R
    from nvfp4_mixture_experts_stage_gb300 import binding, runtime
    B, R = binding, runtime


@pytest.fixture(params=["tiled", "tiled1", "tiledp", "stream32", "stream64"], autouse=True)
def gemm_kernel(request, _lib):
    """Run every test with each grouped-GEMM kernel (and streaming chunk) forced:
    tiled = the default tiled choice (L2's 256-wide tiles on CTA pairs), tiled1 =
    single-CTA tiles only, tiledp = CTA pairs for both GEMMs' 256-wide tiles."""
    pol = {"tiled": B.MOE_GEMM_TILED, "tiled1": B.MOE_GEMM_TILED_1CTA, "tiledp": B.MOE_GEMM_TILED_PAIR,
           "stream32": B.MOE_GEMM_STREAMING_N32, "stream64": B.MOE_GEMM_STREAMING_N64}[request.param]
    old = B.moe_set_gemm_policy(pol)
    yield request.param
    B.moe_set_gemm_policy(old)


def _layer(W, wl):
    return R.layer_from_nvfp4(W["w1_codes"], W["w1_sf"], W["gs_w1_gate"], W["gs_w1_up"], W["w2_codes"],
                              W["w2_sf"], W["gs_w2"], wl.topk, wl.expert_offset)


def _run(wl, W, mode, gs_h=None, ids=None, w=None, x=None):
    x = workloads.activations(wl) if x is None else x
    if ids is None:
        ids, w = workloads.routing(wl)
    layer = _layer(W, wl)
    fw = R.Forward(layer, wl.T, mode)
    if gs_h is not None:
        fw.gs_h.fill_(float(gs_h))
    out = fw(x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert fw.status.item() == 0
    return out.float().cpu().numpy(), fw.gs_h.item(), x, ids, w


SMALL = [
    workloads.WORKLOADS["tiny"],
    workloads.small("mid", T=200, K=512, I=256, E=6, topk=3, expert_offset=12, n_global=24),
    workloads.small("ragged", T=77, K=384, I=192, E=5, topk=2, routing="softmax_topk", x_kind="outliers"),
    workloads.small("top1", T=300, K=256, I=128, E=4, topk=1),
    workloads.small("bigrows", T=130, K=256, I=64, E=3, topk=2, x_kind="big_rows"),
    # three 256-deep k-blocks per tile in both GEMMs (an odd count)
    workloads.small("odd_kblocks", T=96, K=768, I=768, E=4, topk=2),
]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", ["dynamic", "fixed"])
def test_forward_matches_oracle(wl, mode):
    W = oracle_weights(wl)
    gs_h = None if mode == "dynamic" else workloads.fixed_gs_h(wl)
    got, g_h, x, ids, w = _run(wl, W, B.MOE_GS_DYNAMIC if mode == "dynamic" else B.MOE_GS_FIXED, gs_h)
    ref = omoe.forward(x.float().numpy(), ids, w, wl.E, wl.expert_offset, W, gs_h=gs_h)
    assert_layer_close(got, ref["out"], wl.name)
    if mode == "dynamic":
        assert abs(g_h - float(ref["gs_h"])) <= 1e-2 * float(ref["gs_h"])
    # tokens with no local expert are exactly zero
    none_local = (ref["route"]["pair_slot"].reshape(wl.T, wl.topk) < 0).all(axis=1)
    assert np.all(got[none_local] == 0)


def test_forward_maximum_experts_and_topk():
    """The API's limits: 256 local experts (most with a handful of slots, some empty) and
    top-32 routing."""
    wl = workloads.small("maxes", T=40, K=256, I=64, E=256, topk=32)
    W = oracle_weights(wl)
    gs_h = workloads.fixed_gs_h(wl)
    got, _, x, ids, w = _run(wl, W, B.MOE_GS_FIXED, gs_h)
    ref = omoe.forward(x.float().numpy(), ids, w, wl.E, wl.expert_offset, W, gs_h=gs_h)
    assert_layer_close(got, ref["out"], wl.name)


def test_forward_empty_batch():
    """T = 0: nothing to do, status OK, no launch touches the (empty) buffers."""
    wl = workloads.small("empty_src", T=8, K=256, I=64, E=4, topk=2)
    W = oracle_weights(wl)
    layer = _layer(W, wl)
    fw = R.Forward(layer, 0, B.MOE_GS_DYNAMIC)
    x = torch.zeros(0, wl.K, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(0, wl.topk, dtype=torch.int32, device="cuda")
    w = torch.zeros(0, wl.topk, dtype=torch.float32, device="cuda")
    out = fw(x, ids, w)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.K) and fw.status.item() == 0


def test_forward_graph_capture_and_replay():
    wl = SMALL[1]
    W = oracle_weights(wl)
    layer = _layer(W, wl)
    fw = R.Forward(layer, wl.T, B.MOE_GS_DYNAMIC)
    x = workloads.activations(wl).cuda()
    ids, w = workloads.routing(wl)
    ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fw(x, ids_d, w_d, stream=s)          # warm-up (configures kernels) outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fw(x, ids_d, w_d)
    # new inputs in the same buffers, then replay
    wl2 = workloads.small("mid2", T=200, K=512, I=256, E=6, topk=3, expert_offset=12, n_global=24, seed=5)
    x2 = workloads.activations(wl2)
    ids2, w2 = workloads.routing(wl2)
    x.copy_(x2.cuda())
    ids_d.copy_(torch.from_numpy(ids2))
    w_d.copy_(torch.from_numpy(w2))
    g.replay()
    torch.cuda.synchronize()
    got = fw.out.float().cpu().numpy()
    ref = omoe.forward(x2.float().numpy(), ids2, w2, wl.E, wl.expert_offset, W)["out"]
    assert_layer_close(got, ref, "graph replay")
    eager = R.Forward(layer, wl.T, B.MOE_GS_DYNAMIC)(x, ids_d, w_d)
    torch.cuda.synchronize()
    assert_layer_close(got, eager.float().cpu().numpy(), "graph vs eager")


@pytest.mark.parametrize("mode", ["dynamic", "fixed"])
def test_forward_many_pairs_scatter_path(mode):
    """More routed pairs than the fused prologue routes (8192): the chunked routing
    kernels and the separate amax kernel run, while the output is small enough for the
    fp32 scatter epilogue.  Experts own 2-3 m-tiles, so most end on a 256-row tile whose
    second half is empty and whose first half is sparse.  The call is then captured
    and replayed many times, L2 flushed in between, each replay checked."""
    wl = workloads.small("many_pairs", T=1100, K=256, I=128, E=32, topk=8)
    assert wl.T * wl.topk > 8192
    W = oracle_weights(wl)
    gs_h = None if mode == "dynamic" else workloads.fixed_gs_h(wl)
    layer = _layer(W, wl)
    fw = R.Forward(layer, wl.T, B.MOE_GS_DYNAMIC if mode == "dynamic" else B.MOE_GS_FIXED)
    if gs_h is not None:
        fw.gs_h.fill_(float(gs_h))
    x = workloads.activations(wl)
    ids, w = workloads.routing(wl)
    ref = omoe.forward(x.float().numpy(), ids, w, wl.E, wl.expert_offset, W, gs_h=gs_h)["out"]
    xd, ids_d, w_d = x.cuda(), torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fw(xd, ids_d, w_d, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert fw.status.item() == 0
    assert_layer_close(fw.out.float().cpu().numpy(), ref, "eager")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fw(xd, ids_d, w_d)
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    for i in range(40):
        flush.sum()
        g.replay()
        if i % 8 == 7:
            torch.cuda.synchronize()
            assert fw.status.item() == 0
            assert_layer_close(fw.out.float().cpu().numpy(), ref, f"replay {i}")


def test_simulated_expert_parallel_sum():
    """Ranks r = 0..3 each run their 6 local experts of 24 global ones on one
    GPU, one after another; the sum of their outputs matches the oracle layer
    over all 24 experts (fixed gs_h, so every rank quantises h the same way)."""
    full = workloads.small("ep", T=64, K=256, I=128, E=24, topk=4)
    W = oracle_weights(full)
    x = workloads.activations(full)
    ids, w = workloads.routing(full)
    gs_h = np.float32(8.0 / 2688.0)
    total = np.zeros((full.T, full.K))
    for r in range(4):
        sl = slice(6 * r, 6 * r + 6)
        Wr = {k: (v[sl] if isinstance(v, np.ndarray) and v.shape[0] == 24 else v) for k, v in W.items()}
        wl_r = workloads.small("ep_r", T=64, K=256, I=128, E=6, topk=4, expert_offset=6 * r)
        got, _, _, _, _ = _run(wl_r, Wr, B.MOE_GS_FIXED, gs_h, ids=ids, w=w, x=x)
        total += got
    ref = omoe.forward(x.float().numpy(), ids, w, 24, 0, W, gs_h=gs_h)["out"]
    assert_layer_close(total, ref, "EP sum")
