"""The number of kernels one moe_forward call launches, as bench.py reports it in
`gpu_launches` (its kernels_per_step): counted from the CUDA activity of one call under
the torch profiler, for a batch on each side of the small-batch path (T*topk <= 8192)
and both modes of the h scale."""

import pytest
import torch

import workloads
from tests.helpers import oracle_weights

pytestmark = pytest.mark.gpu


def _kernels_in_one_call(fw, x, ids, w):
    from torch.profiler import ProfilerActivity, profile
    fw(x, ids, w)
    torch.cuda.synchronize()
    # the first profiling session of a process can miss the activity records while the
    # tracer starts: take the second one if the first saw no kernel
    for _ in range(2):
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            fw(x, ids, w)
            torch.cuda.synchronize()
        names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        kernels = [n for n in names if "moe::" in n]
        if kernels:
            return kernels
    return []


@pytest.mark.parametrize("T", [64, 2048])
@pytest.mark.parametrize("dynamic_h", [False, True])
def test_kernels_per_call_match_the_bench_count(T, dynamic_h):
    import bench
    from nvfp4_mixture_experts_stage_gb300 import binding as B, runtime as R
    wl = workloads.small("launches", T=T, K=256, I=128, E=8, topk=8)
    W = oracle_weights(wl)
    layer = R.layer_from_nvfp4(W["w1_codes"], W["w1_sf"], W["gs_w1_gate"], W["gs_w1_up"], W["w2_codes"],
                               W["w2_sf"], W["gs_w2"], wl.topk, wl.expert_offset)
    x = workloads.activations(wl).cuda()
    ids, w = workloads.routing(wl)
    ids, w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    fw = R.Forward(layer, wl.T, B.MOE_GS_DYNAMIC if dynamic_h else B.MOE_GS_FIXED)
    if not dynamic_h:
        fw.gs_h.fill_(float(workloads.fixed_gs_h(wl)))
    kernels = _kernels_in_one_call(fw, x, ids, w)
    if not kernels:
        pytest.skip("no CUDA kernel activity recorded by the profiler on this machine")
    assert int(fw.status.item()) == 0
    assert len(kernels) == bench.kernels_per_step(T, wl.topk, dynamic_h), kernels
