"""The SiLU of the L1 epilogue on every gate value it can meet, against an fp64 bound.

The "complete pipeline" commit of the tests page computes h = SiLU(gate) * up in BF16
from the BF16 L1 outputs, SiLU(g) = g / (1 + exp(-g)).  The epilogue evaluates it in fp32
with the fast exponential and division intrinsics and rounds h to BF16 after the product
with up; the oracle uses the correctly rounded exponential.  Since g is a BF16 value,
sweeping all finite BF16 values covers every input the epilogue's SiLU receives.

Bound (relative to the exact value s = g / (1 + e^-g)): the fast exponential's error
grows with |x|; the test allows it 2 + floor(1.2 |g|) ulp (the CUDA documentation of the
intrinsic gives a bound of the same form), the fp32 add 1/2 ulp and the fast division
2 ulp, so |s_dev - s| <= (Ne + 3) * 2^-23 * |s| with Ne = 2 + floor(1.2 |g|), plus an
absolute 2^-126 for results below the normal range (and for g < -87, where the
intrinsic division by 1 + e^-g > 2^126 returns 0 while |s| < 1e-36).  Up to |g| = 100
that is below 2^-15 relative, under 1/64 of a BF16 half-step, so h = bf16(SiLU(g) * up)
can differ from the correctly rounded value only by one BF16 step next to a rounding
midpoint."""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as q

pytestmark = pytest.mark.gpu


def _every_finite_bf16():
    f = q.bf16_from_bits(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    return f[np.isfinite(f)]


def test_epilogue_silu_every_bf16_gate_within_bound():
    from nvfp4_mixture_experts_stage_gb300 import binding as B
    g = _every_finite_bf16()
    gd = torch.from_numpy(g).cuda()
    sd = torch.empty_like(gd)
    B.moe_selftest_silu(gd, sd)
    torch.cuda.synchronize()
    s_dev = sd.cpu().numpy().astype(np.float64)
    g64 = g.astype(np.float64)
    with np.errstate(over="ignore"):
        s_ref = g64 / (1.0 + np.exp(-g64))
    ne = 2.0 + np.floor(1.2 * np.abs(g64))
    bound = (ne + 3.0) * 2.0 ** -23 * np.abs(s_ref) + 2.0 ** -126
    # below g = -87 the intrinsic division by 1 + e^-g > 2^126 returns 0: |s| < 1e-35 there
    bound = np.where(g64 < -87.0, np.maximum(bound, np.abs(s_ref)), bound)
    assert np.abs(s_ref[g64 < -87.0]).max() < 1e-35
    err = np.abs(s_dev - s_ref)
    bad = err > bound
    assert not bad.any(), (g[bad][:8], s_dev[bad][:8], s_ref[bad][:8])
    # special values: silu(0) = 0, large positive g passes through, large negative gives -0/0
    assert s_dev[g == 0].max() == 0.0
    big = g > 100
    assert np.array_equal(s_dev[big], g64[big])
    assert np.abs(s_dev[g < -100]).max() == 0.0
    # consequence for h = bf16(silu(g) * 1): at most one BF16 step from the correctly
    # rounded value, and only next to a rounding midpoint (a small fraction of inputs)
    # leave out results in the subnormal range, and g < -87 (the device gives 0 there)
    nrm = (np.abs(g64) >= 2.0 ** -120) & (g64 >= -87.0)
    h_dev = q.bf16_round(s_dev[nrm].astype(np.float32)).astype(np.float64)
    h_ref = q.bf16_round(s_ref[nrm].astype(np.float32)).astype(np.float64)
    step = np.abs(q.bf16_round((np.abs(h_ref) * (1 + 2.0 ** -7)).astype(np.float32)) - np.abs(h_ref))
    diff = np.abs(h_dev - h_ref)
    assert np.all(diff <= np.maximum(step, 2.0 ** -133))
    assert (diff > 0).mean() < 0.01
