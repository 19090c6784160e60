"""The device's two code encoders over every fp32 input.

The quantisers, the requantiser and the L1 requant epilogue encode a scaled value as an
E2M1 code and a block scale as a UE4M3 byte (nvfp4-megamoe-kernel, "NVFP4 quantisation"
commits: nearest E2M1 value of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with the sign in bit 3; block
scales as float8 e4m3fn bytes, at most 448).  Both encodings of a non-negative value are
non-decreasing step functions of its bit pattern, so one is fixed by where its steps
are.  The tests sweep every non-negative pattern (+0 up to +inf) through the device
encoders (moe_selftest_codecs), check that the outputs never decrease, and check that the
steps sit exactly where rounding to nearest (ties to the even code) over the grid puts
them: the midpoint of two neighbouring grid values, or the pattern after it when the tie
goes down.  Every negative pattern must give the E2M1 code of its magnitude with bit 3
set.  The oracle's encoders are compared on both sides of every step and on a random
sample of patterns."""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as q

pytestmark = pytest.mark.gpu

B = None
CHUNK = 1 << 28
POS_INF = 0x7F800000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B
    from nvfp4_mixture_experts_stage_gb300 import binding
    B = binding


def _bits(f):
    return int(np.array(f, np.float32).view(np.uint32))


def _expected_steps(grid):
    """(first pattern, code) of every step of round-to-nearest over an increasing grid
    whose codes are 0, 1, 2, ...: a tie goes to the even code."""
    steps = []
    for c in range(1, len(grid)):
        mid = (grid[c - 1] + grid[c]) / 2.0
        assert float(np.float32(mid)) == mid          # midpoints of these grids are fp32 values
        steps.append((_bits(mid) if c % 2 == 0 else _bits(mid) + 1, c))
    return steps


E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_grid():
    """Values of the bytes 0x00 .. 0x7E from the e4m3fn bit layout (4 exponent bits,
    bias 7, 3 mantissa bits, subnormals below 2**-6); 0x7E = 448 is the largest."""
    out = []
    for b in range(0x7F):
        e, m = b >> 3, b & 7
        out.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    assert out[-1] == 448.0
    return out


@pytest.fixture(scope="module")
def sweep(_lib):
    """Steps of both encoders over patterns 0 .. +inf, after checking that neither
    output decreases anywhere; also checks the sign rule on every negative pattern."""
    steps = {"e2m1": [], "e4m3": []}
    last = {"e2m1": None, "e4m3": None}
    sample = np.sort(np.concatenate([
        np.random.default_rng(11).integers(0, POS_INF + 1, 1 << 20, dtype=np.uint64),
        np.array([0, POS_INF, _bits(448.0), _bits(464.0), _bits(6.0), _bits(2.0 ** -10)], np.uint64)]))
    got = {"e2m1": [], "e4m3": []}
    c2 = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    c4 = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    n2 = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    n4 = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    first = 0
    while first <= POS_INF:
        n = min(CHUNK, POS_INF + 1 - first)
        B.moe_selftest_codecs(first, c2[:n], c4[:n])
        B.moe_selftest_codecs(first | 0x80000000, n2[:n], n4[:n])
        for name, c in (("e2m1", c2[:n]), ("e4m3", c4[:n])):
            v = c.to(torch.int16)
            assert bool((v[1:] >= v[:-1]).all()), f"{name} decreases inside patterns {first:#x}+"
            if last[name] is None:
                steps[name].append((first, int(v[0])))
            elif int(v[0]) != last[name]:
                assert int(v[0]) > last[name]
                steps[name].append((first, int(v[0])))
            idx = torch.nonzero(v[1:] != v[:-1]).flatten() + 1
            for i, code in zip(idx.tolist(), v[idx].tolist()):
                steps[name].append((first + i, code))
            last[name] = int(v[-1])
        lo, hi = np.searchsorted(sample, [first, first + n])
        if hi > lo:
            off = torch.from_numpy((sample[lo:hi] - first).astype(np.int64)).cuda()
            got["e2m1"].append(c2[off].cpu().numpy())
            got["e4m3"].append(c4[off].cpu().numpy())
        # a negative value codes as its magnitude with the sign bit set (-0 included)
        assert bool((n2[:n] == (c2[:n] | 8)).all()), f"sign rule fails at patterns {first | 0x80000000:#x}+"
        first += n
    torch.cuda.synchronize()
    return {"steps": steps, "sample": sample.astype(np.uint32),
            "sample_e2m1": np.concatenate(got["e2m1"]), "sample_e4m3": np.concatenate(got["e4m3"])}


def test_e2m1_encoder_on_every_nonnegative_fp32(sweep):
    st = sweep["steps"]["e2m1"]
    assert st[0] == (0, 0)
    assert st[1:] == _expected_steps(E2M1_GRID)
    # +inf saturates to the largest magnitude (the sweep's last step is to index 7)
    assert st[-1][1] == 7


def test_e4m3_encoder_on_every_nonnegative_fp32(sweep):
    st = sweep["steps"]["e4m3"]
    assert st[0] == (0, 0)
    assert st[1:] == _expected_steps(_e4m3_grid())
    assert st[-1][1] == 0x7E                           # saturates at 448, +inf included


def test_oracle_encoders_agree_at_every_step_and_on_a_sample(sweep):
    """The oracle's encoders give the device's code on both sides of every device step,
    and on 2**20 random non-negative patterns plus the saturation and tie points."""
    enc = {"e2m1": q.e2m1_index, "e4m3": q.e4m3_encode_satfinite}
    for name, f in enc.items():
        st = sweep["steps"][name]
        for (_, c_prev), (p, c) in zip(st, st[1:]):
            below, at = f(np.array([p - 1, p], np.uint32).view(np.float32))
            assert (int(below), int(at)) == (c_prev, c), (name, hex(p))
    vals = sweep["sample"].view(np.float32)
    assert np.array_equal(sweep["sample_e2m1"] & 7, q.e2m1_index(vals))
    assert np.array_equal(sweep["sample_e2m1"] >> 3, np.zeros_like(sweep["sample_e2m1"]))
    assert np.array_equal(sweep["sample_e4m3"], q.e4m3_encode_satfinite(vals))
