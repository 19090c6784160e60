"""GPU parity of the grouped GEMMs (tcgen05 block-scaled MMA) against the oracle.

Exact-arithmetic cases (block scales that are powers of two, alpha = 1, sums
well inside fp32's 24-bit range) must match bit for bit whatever the
summation order: they pin the operand and scale layouts and the gate/up
split, up to the layer's production contraction (K = 4096 for L1, I = 3072 for
L2).  General cases use the layer tolerance."""

import functools

import numpy as np
import pytest
import torch

from oracle import moe as omoe, nvfp4 as q
from tests.helpers import assert_layer_close, dev

pytestmark = pytest.mark.gpu

B = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B
    from nvfp4_mixture_experts_stage_gb300 import binding
    B = binding


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


POW2_BYTES = np.array([0x28, 0x30, 0x38, 0x40, 0x48], np.uint8)  # 0.25 .. 4
POW2_BYTES_NARROW = np.array([0x30, 0x38, 0x40], np.uint8)       # 0.5 .. 2


def _slots(counts, topk=1, tight=False):
    """Routing tables for per-expert slot counts; tight: the slot capacity ends at
    the last expert's padded rows (no spare rows after them)."""
    counts = np.asarray(counts, np.int64)
    E = counts.size
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    poff = np.concatenate([[0], np.cumsum(-(-counts // 128) * 128)]).astype(np.int32)
    T = int(counts.sum())
    cap = B.moe_slot_capacity(max(T, 1), topk, E)
    cap = max(cap, int(poff[-1]))
    cap = -(-cap // 128) * 128
    if tight:
        cap = int(poff[-1])
    return {"counts": counts.astype(np.int32), "offsets": offs, "padded_offsets": poff}, cap


def _rand_operands(r, rows, K, exact):
    codes = r.integers(0, 256, (rows, K // 2)).astype(np.uint8)
    if exact:
        # every partial sum is a multiple of the smallest product unit and stays below
        # 2**24 units: K <= 256 with scales 0.25..4 (units 2**-6, |sum| <= 256*36*16),
        # K <= 4096 with scales 0.5..2 (units 2**-4, |sum| <= 4096*36*4 = 589824 =
        # 9437184 units)
        pool = POW2_BYTES if K <= 256 else POW2_BYTES_NARROW
        assert K <= 4096
        sf = pool[r.integers(0, pool.size, (rows, K // 16))]
    else:
        sf = r.integers(0x20, 0x58, (rows, K // 16)).astype(np.uint8)
    return codes, sf


@functools.lru_cache(maxsize=None)
def _l1_ref(counts, K, I, exact, seed, gs, tight):
    """Operands and the oracle's g, u for one L1 case (computed once for all five kernel
    choices)."""
    r = np.random.default_rng(seed)
    rt, cap = _slots(counts, tight=tight)
    E = len(counts)
    a_codes, a_sf = _rand_operands(r, cap, K, exact)        # padding rows hold garbage too
    w1c, w1s = _rand_operands(r, E * 2 * I, K, exact)
    w1c = w1c.reshape(E, 2 * I, K // 2)
    w1s = w1s.reshape(E, 2 * I, K // 16)
    if gs is None:
        gs_a, gg, gu = np.float32(1), np.ones(E, np.float32), np.ones(E, np.float32)
    else:
        gs_a = np.float32(gs)
        gg = r.uniform(1e-3, 2e-3, E).astype(np.float32)
        gu = r.uniform(1e-3, 2e-3, E).astype(np.float32)
    g, u = omoe.gemm_l1(a_codes, a_sf, gs_a, rt, w1c, w1s, gg, gu)
    valid = np.zeros(cap, bool)
    for e in range(E):
        valid[rt["padded_offsets"][e]:rt["padded_offsets"][e] + rt["counts"][e]] = True
    return rt, cap, a_codes, a_sf, w1c, w1s, gs_a, gg, gu, g, u, valid


def _l1_case(counts, K, I, exact, seed, epilogue, gs=None, tight=False):
    rt, cap, a_codes, a_sf, w1c, w1s, gs_a, gg, gu, g, u, valid = _l1_ref(tuple(counts), K, I, exact, seed, gs,
                                                                           tight)
    E = len(counts)
    d_wsf = torch.empty(w1s.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(dev(w1s), d_wsf, E, 2 * I, K, B.MOE_PREP_W1)
    out_cols = 2 * I if epilogue == B.MOE_L1_GATEUP_BF16 else I
    out = torch.zeros(cap, out_cols, dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_l1(dev(a_codes), dev(q.swizzle(a_sf)), dev(np.array([gs_a])), dev(rt["offsets"]),
                          dev(rt["padded_offsets"]), E, K, I, dev(w1c), d_wsf, dev(gg), dev(gu), epilogue,
                          out_bf16=out, h_amax=amax, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return out.float().cpu().numpy(), g, u, valid, amax.item()


@pytest.mark.parametrize("counts,K,I", [([5, 0, 140], 256, 128), ([1], 256, 64), ([128, 129, 3, 0, 0, 77], 256, 192),
                                        ([300, 17], 512, 64), ([200, 0, 129], 4096, 3072)])
def test_l1_gateup_exact_arithmetic_bit_exact(counts, K, I):
    got, g, u, valid, _ = _l1_case(counts, K, I, True, 11, B.MOE_L1_GATEUP_BF16)
    assert np.array_equal(got[valid, :I], g[valid])
    assert np.array_equal(got[valid, I:], u[valid])


@pytest.mark.parametrize("counts,K,I", [([37, 200, 0, 5], 4096, 128), ([130], 1024, 256), ([3, 9], 128, 64),
                                        ([200, 61], 384, 128)])
def test_l1_gateup_random_scales(counts, K, I):
    got, g, u, valid, _ = _l1_case(counts, K, I, False, 12, B.MOE_L1_GATEUP_BF16, gs=0.7)
    assert_layer_close(got[valid, :I], g[valid], "gate")
    assert_layer_close(got[valid, I:], u[valid], "up")


@pytest.mark.parametrize("counts", [[100, 0, 45], [300, 129]])
def test_l1_capacity_ends_at_last_expert(counts):
    """Slot capacity = the last expert's padded end: a 256-row pair tile of an expert
    with an odd number of 128-row tiles must not read past it (the peer's half is
    empty there)."""
    got, g, u, valid, _ = _l1_case(counts, 512, 128, True, 14, B.MOE_L1_GATEUP_BF16, tight=True)
    assert got.shape[0] == sum(-(-c // 128) * 128 for c in counts)
    assert np.array_equal(got[valid, :128], g[valid])
    assert np.array_equal(got[valid, 128:], u[valid])


def test_l1_silu_and_amax():
    got, g, u, valid, amax = _l1_case([70, 0, 300], 512, 128, False, 13, B.MOE_L1_SILU_BF16, gs=0.9)
    h = omoe.silu_mul(g, u)
    assert_layer_close(got[valid], h[valid], "h")
    # amax is the max over the valid rows the kernel itself produced
    assert amax == np.abs(got[valid]).max()


@functools.lru_cache(maxsize=None)
def _l2_ref(counts, I, K, exact, seed, gs, tight):
    """Operands and the oracle's y for one L2 case (computed once for all five kernel
    choices)."""
    r = np.random.default_rng(seed)
    rt, cap = _slots(counts, tight=tight)
    E = len(counts)
    h_codes, h_sf = _rand_operands(r, cap, I, exact)
    w2c, w2s = _rand_operands(r, E * K, I, exact)
    w2c = w2c.reshape(E, K, I // 2)
    w2s = w2s.reshape(E, K, I // 16)
    gs_h = np.float32(1 if gs is None else gs)
    g2 = np.ones(E, np.float32) if gs is None else r.uniform(1e-3, 2e-3, E).astype(np.float32)
    ref = omoe.gemm_l2(h_codes, h_sf, gs_h, rt, w2c, w2s, g2)
    valid = np.zeros(cap, bool)
    for e in range(E):
        valid[rt["padded_offsets"][e]:rt["padded_offsets"][e] + rt["counts"][e]] = True
    return rt, cap, h_codes, h_sf, w2c, w2s, gs_h, g2, ref, valid


def _l2_case(counts, I, K, exact, seed, epilogue, gs=None, slot_token=None, slot_weight=None, T=0, tight=False):
    rt, cap, h_codes, h_sf, w2c, w2s, gs_h, g2, ref, valid = _l2_ref(tuple(counts), I, K, exact, seed, gs, tight)
    E = len(counts)
    d_wsf = torch.empty(w2s.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(dev(w2s), d_wsf, E, K, I, B.MOE_PREP_W2)
    y = torch.zeros(cap, K, dtype=torch.bfloat16, device="cuda")
    out32 = torch.zeros(max(T, 1), K, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_l2(dev(h_codes), dev(q.swizzle(h_sf)), dev(np.array([gs_h])), dev(rt["offsets"]),
                          dev(rt["padded_offsets"]), E, I, K, dev(w2c), d_wsf, dev(g2), epilogue, y_rows=y,
                          slot_token=None if slot_token is None else dev(slot_token),
                          slot_weight=None if slot_weight is None else dev(slot_weight), out32=out32, T=T,
                          dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return y.float().cpu().numpy(), ref, valid, out32.cpu().numpy(), rt


@pytest.mark.parametrize("counts,I,K", [([5, 0, 140], 128, 256), ([128, 3], 256, 384), ([1, 1, 1], 64, 128),
                                        ([260], 512, 128), ([200, 0, 129], 3072, 4096)])
def test_l2_rows_exact_arithmetic_bit_exact(counts, I, K):
    got, ref, valid, _, _ = _l2_case(counts, I, K, True, 21, B.MOE_L2_ROWS_BF16)
    assert np.array_equal(got[valid], ref[valid])


@pytest.mark.parametrize("counts,I,K", [([40, 0, 170], 3072, 256), ([2], 192, 512)])
def test_l2_rows_random_scales(counts, I, K):
    got, ref, valid, _, _ = _l2_case(counts, I, K, False, 22, B.MOE_L2_ROWS_BF16, gs=0.5)
    assert_layer_close(got[valid], ref[valid], "y")


def test_l2_capacity_ends_at_last_expert():
    got, ref, valid, _, _ = _l2_case([129, 5], 256, 512, True, 25, B.MOE_L2_ROWS_BF16, tight=True)
    assert got.shape[0] == 384
    assert np.array_equal(got[valid], ref[valid])


def test_l2_scatter_weighted_sum():
    counts = [50, 0, 140, 7]
    rt, cap = _slots(counts)
    T = 90
    r = np.random.default_rng(23)
    st = np.full(cap, -1, np.int32)
    sw = np.zeros(cap, np.float32)
    for e in range(len(counts)):
        lo = rt["padded_offsets"][e]
        st[lo:lo + counts[e]] = r.integers(0, T, counts[e])
        sw[lo:lo + counts[e]] = r.random(counts[e]).astype(np.float32)
    y, ref, valid, out32, _ = _l2_case(counts, 256, 256, False, 24, B.MOE_L2_SCATTER, gs=0.3, slot_token=st,
                                       slot_weight=sw, T=T)
    expect = np.zeros((T, 256), np.float64)
    for p in np.nonzero(valid)[0]:
        expect[st[p]] += np.float64(sw[p]) * ref[p]
    assert_layer_close(out32, expect, "scatter")
