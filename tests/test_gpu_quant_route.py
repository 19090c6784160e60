"""GPU parity of the quantiser and the router against the oracle: bit-exact."""

import numpy as np
import pytest
import torch

import workloads
from oracle import nvfp4 as q
from oracle.route import route as oroute
from tests.helpers import bf16_dev

pytestmark = pytest.mark.gpu

B = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B
    from nvfp4_mixture_experts_stage_gb300 import binding
    B = binding


def _stage(x_f32, layout, gs_fixed=None):
    T, K = x_f32.shape
    x = bf16_dev(x_f32)
    codes = torch.zeros(T, K // 2, dtype=torch.uint8, device="cuda")
    rows = -(-T // 128) * 128 if layout == 1 else T
    sf = torch.zeros(rows * K // 16, dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(B.moe_stage_workspace_size(), dtype=torch.uint8, device="cuda")
    gfix = None if gs_fixed is None else torch.tensor([gs_fixed], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_stage_activation(x, codes, sf, layout, gs, gs_fixed=gfix, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return codes.cpu().numpy(), sf.cpu().numpy(), np.float32(gs.item())


def _rand_x(T, K, seed, scale=1.0, outliers=False):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, K)).astype(np.float32) * np.float32(scale)
    if outliers:
        x = np.where(r.random((T, K)) < 0.01, x * 20, x).astype(np.float32)
    return q.bf16_round(x)


@pytest.mark.parametrize("T,K,scale,outl", [(1, 64, 1.0, False), (7, 192, 1.0, True), (33, 320, 3.0, False),
                                            (130, 4096, 1.0, True), (256, 7168, 1e4, False),
                                            (5, 256, 1e-3, False), (64, 512, 1e30, False)])
@pytest.mark.parametrize("layout", [0, 1])
def test_stage_activation_bit_exact(T, K, scale, outl, layout):
    x = _rand_x(T, K, T * 1000 + K, scale, outl)
    codes, sf, gs = _stage(x, layout)
    rc, rs, rg = q.quantize(x)
    assert gs == rg
    assert np.array_equal(codes, rc)
    if layout == 0:
        assert np.array_equal(sf.reshape(T, K // 16), rs)
    else:
        assert np.array_equal(q.unswizzle(sf, T, K // 16), rs)


@pytest.mark.parametrize("gs_fixed", [1.0, 0.5, 1e-3, 7.0 / 2688.0, 0.0, 1e-42])
def test_stage_activation_fixed_scale_bit_exact(gs_fixed):
    x = _rand_x(48, 256, 5, 2.0, True)
    codes, sf, gs = _stage(x, 0, gs_fixed)
    rc, rs, _ = q.quantize(x, np.float32(gs_fixed))
    assert gs == np.float32(gs_fixed)
    assert np.array_equal(codes, rc)
    assert np.array_equal(sf.reshape(48, 16), rs)


def _golden_blocks():
    from tests.test_oracle_quantize import _golden_blocks as g
    return g()


@pytest.mark.parametrize("case", _golden_blocks(), ids=lambda c: c[0])
def test_hand_derived_blocks_on_device(case):
    """The hand-derived blocks of tests/golden/quant_blocks.txt (derived from the pages'
    encoding, not from either implementation) through the device quantiser: the block
    sits first in a 64-wide row of zeros (the API quantises 64 columns at a time), so its
    scale byte and codes must be the golden ones; "data" cases take the global scale from
    the row's amax (the block's own).  Every input is a BF16 value, subnormals included."""
    name, gs, x, sb, nibs, bts = case
    row = np.zeros((1, 64), np.float32)
    row[0, :16] = x
    assert np.array_equal(q.bf16_round(row), row)          # BF16 inputs, exactly
    codes, sf, g = _stage(row, 0, gs)
    assert sf[0] == sb
    assert list(codes[0, :8]) == bts
    assert not codes[0, 8:].any() and not sf[1:4].any()
    if gs is None:
        assert g == np.float32(1.0)


def _finite_bf16():
    f = q.bf16_from_bits(np.arange(65536, dtype=np.uint32).astype(np.uint16))
    return f[np.isfinite(f)]


def _blocks_to_rows(blocks):
    """[n, 16] blocks -> rows of K = 256 (zero blocks pad the last row)."""
    n = -(-len(blocks) // 16) * 16
    out = np.zeros((n, 16), np.float32)
    out[:len(blocks)] = blocks
    return out.reshape(-1, 256)


@pytest.mark.parametrize("bm", [6.0, 3.0, 0.375])
def test_every_bf16_value_codes_bit_exact(bm):
    """The E2M1 encoder on every finite BF16 value v with |v| <= bm, both signs and -0:
    each block holds bm and 15 such values, so with gs = 1 the block scale is bm/6 (an
    exact e4m3 value: 1, 0.5, 0.0625) and every code is the encoder's rounding of v*6/bm."""
    f = _finite_bf16()
    v = f[np.abs(f) <= bm]
    n = -(-len(v) // 15)
    vals = np.zeros(n * 15, np.float32)
    vals[:len(v)] = v
    blocks = np.concatenate([np.full((n, 1), bm, np.float32), vals.reshape(n, 15)], axis=1)
    x = _blocks_to_rows(blocks)
    codes, sf, _ = _stage(x, 0, 1.0)
    rc, rs, _ = q.quantize(x, np.float32(1.0))
    assert np.array_equal(codes, rc)
    assert np.array_equal(sf.reshape(rs.shape), rs)


@pytest.mark.parametrize("gs_fixed", [1.0, 1.0 / 3.0])
def test_every_bf16_block_max_scale_bit_exact(gs_fixed):
    """The E4M3 scale encoder on every positive finite BF16 block maximum bm (zero,
    subnormal, normal and saturating scales bm*rg/6), with the block's other values
    -bm, bm/2 and zeros."""
    f = _finite_bf16()
    bms = f[f > 0]
    blocks = np.zeros((len(bms), 16), np.float32)
    blocks[:, 0] = bms
    blocks[:, 1] = -bms
    blocks[:, 2] = q.bf16_round(bms / 2)
    x = _blocks_to_rows(blocks)
    codes, sf, _ = _stage(x, 0, gs_fixed)
    rc, rs, _ = q.quantize(x, np.float32(gs_fixed))
    assert np.array_equal(sf.reshape(rs.shape), rs)
    assert np.array_equal(codes, rc)


def test_stage_activation_ties_signs_and_golden_blocks():
    # every E2M1 tie and grid point, both signs, with scale 1 (block max 6, gs 1)
    vals = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0],
                    np.float32)
    rows = [vals, -vals, np.where(np.arange(16) % 2 == 0, -0.0, 0.0).astype(np.float32),
            np.array([6.0] + [1e-6] * 15, np.float32), np.array([-6.0] + [-1e-6] * 15, np.float32)]
    x = np.stack(rows).astype(np.float32)
    x = np.tile(x, (1, 4))
    codes, sf, gs = _stage(x, 0, 1.0)
    rc, rs, _ = q.quantize(x, np.float32(1.0))
    assert np.array_equal(codes, rc)
    assert np.array_equal(sf.reshape(len(rows), 4), rs)
    # -0.0 and tiny negatives code as 0x8 (sign bit kept)
    assert np.all(q.unpack_nibbles(codes)[2, 0::2] == 8)


def test_stage_activation_all_zero():
    x = np.zeros((3, 64), np.float32)
    codes, sf, gs = _stage(x, 0)
    assert gs == 0.0 and not codes.any() and not sf.any()


def _route_dev(ids, w, E, off):
    T, k = ids.shape
    cap = B.moe_slot_capacity(T, k, E)
    d = lambda n, dt=torch.int32: torch.full((n,), -7, dtype=dt, device="cuda")
    counts, offs, poff = d(E), d(E + 1), d(E + 1)
    st, sw, ps = d(cap), d(cap, torch.float32), d(T * k)
    ws = torch.empty(B.moe_route_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    B.moe_route(torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), E, off, counts, offs, poff, st, sw, ps, ws)
    torch.cuda.synchronize()
    return {k_: v.cpu().numpy() for k_, v in dict(counts=counts, offsets=offs, padded_offsets=poff,
                                                   slot_token=st, slot_weight=sw, pair_slot=ps).items()}


def _check_route(ids, w, E, off):
    got = _route_dev(ids, w, E, off)
    ref = oroute(ids, w, E, off)
    for k_ in ref:
        assert np.array_equal(got[k_], ref[k_]), k_
    return got


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skew_top1", "skew_top8", "sweep_1k",
                                  "sweep_64k"])
def test_route_bit_exact_on_workloads(name):
    wl = workloads.WORKLOADS[name]
    ids, w = workloads.routing(wl)
    _check_route(ids, w, wl.E, wl.expert_offset)


@pytest.mark.parametrize("seed", range(4))
def test_route_bit_exact_random_with_invalid_ids(seed):
    r = np.random.default_rng(100 + seed)
    T, k, E = int(r.integers(1, 3000)), int(r.integers(1, 9)), int(r.integers(1, 257))
    off = int(r.integers(0, 4)) * E
    ids = r.integers(-3, 5 * E, (T, k)).astype(np.int32)
    w = r.random((T, k)).astype(np.float32)
    _check_route(ids, w, E, off)


@pytest.mark.parametrize("P", [4096, 4097, 8192, 8193])
def test_route_bit_exact_at_path_boundaries(P):
    """Pair counts around the switch from the one-block kernel to the chunked kernels."""
    r = np.random.default_rng(P)
    k, E = 1, 48
    ids = r.integers(0, E + 8, (P, k)).astype(np.int32)   # some pairs belong to other ranks
    w = r.random((P, k)).astype(np.float32)
    _check_route(ids, w, E, 0)


def test_route_identity_for_sorted_top1():
    wl = workloads.WORKLOADS["skew_top1"]
    ids, w = workloads.routing(wl)
    got = _check_route(ids, w, wl.E, wl.expert_offset)
    st = got["slot_token"]
    assert np.array_equal(st[st >= 0], np.arange(wl.T))


def test_route_no_local_experts():
    ids = np.full((40, 3), 999, np.int32)
    w = np.ones((40, 3), np.float32)
    got = _check_route(ids, w, 8, 0)
    assert got["offsets"][-1] == 0 and np.all(got["pair_slot"] == -1)


@pytest.mark.parametrize("T,K,topk,E,nonlocal_", [(300, 512, 3, 5, False), (77, 320, 8, 10, False),
                                                  (64, 4096, 8, 48, True), (50, 256, 9, 12, False),
                                                  (129, 1152, 2, 4, True)])
def test_stage_to_slots_bit_exact(T, K, topk, E, nonlocal_):
    """Every slot holds its token's codes and scales: runs of segments ending inside a
    row (K = 320, 1152), top-8, top-9 (the general kernel), pairs of other ranks' experts
    (no slot)."""
    wl = workloads.small("slots", T=T, K=K, I=64, E=E, topk=topk)
    ids, w = workloads.routing(wl)
    if nonlocal_:
        ids = ids.copy()
        ids[::3] += E          # every third pair belongs to another rank
    x = workloads.activations(wl)
    rt = oroute(ids, w, wl.E, 0)
    cap = B.moe_slot_capacity(wl.T, wl.topk, wl.E)
    a = torch.zeros(cap, wl.K // 2, dtype=torch.uint8, device="cuda")
    asf = torch.zeros(cap * wl.K // 16, dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(B.moe_stage_workspace_size(), dtype=torch.uint8, device="cuda")
    B.moe_stage_activation_to_slots(x.cuda(), torch.from_numpy(rt["pair_slot"]).cuda(), wl.topk, cap, a, asf, gs,
                                    ws=ws)
    torch.cuda.synchronize()
    rc, rs, rg = q.quantize(x.float().numpy())
    # the oracle's slot table ends at the last expert's padded end; rows after it stay zero
    slot_token = np.full(cap, -1, np.int64)
    slot_token[:len(rt["slot_token"])] = rt["slot_token"]
    valid = slot_token >= 0
    assert np.float32(gs.item()) == rg
    got = a.cpu().numpy()
    assert np.array_equal(got[valid], rc[slot_token[valid]])
    assert not got[len(rt["slot_token"]):].any()
    got_sf = q.unswizzle(asf.cpu().numpy(), cap, wl.K // 16)
    assert np.array_equal(got_sf[valid], rs[slot_token[valid]])


def test_prepare_weights_layout():
    r = np.random.default_rng(3)
    E, I, K = 3, 192, 256
    sf1 = r.integers(0, 127, (E, 2 * I, K // 16)).astype(np.uint8)
    sf2 = r.integers(0, 127, (E, K, I // 16)).astype(np.uint8)
    d1 = torch.empty(sf1.size, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(sf2.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(torch.from_numpy(sf1).cuda(), d1, E, 2 * I, K, B.MOE_PREP_W1)
    B.moe_prepare_weights(torch.from_numpy(sf2).cuda(), d2, E, K, I, B.MOE_PREP_W2)
    torch.cuda.synchronize()
    g1 = d1.cpu().numpy().reshape(E, -1)
    g2 = d2.cpu().numpy().reshape(E, -1)
    for e in range(E):
        assert np.array_equal(q.unswizzle(g2[e], K, I // 16), sf2[e])
        # W1: atoms hold 64 gate rows then the 64 matching up rows
        inter = np.concatenate([np.concatenate([sf1[e, 64 * j:64 * j + 64], sf1[e, I + 64 * j:I + 64 * j + 64]])
                                for j in range(I // 64)])
        assert np.array_equal(q.unswizzle(g1[e], 2 * I, K // 16), inter)


@pytest.mark.parametrize("gg,gu", [(1e-2, 6e-3), (2e-3, 8e-3), (5e-4, 5e-4), (0.0, 0.0), (1e-2, 1e-9),
                                   (3e-3, 3e-3 / 1024), (7.0, 0.0)])
def test_fold_gate_up_scales_bit_exact(gg, gu):
    """The pages' one-alpha W1 form: the GPU fold of every scale byte equals the oracle's."""
    from oracle import moe as omoe
    E, I, K = 3, 128, 2048
    r = np.random.default_rng(int(gg * 1e4) + int(gu * 1e6) + 11)
    sf = r.integers(0, 0x7F, (E, 2 * I, K // 16)).astype(np.uint8)
    sf[:, 0, :127] = np.arange(127)          # every finite byte in both halves
    sf[:, I, :127] = np.arange(127)
    g_gate = np.array([gg, gg * 0.5, 1e-3], np.float32)
    g_up = np.array([gu, gu, 1e-3], np.float32)
    d = torch.from_numpy(sf.copy()).cuda()
    common = torch.zeros(E, dtype=torch.float32, device="cuda")
    B.moe_fold_gate_up_scales(d, torch.from_numpy(g_gate).cuda(), torch.from_numpy(g_up).cuda(), common)
    torch.cuda.synchronize()
    ref, rcommon = omoe.fold_gate_up_scales(sf, g_gate, g_up)
    assert np.array_equal(d.cpu().numpy(), ref)
    assert np.array_equal(common.cpu().numpy(), rcommon)



def test_quantize_weights_on_device_bit_exact():
    """moe_quantize_weights: codes and global scales equal the oracle's per-projection
    quantisation; the scales equal moe_prepare_weights of the oracle's row-major ones."""
    from oracle import moe as omoe
    E, I, K = 3, 128, 256
    r = np.random.default_rng(12)
    w1 = q.bf16_round((r.standard_normal((E, 2 * I, K)) * 0.02).astype(np.float32))
    w2 = q.bf16_round((r.standard_normal((E, K, I)) * 0.02).astype(np.float32))
    w1[1, :I] = q.bf16_round(w1[1, :I] * 50)  # gate and up of expert 1 on different scales
    ref = omoe.quantize_weights(w1, w2)
    t = lambda a: torch.from_numpy(a).to(torch.bfloat16).cuda()
    u8 = lambda *sh: torch.zeros(*sh, dtype=torch.uint8, device="cuda")
    f32 = lambda n: torch.zeros(n, dtype=torch.float32, device="cuda")
    w1c, w1s, w2c, w2s = u8(E, 2 * I, K // 2), u8(E * 2 * I * K // 16), u8(E, K, I // 2), u8(E * K * I // 16)
    gg, gu, g2 = f32(E), f32(E), f32(E)
    ws = u8(B.moe_quantize_weights_workspace_size(E, I, K))
    B.moe_quantize_weights(t(w1), t(w2), w1c, w1s, gg, gu, w2c, w2s, g2, ws)
    torch.cuda.synchronize()
    assert np.array_equal(w1c.cpu().numpy(), ref["w1_codes"])
    assert np.array_equal(w2c.cpu().numpy(), ref["w2_codes"])
    for got, key in ((gg, "gs_w1_gate"), (gu, "gs_w1_up"), (g2, "gs_w2")):
        assert np.array_equal(got.cpu().numpy(), ref[key])
    e1 = torch.empty_like(w1s)
    e2 = torch.empty_like(w2s)
    B.moe_prepare_weights(torch.from_numpy(ref["w1_sf"]).cuda(), e1, E, 2 * I, K, B.MOE_PREP_W1)
    B.moe_prepare_weights(torch.from_numpy(ref["w2_sf"]).cuda(), e2, E, K, I, B.MOE_PREP_W2)
    torch.cuda.synchronize()
    assert torch.equal(w1s, e1) and torch.equal(w2s, e2)


@pytest.mark.parametrize("cap,I,big", [(384, 192, False), (256, 3072, True), (128, 64, False)])
def test_requant_bit_exact_on_masked_rows(cap, I, big):
    """moe_requant (the dynamic h scale's pass, teacher-forced): given BF16 h and the max
    |h| over the valid rows, the codes, swizzled scales and the h global scale equal the
    oracle's quantisation of the valid rows; padding rows are not written."""
    r = np.random.default_rng(cap + I)
    h = q.bf16_round(r.standard_normal((cap, I)).astype(np.float32))
    if big:
        h[5] = q.bf16_round(h[5] * 1e4)
    st = np.where(r.random(cap) < 0.6, np.arange(cap), -1).astype(np.int32)
    st[5] = 5
    valid = st >= 0
    amax = np.float32(np.abs(h[valid]).max())
    hd = torch.from_numpy(h).to(torch.bfloat16).cuda()
    codes = torch.zeros(cap, I // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(cap * I // 16, dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    stat = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_requant(hd, torch.from_numpy(st).cuda(), torch.tensor([amax], device="cuda"), gs, codes, sf, dev_status=stat)
    torch.cuda.synchronize()
    assert stat.item() == 0
    rc, rs, rg = q.quantize(h[valid])
    assert np.float32(gs.item()) == rg
    got = codes.cpu().numpy()
    assert np.array_equal(got[valid], rc)
    assert not got[~valid].any()
    got_sf = q.unswizzle(sf.cpu().numpy(), cap, I // 16)
    assert np.array_equal(got_sf[valid], rs)
    assert not got_sf[~valid].any()
