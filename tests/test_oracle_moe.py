"""Pins for the oracle's GEMMs and whole layer (CPU only).

* a per-token brute force with no slot machinery (Python loops, exact
  rational dot products) must reproduce the grouped oracle;
* an exact-arithmetic case (all block scales 1, alpha 1) against integer dot
  products;
* top-1 with unit weights reduces the layer to a dense per-token FFN;
* simulated expert parallelism: rank-local outputs sum to the all-expert
  layer;
* the tests-page "scale transpose" commit's failure mode (weight scales read
  as (K_sf, N)) collapses the cosine;
* SiLU identities.
"""

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads
from oracle import moe, nvfp4 as q
from oracle.route import route

F32 = np.float32


def _tiny_weights(wl):
    w1 = np.stack([workloads.expert_w1(wl, e).float().numpy() for e in range(wl.E)])
    w2 = np.stack([workloads.expert_w2(wl, e).float().numpy() for e in range(wl.E)])
    return moe.quantize_weights(w1, w2)


# independent decoders for the brute force: torch's float8 view for scales and
# the golden nibble table for codes
_NIB = {}
for _line in open(__file__.replace("test_oracle_moe.py", "golden/e2m1_grid.txt")):
    if _line.strip() and not _line.startswith("#"):
        a, b = _line.split()
        _NIB[int(a)] = Fraction(b) if float(b) != 0 else Fraction(0)


def _scale(b):
    return Fraction(float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float()))


def _row_values(codes_row, sf_row):
    vals = []
    for i in range(codes_row.size * 2):
        byte = int(codes_row[i // 2])
        nib = (byte >> 4) if i % 2 else (byte & 0xF)
        vals.append(_NIB[nib] * _scale(sf_row[i // 16]))
    return vals


def _f32(fr):
    """Nearest fp32 of an exact rational (via fp64; no ties occur here)."""
    return F32(float(fr))


def _bf16(f):
    return F32(torch.tensor([float(f)], dtype=torch.float32).to(torch.bfloat16).float().item())


def _silu_ref(g):
    e = F32(math.exp(-float(g))) if -float(g) < 88 else F32(np.inf)
    return F32(F32(g) / (F32(1.0) + e))


def test_layer_matches_per_token_brute_force():
    wl = workloads.small("bf", T=5, K=64, I=64, E=3, topk=2, routing="softmax_topk",
                         x_kind="outliers")
    x = workloads.activations(wl).float().numpy()
    ids, w = workloads.routing(wl)
    W = _tiny_weights(wl)
    ref = moe.forward(x, ids, w, wl.E, 0, W)

    xc, xs, gs_x = q.quantize(x)
    I, K = wl.I, wl.K
    # L1 + SiLU per (token, j), no slots
    hs = {}
    for t in range(wl.T):
        a = _row_values(xc[t], xs[t])
        for j in range(wl.topk):
            e = int(ids[t, j])
            ag = F32(gs_x * W["gs_w1_gate"][e])
            au = F32(gs_x * W["gs_w1_up"][e])
            h = np.empty(I, F32)
            for n in range(I):
                wg = _row_values(W["w1_codes"][e, n], W["w1_sf"][e, n])
                wu = _row_values(W["w1_codes"][e, I + n], W["w1_sf"][e, I + n])
                g = _bf16(F32(ag * _f32(sum(p * r for p, r in zip(a, wg)))))
                u = _bf16(F32(au * _f32(sum(p * r for p, r in zip(a, wu)))))
                h[n] = _bf16(F32(_silu_ref(g) * u))
            hs[t, j] = h
    amax = max(float(np.abs(v).max()) for v in hs.values())
    gs_h = F32(F32(amax) / F32(2688.0))
    out = np.zeros((wl.T, K), F32)
    for t in range(wl.T):
        acc = np.zeros(K, F32)
        for j in range(wl.topk):
            e = int(ids[t, j])
            hc, hsf, _ = q.quantize(hs[t, j][None, :], gs_h)
            hv = _row_values(hc[0], hsf[0])
            a2 = F32(gs_h * W["gs_w2"][e])
            y = np.array([_bf16(F32(a2 * _f32(sum(p * r for p, r in zip(
                hv, _row_values(W["w2_codes"][e, n], W["w2_sf"][e, n])))))) for n in range(K)], F32)
            acc = acc + F32(w[t, j]) * y
        out[t] = q.bf16_round(acc)
    assert ref["gs_h"] == gs_h
    assert np.array_equal(ref["out"], out)


def test_exact_arithmetic_gemm_equals_integer_dot_products():
    r = np.random.default_rng(11)
    M, N, K = 7, 9, 128
    ac = r.integers(0, 256, (M, K // 2)).astype(np.uint8)
    wc = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    ones_a = np.full((M, K // 16), 0x38, np.uint8)
    ones_w = np.full((N, K // 16), 0x38, np.uint8)
    acc = moe.expert_gemm(ac, ones_a, wc, ones_w)
    # integer arithmetic in units of 1/4: value*2 is an integer for every code
    def ints(c):
        nib = np.stack([c & 0xF, c >> 4], -1).reshape(c.shape[0], -1)
        mag = np.array([0, 1, 2, 3, 4, 6, 8, 12])[nib & 7]
        return np.where(nib & 8, -mag, mag).astype(np.int64)
    exact = ints(ac) @ ints(wc).T            # = 4 * sum
    assert np.array_equal(acc * 4, exact.astype(np.float32))


def test_gemm_is_the_exact_sum_rounded_once():
    """Closed form: with random scales the fp64 contraction, rounded to fp32,
    equals the exact rational sum rounded to fp32 (within one fp32 ulp for the
    double rounding)."""
    r = np.random.default_rng(12)
    M, N, K = 3, 4, 96
    ac = r.integers(0, 256, (M, K // 2)).astype(np.uint8)
    wc = r.integers(0, 256, (N, K // 2)).astype(np.uint8)
    asf = r.integers(0x10, 0x60, (M, K // 16)).astype(np.uint8)
    wsf = r.integers(0x10, 0x60, (N, K // 16)).astype(np.uint8)
    acc = moe.expert_gemm(ac, asf, wc, wsf)
    for m in range(M):
        a = _row_values(ac[m], asf[m])
        for n in range(N):
            ex = sum(p * q_ for p, q_ in zip(a, _row_values(wc[n], wsf[n])))
            ref = F32(float(ex))
            assert abs(acc[m, n] - ref) <= np.spacing(np.abs(ref))


def test_top1_unit_weight_is_a_dense_ffn():
    wl = workloads.small("d", T=6, K=64, I=64, E=4, topk=1)
    x = workloads.activations(wl).float().numpy()
    ids = np.array([[0], [3], [1], [0], [2], [3]], np.int32)
    w = np.ones((6, 1), np.float32)
    W = _tiny_weights(wl)
    res = moe.forward(x, ids, w, 4, 0, W)
    ps = res["route"]["pair_slot"]
    assert np.array_equal(res["out"], res["y"][ps])


def test_simulated_expert_parallel_ranks_sum_to_all_experts():
    """The "global expert ids" commit: each rank computes its local experts'
    share; the caller's reduction of the rank outputs gives the full layer."""
    wl = workloads.small("ep", T=12, K=64, I=64, E=16, topk=3)
    x = workloads.activations(wl).float().numpy()
    ids, w = workloads.routing(wl)
    W = _tiny_weights(wl)
    gs_h = F32(1.0 / 2688.0)
    full = moe.forward(x, ids, w, 16, 0, W, gs_h=gs_h)["out"]
    total = np.zeros_like(full)
    for rank in range(4):
        sl = slice(4 * rank, 4 * rank + 4)
        Wr = {k: (v[sl] if isinstance(v, np.ndarray) and v.shape[0] == 16 else v)
              for k, v in W.items()}
        total += moe.forward(x, ids, w, 4, 4 * rank, Wr, gs_h=gs_h)["out"]
    err = np.abs(total - full).max()
    assert err <= 1e-2 * np.abs(full).max()
    cos = (total * full).sum() / np.sqrt((total ** 2).sum() * (full ** 2).sum())
    assert cos > 0.9999


def test_transposed_weight_scales_collapse_the_output():
    """Mirror of the tests-page "scale transpose" commit: scales stored as
    (N, K_sf) but read as if they were (K_sf, N) scramble the layer."""
    wl = workloads.small("m2", T=32, K=128, I=128, E=2, topk=1)
    x = workloads.activations(wl).float().numpy()
    ids, w = workloads.routing(wl)
    W = _tiny_weights(wl)
    good = moe.forward(x, ids, w, 2, 0, W)["out"]
    bad_w = dict(W)
    E, N, ksf = W["w1_sf"].shape
    bad_w["w1_sf"] = W["w1_sf"].transpose(0, 2, 1).reshape(E, N, ksf).copy()
    bad = moe.forward(x, ids, w, 2, 0, bad_w)["out"]
    cos = (good * bad).sum() / np.sqrt((good ** 2).sum() * (bad ** 2).sum())
    assert cos < 0.95


def test_silu_identities():
    g = q.bf16_round(np.random.default_rng(13).standard_normal(10000).astype(F32) * 8)
    one = np.ones_like(g)
    s = moe.silu_mul(g, one)           # bf16(silu(g))
    assert moe.silu_mul(np.zeros(1, F32), np.ones(1, F32))[0] == 0.0
    # silu(x) - silu(-x) = x  (each side rounded to bf16: within 2 bf16 ulps of x)
    d = s - moe.silu_mul(-g, one)
    assert np.all(np.abs(d - g) <= 2 * np.abs(g) * 2.0 ** -8 + 1e-30)
    # against an fp64 reference
    ref = g.astype(np.float64) / (1 + np.exp(-g.astype(np.float64)))
    assert np.all(np.abs(s - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)
    # large negative gate -> -0/0, large positive -> g
    assert moe.silu_mul(np.array([-200.0], F32), np.ones(1, F32))[0] == 0.0
    assert moe.silu_mul(np.array([200.0], F32), np.ones(1, F32))[0] == 200.0


def test_bf16_reference_layer_brute_force_and_close_to_nvfp4():
    """The unquantised reference layer: a plain per-token loop over the dense
    projections reproduces it, and the NVFP4 layer stays close to it (block-scaled
    FP4 keeps the outputs well correlated; the pages report cosines of 0.989-0.995 on
    a real checkpoint)."""
    import workloads
    from oracle import moe as omoe, nvfp4 as q
    wl = workloads.WORKLOADS["tiny"]
    x = workloads.activations(wl).float().numpy()
    ids, w = workloads.routing(wl)
    w1 = lambda e: workloads.expert_w1(wl, e).float().numpy()
    w2 = lambda e: workloads.expert_w2(wl, e).float().numpy()
    ref = omoe.forward_bf16(x, ids, w, wl.E, wl.expert_offset, w1, w2)
    # brute force: float64 throughout, rounding at the same points
    bf = lambda a: q.bf16_round(np.asarray(a, np.float32))
    for t in (0, 7, wl.T - 1):
        acc = np.zeros(wl.K, np.float32)
        for j in range(wl.topk):
            e = int(ids[t, j]) - wl.expert_offset
            W1, W2 = w1(e).astype(np.float64), w2(e).astype(np.float64)
            g = bf(W1[:wl.I] @ x[t])
            u = bf(W1[wl.I:] @ x[t])
            h = bf((g / (1 + np.exp(-g.astype(np.float64)).astype(np.float32))).astype(np.float32) * u)
            y = bf(W2 @ h.astype(np.float64))
            acc = acc + np.float32(w[t, j]) * y
        assert np.array_equal(ref[t], bf(acc))
    W = omoe.quantize_weights(np.stack([w1(e) for e in range(wl.E)]), np.stack([w2(e) for e in range(wl.E)]))
    out = omoe.forward(x, ids, w, wl.E, wl.expert_offset, W)["out"]
    cos = float((out * ref).sum() / np.sqrt((out * out).sum() * (ref * ref).sum()))
    assert cos > 0.95   # 0.975 here: the tiny inputs carry 1 % outliers at 20x


def test_bf16_reference_layer_closed_form():
    """forward_bf16 on a hand-built layer whose every intermediate is known exactly, so
    each BF16 rounding point of the pages' pipeline ([tests] "complete pipeline": L1 out
    g and u in BF16, SiLU(g) * up in BF16, L2 out in BF16, the weighted sum in BF16) and
    the gate/up split show in the output.  One token, x = e_0 (so g and u are column 0
    of the gate and up rows), two local experts with routing weights 1 and 0.5.

    Expert 0 (gate, up) in column 0, by row i of h:
      i=0: (128.75, 1.5)         g = bf16(128.75) = 129 (spacing 1 on [128, 256));
                                 silu(129) = 129 exactly in fp32 (exp(-129) underflows);
                                 h = bf16(193.5) = 194 (tie -> even mantissa)
      i=1: (192, 1.005859375)    u = bf16(1 + 3/512) = 1.0078125; h = bf16(193.5) = 194
      i=2: (0, 5)                silu(0) = 0 -> h = 0
      i=3: (-192, 5)             exp(192) overflows fp32: silu = -192/inf = -0 -> h = 0
      i=4: (128, 1)              h = 128
      i=5: (1, 1)                silu(1) = 1/(1 + e^-1) = 0.7310586 -> h = bf16 = 0.73046875
                                 (187.15 steps of 2^-8, far from a rounding midpoint)
    Expert 0 down rows (output column k: weights on h):
      k=0: 1*h0                  -> 194
      k=1: 1*h0 + 2^-9*h1        -> bf16(194.37890625) = 194
      k=2: 1*h0 - 1.5078125*h4   -> 194 - 193 = 1
      k=3: 1*h1 - 1.5078125*h4   -> 1
      k=4: 1*h2 + 1*h3           -> 0
      k=5: 1*h5                  -> 0.73046875
    Expert 1: gate/up (128, 1) in row 0 -> h'0 = 128; down row k=1: 0.005859375*h'0 = 0.75.
    out = bf16(1*y0 + 0.5*y1), in fp32: k=1 gives bf16(194 + 0.375) = 194; the rest as y0.

    A missing rounding of g gives 193 in column 0 (h0 = bf16(128.75*1.5) = 193); of u gives
    0 in column 3 (h1 = 193); of h gives 0.5 in column 2; of y gives 195 in column 1
    (194.3789 + 0.375); of the output gives 194.375 in column 1; gate and up swapped give
    other values in column 0; a sign error in SiLU gives -960 in column 4."""
    K, I, E = 16, 16, 2
    x = np.zeros((1, K), F32)
    x[0, 0] = 1.0
    w1 = np.zeros((E, 2 * I, K), F32)
    w2 = np.zeros((E, K, I), F32)
    for i, (g, u) in enumerate([(128.75, 1.5), (192.0, 1.005859375), (0.0, 5.0), (-192.0, 5.0), (128.0, 1.0),
                                (1.0, 1.0)]):
        w1[0, i, 0], w1[0, I + i, 0] = g, u
    w2[0, 0, 0] = 1.0
    w2[0, 1, 0], w2[0, 1, 1] = 1.0, 2.0 ** -9
    w2[0, 2, 0], w2[0, 2, 4] = 1.0, -1.5078125
    w2[0, 3, 1], w2[0, 3, 4] = 1.0, -1.5078125
    w2[0, 4, 2], w2[0, 4, 3] = 1.0, 1.0
    w2[0, 5, 5] = 1.0
    w1[1, 0, 0], w1[1, I, 0] = 128.0, 1.0
    w2[1, 1, 0] = 0.005859375
    ids = np.array([[0, 1]], np.int32)
    wts = np.array([[1.0, 0.5]], F32)
    out = moe.forward_bf16(x, ids, wts, E, 0, lambda e: w1[e], lambda e: w2[e])
    expect = np.zeros(K, F32)
    expect[:6] = [194.0, 194.0, 1.0, 1.0, 0.0, 0.73046875]
    assert out.shape == (1, K)
    assert np.array_equal(out[0], expect), out[0]
    # tokens routed to no local expert (foreign id, -1) give exactly zero
    out2 = moe.forward_bf16(np.concatenate([x, x]), np.array([[0, 1], [5, -1]], np.int32),
                            np.concatenate([wts, wts]), E, 0, lambda e: w1[e], lambda e: w2[e])
    assert np.array_equal(out2[0], expect) and not out2[1].any()


# ------------------------------------------------------------- gate/up scale fold
def _nearest_e4m3_brute(v):
    """Nearest UE4M3 byte to v >= 0 by search over every finite byte (torch's float8
    view decodes them), ties to the even byte (even mantissa)."""
    best, best_d = None, None
    for b in range(0x7F):
        d = abs(_scale(b) - Fraction(float(v)))
        if best is None or d < best_d or (d == best_d and b % 2 == 0):
            best, best_d = b, d
    return best


def test_fold_equal_scales_is_identity():
    r = np.random.default_rng(40)
    sf = r.integers(0, 0x7F, (3, 16, 4)).astype(np.uint8)
    g = np.array([1e-3, 2.5e-4, 0.0], F32)
    out, common = moe.fold_gate_up_scales(sf, g, g)
    assert np.array_equal(out, sf) and np.array_equal(common, g)


def test_fold_power_of_two_ratio_shifts_the_exponent():
    """gs_up = gs_gate / 4: every up scale whose exponent field is at least 3 drops by two
    binades (byte - 16) and the gate half is untouched; the common scale is gs_gate."""
    sf = np.tile(np.arange(0, 0x7F, dtype=np.uint8), (2, 1)).reshape(1, 2, 127)   # gate row, up row
    out, common = moe.fold_gate_up_scales(sf, np.array([8e-3], F32), np.array([2e-3], F32))
    assert common[0] == F32(8e-3)
    assert np.array_equal(out[0, 0], sf[0, 0])
    normal = np.arange(127) >= 3 * 8
    assert np.array_equal(out[0, 1][normal], (np.arange(127)[normal] - 16).astype(np.uint8))


@pytest.mark.parametrize("ratio_num,ratio_den", [(3, 5), (1, 3), (7, 1000), (1, 1 << 20)])
def test_fold_matches_nearest_search_on_every_byte(ratio_num, ratio_den):
    """Every finite scale byte times an arbitrary ratio lands on the nearest UE4M3 value
    (brute-force search over all bytes, ties even), the gate half being the larger."""
    gate = F32(1e-2)
    up = F32(F32(gate) * F32(ratio_num / ratio_den))
    sf = np.tile(np.arange(0, 0x7F, dtype=np.uint8), (2, 1)).reshape(1, 2, 127)
    out, common = moe.fold_gate_up_scales(sf, np.array([gate]), np.array([up]))
    ratio = F32(up) / F32(gate)
    for b in range(0x7F):
        v = F32(F32(float(_scale(b))) * ratio)
        assert out[0, 1, b] == _nearest_e4m3_brute(v), (b, float(v))
    assert np.array_equal(out[0, 0], sf[0, 0])
    # the folded weights, at the common scale, equal the original ones within the
    # UE4M3 rounding of the folded scale (half a step: 2**-4 relative for normal values)
    orig = np.array([float(_scale(b)) for b in range(127)]) * float(up)
    new = np.array([float(_scale(b)) for b in out[0, 1]]) * float(common[0])
    normal = new >= 2.0 ** -6 * float(common[0])
    assert np.all(np.abs(new - orig)[normal] <= 2.0 ** -4 * orig[normal] * (1 + 1e-6))


def test_fold_gives_one_alpha_l1_close_to_two_alphas():
    """L1 with the folded scales and one alpha per expert stays within the UE4M3 rounding
    of the exact two-alpha L1 (the pages' accuracy trade-off)."""
    wl = workloads.WORKLOADS["tiny"]
    W = _tiny_weights(wl)
    x = workloads.activations(wl).float().numpy()
    ids, w = workloads.routing(wl)
    rt = route(ids, w, wl.E, wl.expert_offset)
    a_codes, a_sf, gs_x = q.quantize(q.bf16_round(x))
    ac = np.zeros((len(rt["slot_token"]), wl.K // 2), np.uint8)
    asf = np.zeros((len(rt["slot_token"]), wl.K // 16), np.uint8)
    valid = rt["slot_token"] >= 0
    ac[valid], asf[valid] = a_codes[rt["slot_token"][valid]], a_sf[rt["slot_token"][valid]]
    g2, u2 = moe.gemm_l1(ac, asf, gs_x, rt, W["w1_codes"], W["w1_sf"], W["gs_w1_gate"], W["gs_w1_up"])
    fsf, common = moe.fold_gate_up_scales(W["w1_sf"], W["gs_w1_gate"], W["gs_w1_up"])
    assert not np.array_equal(fsf, W["w1_sf"])      # the two halves' scales differ here
    g1, u1 = moe.gemm_l1(ac, asf, gs_x, rt, W["w1_codes"], fsf, common, common)
    for a, b in ((g1, g2), (u1, u2)):
        a, b = a[valid].astype(np.float64), b[valid].astype(np.float64)
        assert np.abs(a - b).max() <= 0.1 * np.abs(b).max()
        assert float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum())) > 0.99


def test_quantize_weights_gate_up_split_scales_and_error_bound():
    """oracle.moe.quantize_weights against closed forms: the gate rows (0..I-1), the up
    rows (I..2I-1) and each down projection get their own global scale amax / 2688
    (fp32 division), scales are row-major [N, K/16], and every dequantised weight q is
    within s * gs of the weight w, s its decoded block scale: in scaled units the error
    is at most half the widest gap of the E2M1 grid (4 to 6), or the overshoot past 6
    when the block scale rounded down (under 0.4)."""
    r = np.random.default_rng(21)
    E, I, K = 3, 32, 64
    w1 = q.bf16_round(r.standard_normal((E, 2 * I, K)).astype(F32) * 0.02)
    w1[:, :I] *= F32(50.0)                       # gate rows far larger than up rows
    w1 = q.bf16_round(w1)
    w2 = q.bf16_round(r.standard_normal((E, K, I)).astype(F32) * 0.03)
    W = moe.quantize_weights(w1, w2)
    assert W["w1_codes"].shape == (E, 2 * I, K // 2) and W["w1_sf"].shape == (E, 2 * I, K // 16)
    assert W["w2_codes"].shape == (E, K, I // 2) and W["w2_sf"].shape == (E, K, I // 16)
    for e in range(E):
        halves = ((slice(0, I), W["gs_w1_gate"][e]), (slice(I, 2 * I), W["gs_w1_up"][e]))
        for rows, gs in halves:
            assert gs == F32(np.abs(w1[e, rows]).max()) / F32(2688.0)
            deq = q.dequantize(W["w1_codes"][e, rows], W["w1_sf"][e, rows]) * float(gs)
            step = np.repeat(q.e4m3_decode(W["w1_sf"][e, rows]).astype(np.float64), 16, axis=1) * float(gs)
            assert np.all(np.abs(w1[e, rows] - deq) <= step * (1 + 1e-6))
        assert W["gs_w2"][e] == F32(np.abs(w2[e]).max()) / F32(2688.0)
        deq2 = q.dequantize(W["w2_codes"][e], W["w2_sf"][e]) * float(W["gs_w2"][e])
        step2 = np.repeat(q.e4m3_decode(W["w2_sf"][e]).astype(np.float64), 16, axis=1) * float(W["gs_w2"][e])
        assert np.all(np.abs(w2[e] - deq2) <= step2 * (1 + 1e-6))
    assert np.all(W["gs_w1_gate"] > 20 * W["gs_w1_up"])
