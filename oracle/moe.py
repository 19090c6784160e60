"""Grouped GEMMs, SiLU*up, requantisation, weighted combine and the whole MoE
layer, restated on the CPU (oracle; test infrastructure only).

Sources on the nvfp4-megamoe-kernel commit pages:

* commits of ``src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py``, the "global
  scale as alpha" commit: each GEMM computes D = alpha * (A @ B) with alpha the
  product of the activation and weight global scales, and the output of the
  layer is the rank-local sum (the cross-rank reduction belongs to the caller);
* commits of ``vllm/nvfp4_cutedsl.py``: the "intermediate_size" commit (the L1
  output is [gate | up], split at I, not I/2), the "dual global scale" commit
  (gate and up carry different weight global scales), the "CUDA graph" commit
  (weighted scatter_add over slots, zero weight on padding) and the "calibrated
  global scale" commit (a fixed activation global scale may replace the
  per-call amax);
* commits of ``tests``: the "complete pipeline" commit -- BF16 -> NVFP4,
  L1 GEMM NVFP4 x NVFP4 -> BF16 (gate|up), SiLU(gate) * up in BF16,
  requantisation to NVFP4, L2 GEMM -> BF16, routing-weighted scatter -> BF16.

Arithmetic (readings where the pages are silent):

* GEMM: operands are dequantised exactly (E2M1 value x UE4M3 scale) in fp64,
  the contraction runs in fp64 (every product is exact there; the sum of
  K <= 2**13 terms has error far below one fp32 ulp), the result is rounded
  once to fp32, multiplied by alpha in fp32 and rounded to BF16 (ties even);
* alpha = fp32(gs_activation * gs_weight); for L1 the gate half uses the gate
  weight scale and the up half the up weight scale (two alphas per expert
  instead of the pages' folding of the ratio into the block scales);
* SiLU: silu(g) = g / (1 + exp(-g)) in fp32 with exp rounded from fp64;
  h = bf16(silu(g) * u) with g and u the BF16 L1 outputs;
* combine: out[t] = bf16(sum_j fp32(w[t, j] * y[slot(t, j)])) summed in j
  order in fp32 from 0; tokens with no local expert give 0.
"""

import numpy as np

from . import nvfp4
from .route import route as route_pairs

F32 = np.float32


def expert_gemm(a_codes, a_sf, w_codes, w_sf):
    """fp32(sum_k deq(A)[m, k] * deq(W)[n, k]) for one expert.

    a_codes [M, K/2], a_sf [M, K/16] row-major; w_codes [N, K/2], w_sf [N, K/16]
    row-major.  Returns float32 [M, N]."""
    A = nvfp4.dequantize(a_codes, a_sf)
    W = nvfp4.dequantize(w_codes, w_sf)
    return (A @ W.T).astype(np.float32)


def apply_alpha_bf16(acc, alpha):
    """bf16(fp32(alpha * acc)); alpha broadcasts over columns."""
    with np.errstate(over="ignore"):
        return nvfp4.bf16_round(np.asarray(acc, np.float32) * np.asarray(alpha, np.float32))


def silu_mul(g, u):
    """h = bf16(silu(g) * u), silu(g) = g / (1 + exp(-g)) in fp32."""
    g = np.asarray(g, np.float32)
    u = np.asarray(u, np.float32)
    with np.errstate(over="ignore"):
        e = np.exp(-g.astype(np.float64)).astype(np.float32)
        s = g / (F32(1.0) + e)
        return nvfp4.bf16_round(s * u)


def gemm_l1(a_codes, a_sf, gs_a, rt, w1_codes, w1_sf, gs_w1_gate, gs_w1_up, rows=None):
    """L1 grouped GEMM over slots.

    a_codes [S, K/2], a_sf [S, K/16]: slot rows (row-major scales).
    rt: routing dict from :func:`oracle.route.route`.
    w1_codes [E, 2I, K/2], w1_sf [E, 2I, K/16]: rows 0..I-1 gate, I..2I-1 up.
    rows: optional boolean mask over slots; only those rows are computed.
    Returns (g, u): float32 [S, I] on the BF16 grid; rows not computed are 0."""
    E, N2, _ = w1_codes.shape
    I = N2 // 2
    S = a_codes.shape[0]
    g = np.zeros((S, I), np.float32)
    u = np.zeros((S, I), np.float32)
    for e in range(E):
        lo = int(rt["padded_offsets"][e])
        n = int(rt["counts"][e])
        sel = np.arange(lo, lo + n)
        if rows is not None:
            sel = sel[rows[sel]]
        if sel.size == 0:
            continue
        acc = expert_gemm(a_codes[sel], a_sf[sel], w1_codes[e], w1_sf[e])
        ag = F32(F32(gs_a) * F32(gs_w1_gate[e]))
        au = F32(F32(gs_a) * F32(gs_w1_up[e]))
        g[sel] = apply_alpha_bf16(acc[:, :I], ag)
        u[sel] = apply_alpha_bf16(acc[:, I:], au)
    return g, u


def gemm_l2(h_codes, h_sf, gs_h, rt, w2_codes, w2_sf, gs_w2, rows=None):
    """L2 grouped GEMM over slots: y = bf16(alpha * (H @ W2[e]^T)).

    h_codes [S, I/2], h_sf [S, I/16]; w2_codes [E, K, I/2], w2_sf [E, K, I/16].
    Returns float32 [S, K] on the BF16 grid; rows not computed are 0."""
    E, K, _ = w2_codes.shape
    S = h_codes.shape[0]
    y = np.zeros((S, K), np.float32)
    for e in range(E):
        lo = int(rt["padded_offsets"][e])
        n = int(rt["counts"][e])
        sel = np.arange(lo, lo + n)
        if rows is not None:
            sel = sel[rows[sel]]
        if sel.size == 0:
            continue
        acc = expert_gemm(h_codes[sel], h_sf[sel], w2_codes[e], w2_sf[e])
        y[sel] = apply_alpha_bf16(acc, F32(F32(gs_h) * F32(gs_w2[e])))
    return y


def combine(y, rt, T, topk, topk_w, tokens=None):
    """out[t] = bf16(sum_j fp32(w[t, j] * y[slot(t, j)])), j ascending, fp32.

    Pairs whose expert is not local contribute nothing."""
    K = y.shape[1]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    w = np.asarray(topk_w, np.float32).reshape(T, topk)
    ps = rt["pair_slot"].reshape(T, topk)
    out = np.zeros((len(tokens), K), np.float32)
    for i, t in enumerate(tokens):
        acc = np.zeros(K, np.float32)
        for j in range(topk):
            p = ps[t, j]
            if p >= 0:
                acc = acc + w[t, j] * y[p]
        out[i] = nvfp4.bf16_round(acc)
    return out


def forward(x, topk_ids, topk_w, E, expert_offset, weights, gs_x=None, gs_h=None,
            tokens=None):
    """The whole rank-local MoE layer.

    x: [T, K] float32 on the BF16 grid.  weights: dict with
      w1_codes [E, 2I, K/2], w1_sf [E, 2I, K/16] (row-major), gs_w1_gate [E],
      gs_w1_up [E], w2_codes [E, K, I/2], w2_sf [E, K, I/16], gs_w2 [E].
    gs_x / gs_h: None -> computed from the data (amax / 2688); else fixed.
    tokens: optional subset of token indices whose outputs are wanted; only
      their slots are computed (requires a fixed gs_h, since a data-derived
      gs_h needs every slot).
    Returns a dict with every intermediate (slot rows of padding are zero)."""
    x = np.asarray(x, np.float32)
    T, K = x.shape
    topk = topk_ids.shape[1]
    rt = route_pairs(topk_ids, topk_w, E, expert_offset)
    S = rt["slot_token"].shape[0]
    x_codes, x_sf, gs_x = nvfp4.quantize(x, gs_x)

    valid = rt["slot_token"] >= 0
    rows = valid.copy()
    if tokens is not None:
        if gs_h is None:
            raise ValueError("a token subset needs a fixed gs_h")
        want = np.zeros(T, bool)
        want[np.asarray(tokens)] = True
        rows &= want[np.maximum(rt["slot_token"], 0)]

    a_codes = np.zeros((S, K // 2), np.uint8)
    a_sf = np.zeros((S, K // 16), np.uint8)
    a_codes[valid] = x_codes[rt["slot_token"][valid]]
    a_sf[valid] = x_sf[rt["slot_token"][valid]]

    g, u = gemm_l1(a_codes, a_sf, gs_x, rt, weights["w1_codes"], weights["w1_sf"],
                   weights["gs_w1_gate"], weights["gs_w1_up"], rows=rows)
    h = silu_mul(g, u)
    h[~rows] = 0.0
    I = h.shape[1]
    h_codes = np.zeros((S, I // 2), np.uint8)
    h_sf = np.zeros((S, I // 16), np.uint8)
    hc, hs, gs_h = nvfp4.quantize(h[rows], gs_h)
    h_codes[rows] = hc
    h_sf[rows] = hs
    y = gemm_l2(h_codes, h_sf, gs_h, rt, weights["w2_codes"], weights["w2_sf"],
                weights["gs_w2"], rows=rows)
    out = combine(y, rt, T, topk, topk_w, tokens=tokens)
    return {
        "route": rt, "gs_x": gs_x, "x_codes": x_codes, "x_sf": x_sf,
        "a_codes": a_codes, "a_sf": a_sf, "g": g, "u": u, "h": h,
        "gs_h": gs_h, "h_codes": h_codes, "h_sf": h_sf, "y": y, "out": out,
        "rows": rows,
    }


def forward_bf16(x, topk_ids, topk_w, E, expert_offset, expert_w1, expert_w2, tokens=None):
    """The same layer without NVFP4 quantisation: the BF16 reference the pages
    compare the NVFP4 layer against (cosine similarity of the outputs).

    g = bf16(x @ W1_gate^T), u = bf16(x @ W1_up^T), h = bf16(silu(g) * u),
    y = bf16(h @ W2^T), out[t] = bf16(sum_j w[t, j] * y_j) in pair order, with the
    contractions in fp64 (rounded to fp32) and the BF16 rounding points of the
    quantised layer.  expert_w1(e) -> [2I, K], expert_w2(e) -> [K, I] (BF16 values
    as fp32); only the experts the chosen tokens route to are requested.
    Returns out [len(tokens), K] float32."""
    x = np.asarray(x, np.float32)
    T, K = x.shape
    topk = topk_ids.shape[1]
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    w = np.asarray(topk_w, np.float32).reshape(T, topk)
    loc = np.asarray(topk_ids, np.int64).reshape(T, topk) - expert_offset
    cache = {}
    out = np.zeros((len(tokens), K), np.float32)
    for i, t in enumerate(tokens):
        acc = np.zeros(K, np.float32)
        for j in range(topk):
            e = int(loc[t, j])
            if not 0 <= e < E:
                continue
            if e not in cache:
                cache[e] = (np.asarray(expert_w1(e), np.float64), np.asarray(expert_w2(e), np.float64))
            w1, w2 = cache[e]
            I = w1.shape[0] // 2
            gu = (w1 @ x[t].astype(np.float64)).astype(np.float32)
            g, u = nvfp4.bf16_round(gu[:I]), nvfp4.bf16_round(gu[I:])
            h = silu_mul(g, u)
            y = nvfp4.bf16_round((w2 @ h.astype(np.float64)).astype(np.float32))
            acc = acc + w[t, j] * y
        out[i] = nvfp4.bf16_round(acc)
    return out


def fold_gate_up_scales(w1_sf, gs_gate, gs_up):
    """The pages' gate/up handling (commits of vllm/nvfp4_cutedsl.py, "dual global scale"):
    both halves of W1 are normalised to the larger of the two global scales, and the
    ratio of the smaller one to it is folded into that half's block scales -- one fp32
    multiply of each decoded scale by the ratio, rounded back to UE4M3 (nearest, ties to
    even, saturating).  The L1 GEMM then needs one alpha per expert (gs_x * common).

    w1_sf: [E, 2I, K/16] row-major UE4M3 bytes, gate rows then up rows; gs_gate, gs_up:
    [E] fp32.  Returns (folded scales, common global scale [E] = max(gs_gate, gs_up));
    an expert whose two scales are equal (or both zero) is unchanged."""
    w1_sf = np.asarray(w1_sf, np.uint8)
    E, N2, _ = w1_sf.shape
    I = N2 // 2
    gg = np.asarray(gs_gate, F32)
    gu = np.asarray(gs_up, F32)
    common = np.maximum(gg, gu).astype(F32)
    out = w1_sf.copy()
    for e in range(E):
        for rows, g in ((slice(0, I), gg[e]), (slice(I, N2), gu[e])):
            if g == common[e] or common[e] == 0:
                continue
            ratio = F32(g) / F32(common[e])                       # fp32, round to nearest even
            scaled = nvfp4.e4m3_decode(out[e, rows]).astype(F32) * ratio   # fp32 multiply
            out[e, rows] = nvfp4.e4m3_encode_satfinite(scaled)
    return out, common


def quantize_weights(w1, w2):
    """Quantise BF16 expert weights the way the layer consumes them.

    w1: [E, 2I, K] float32 (gate rows then up rows), w2: [E, K, I].
    Gate and up of each expert get their own global scale; each down
    projection gets one.  Scales are row-major [N, K/16] (the checkpoint
    layout (N, K_sf) of the tests-page "scale transpose" commit)."""
    E, N2, K = w1.shape
    I = N2 // 2
    w1c = np.empty((E, N2, K // 2), np.uint8)
    w1s = np.empty((E, N2, K // 16), np.uint8)
    gg = np.empty(E, np.float32)
    gu = np.empty(E, np.float32)
    w2c = np.empty((E, K, I // 2), np.uint8)
    w2s = np.empty((E, K, I // 16), np.uint8)
    g2 = np.empty(E, np.float32)
    for e in range(E):
        c, s, gg[e] = nvfp4.quantize(w1[e, :I])
        w1c[e, :I], w1s[e, :I] = c, s
        c, s, gu[e] = nvfp4.quantize(w1[e, I:])
        w1c[e, I:], w1s[e, I:] = c, s
        w2c[e], w2s[e], g2[e] = nvfp4.quantize(w2[e])
    return {"w1_codes": w1c, "w1_sf": w1s, "gs_w1_gate": gg, "gs_w1_up": gu,
            "w2_codes": w2c, "w2_sf": w2s, "gs_w2": g2}
