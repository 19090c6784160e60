"""Seeded synthetic inputs for the NVFP4 MoE stage.

This module only *draws* inputs; it holds none of the layer's arithmetic (no
quantisation, no routing, no GEMM).  Both the CUDA library's tests/benchmark
and the CPU oracle take their inputs from here, so the two sides see the same
bytes.  BF16 rounding of the drawn fp32 values is done by torch's CPU cast.

Streams: numpy ``Generator(PCG64)``; ``SeedSequence(seed).spawn(n)`` gives one
child stream per tensor, so any single expert's weights can be regenerated
without drawing the others.

Workloads (sizes from the MoE layer they stand in for: DeepSeek-V4-Pro style
routed experts, 384 global experts, 48 per rank, hidden 4096, intermediate
3072, top-8; no dataset or checkpoint is used):

========== ===== ===== ===== ==== ==== ====== ===============================
name           T     K     I    E topk offset routing
========== ===== ===== ===== ==== ==== ====== ===============================
tiny          16   256   128    8    2      0 softmax of N(0,1) logits, top-2
decode       256  4096  3072   48    8    144 8 distinct of 384 global ids
prefill     8192  4096  3072   48    8      0 8 distinct of the 48 local ids
skew_top1   4096  4096  3072   48    1      0 Zipf(1.2) quota over 40 experts
skew_top8   4096  4096  3072   48    8      0 Gumbel-top-8 on Zipf(1.2) p
sweep_*    1k/16k/64k 7168  -  48    8      0 8 distinct of 48 (stage+route)
========== ===== ===== ===== ==== ==== ====== ===============================
"""

from dataclasses import dataclass, field

import numpy as np
import torch

N_STREAMS_FIXED = 8  # x, routing, outliers, row scales, ... ; weights follow


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    K: int
    I: int
    E: int
    topk: int
    expert_offset: int = 0
    n_global: int = 0            # >0: ids drawn from 0..n_global-1 (global)
    routing: str = "uniform"     # uniform | softmax_topk | zipf_top1 | zipf_topk
    x_kind: str = "normal"       # normal | outliers | big_rows
    seed: int = 0
    extra: dict = field(default_factory=dict, compare=False, hash=False)


WORKLOADS = {
    "tiny": Workload("tiny", 16, 256, 128, 8, 2, routing="softmax_topk", x_kind="outliers"),
    "decode": Workload("decode", 256, 4096, 3072, 48, 8, expert_offset=144, n_global=384),
    "prefill": Workload("prefill", 8192, 4096, 3072, 48, 8, x_kind="big_rows"),
    "skew_top1": Workload("skew_top1", 4096, 4096, 3072, 48, 1, routing="zipf_top1"),
    "skew_top8": Workload("skew_top8", 4096, 4096, 3072, 48, 8, routing="zipf_topk"),
    "sweep_1k": Workload("sweep_1k", 1024, 7168, 0, 48, 8),
    "sweep_16k": Workload("sweep_16k", 16384, 7168, 0, 48, 8),
    "sweep_64k": Workload("sweep_64k", 65536, 7168, 0, 48, 8),
}


def small(name, T, K, I, E, topk, expert_offset=0, n_global=0, routing="uniform",
          x_kind="normal", seed=0):
    """An ad-hoc workload with the same recipe at a test-chosen size."""
    return Workload(name, T, K, I, E, topk, expert_offset, n_global, routing, x_kind, seed)


def _streams(wl: Workload):
    n = N_STREAMS_FIXED + 2 * max(wl.E, 1)
    return np.random.SeedSequence(wl.seed).spawn(n)


def _rng(wl, i):
    return np.random.Generator(np.random.PCG64(_streams(wl)[i]))


def to_bf16(a):
    """fp32 numpy array -> torch.bfloat16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------

def activations(wl: Workload):
    """x [T, K] as a torch.bfloat16 CPU tensor."""
    x = _rng(wl, 0).standard_normal((wl.T, wl.K), dtype=np.float32)
    if wl.x_kind == "outliers":
        # 1% of elements (iid Bernoulli(0.01)) scaled by 20
        mask = _rng(wl, 2).random((wl.T, wl.K)) < 0.01
        x = np.where(mask, x * np.float32(20.0), x)
    elif wl.x_kind == "big_rows":
        # 16 rows rescaled to a row amax of 10**U(1, 4); the first of them
        # gets its largest element set to exactly 9984 (= bf16(1e4)).
        r = _rng(wl, 3)
        rows = r.choice(wl.T, size=min(16, wl.T), replace=False)
        targets = 10.0 ** r.uniform(1.0, 4.0, size=rows.size)
        for i, (row, tgt) in enumerate(zip(rows, targets)):
            v = x[row].astype(np.float64)
            v = v * (tgt / np.abs(v).max())
            if i == 0:
                j = int(np.abs(v).argmax())
                v[j] = 9984.0 if v[j] > 0 else -9984.0
            x[row] = v.astype(np.float32)
    return to_bf16(x)


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------

def _softmax_rows(logits):
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


def _distinct_uniform(r, T, k, n):
    """k distinct ids per row, uniform over 0..n-1 (argsort of iid uniforms)."""
    return np.argsort(r.random((T, n)), axis=1)[:, :k]


def zipf_probs(n_ranks=40, alpha=1.2, n_experts=48):
    p = np.zeros(n_experts)
    ranks = np.arange(1, n_ranks + 1, dtype=np.float64)
    p[:n_ranks] = ranks ** -alpha
    return p / p.sum()


def quota_counts(p, T):
    """Largest-remainder apportionment of T tokens to probabilities p."""
    q = p * T
    c = np.floor(q).astype(np.int64)
    rem = T - c.sum()
    order = np.argsort(-(q - c), kind="stable")
    c[order[:rem]] += 1
    return c


def routing(wl: Workload):
    """(topk_ids [T, topk] int32 global ids, topk_w [T, topk] float32)."""
    r = _rng(wl, 1)
    T, k, E = wl.T, wl.topk, wl.E
    if wl.routing == "softmax_topk":
        logits = r.standard_normal((T, E)).astype(np.float32).astype(np.float64)
        p = _softmax_rows(logits)
        ids = np.argsort(-p, axis=1, kind="stable")[:, :k]  # ties -> lower id
        w = np.take_along_axis(p, ids, axis=1)
        w = w / w.sum(axis=1, keepdims=True)
        return (ids + wl.expert_offset).astype(np.int32), w.astype(np.float32)
    if wl.routing == "uniform":
        n = wl.n_global if wl.n_global else E
        ids = _distinct_uniform(r, T, k, n)
        if not wl.n_global:
            ids = ids + wl.expert_offset
        w = _softmax_rows(r.standard_normal((T, k)))
        return ids.astype(np.int32), w.astype(np.float32)
    p = zipf_probs(40, 1.2, E)
    perm = r.permutation(E)            # rank i -> expert perm[i]
    p_exp = np.zeros(E)
    p_exp[perm] = p
    if wl.routing == "zipf_top1":
        counts = quota_counts(p, T)    # per rank
        ids = np.repeat(perm, counts)  # tokens ordered by rank...
        ids = np.sort(ids)             # ...then by expert id
        w = np.ones((T, 1), np.float32)
        return (ids[:, None] + wl.expert_offset).astype(np.int32), w
    if wl.routing == "zipf_topk":
        with np.errstate(divide="ignore"):
            logp = np.log(p_exp)
        gumbel = -np.log(-np.log(r.random((T, E))))
        ids = np.argsort(-(logp[None, :] + gumbel), axis=1, kind="stable")[:, :k]
        w = _softmax_rows(r.standard_normal((T, k)))
        return (ids + wl.expert_offset).astype(np.int32), w.astype(np.float32)
    raise ValueError(wl.routing)


def shuffled_twin(ids, w, seed=1):
    """Same routing with the token order permuted (the unsorted twin of the
    top-1 skew case)."""
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(ids.shape[0])
    return ids[perm], w[perm]


# --------------------------------------------------------------------------
# expert weights
# --------------------------------------------------------------------------

def expert_w1(wl: Workload, e):
    """W1 of expert e: [2I, K] BF16 (rows 0..I-1 gate, I..2I-1 up), N(0, 0.02)."""
    a = _rng(wl, N_STREAMS_FIXED + 2 * e).standard_normal((2 * wl.I, wl.K), dtype=np.float32)
    return to_bf16(a * np.float32(0.02))


def expert_w2(wl: Workload, e):
    """W2 (down) of expert e: [K, I] BF16, N(0, 0.02)."""
    a = _rng(wl, N_STREAMS_FIXED + 2 * e + 1).standard_normal((wl.K, wl.I), dtype=np.float32)
    return to_bf16(a * np.float32(0.02))


def fixed_gs_h(wl: Workload):
    """A fixed (calibrated-mode) global scale for the requantised activation,
    used where a test needs the h scale without computing every slot: the
    amax of h = silu(g) * u expected at five standard deviations of g and u
    (std of g ~ 0.02 * sqrt(K) for N(0,1) activations), divided by 2688."""
    s = 5.0 * 0.02 * np.sqrt(wl.K)
    return np.float32(max(s * s, 1.0) / 2688.0)
