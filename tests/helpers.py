"""Shared test helpers: seeded inputs, oracle-quantised weights, device upload
and comparisons.  Expected values always come from the oracle on the CPU."""

import numpy as np
import torch

import workloads
from oracle import moe as omoe, nvfp4 as q


def oracle_weights(wl):
    """Expert weights of a workload quantised by the oracle (row-major scales)."""
    w1 = np.stack([workloads.expert_w1(wl, e).float().numpy() for e in range(wl.E)])
    w2 = np.stack([workloads.expert_w2(wl, e).float().numpy() for e in range(wl.E)])
    return omoe.quantize_weights(w1, w2)


def oracle_weights_streamed(wl, experts=None):
    """Same, one expert at a time (for the full-size workloads)."""
    E, I, K = wl.E, wl.I, wl.K
    W = {"w1_codes": np.zeros((E, 2 * I, K // 2), np.uint8), "w1_sf": np.zeros((E, 2 * I, K // 16), np.uint8),
         "gs_w1_gate": np.zeros(E, np.float32), "gs_w1_up": np.zeros(E, np.float32),
         "w2_codes": np.zeros((E, K, I // 2), np.uint8), "w2_sf": np.zeros((E, K, I // 16), np.uint8),
         "gs_w2": np.zeros(E, np.float32)}
    for e in (range(E) if experts is None else experts):
        w1 = workloads.expert_w1(wl, e).float().numpy()
        w2 = workloads.expert_w2(wl, e).float().numpy()
        W["w1_codes"][e, :I], W["w1_sf"][e, :I], W["gs_w1_gate"][e] = q.quantize(w1[:I])
        W["w1_codes"][e, I:], W["w1_sf"][e, I:], W["gs_w1_up"][e] = q.quantize(w1[I:])
        W["w2_codes"][e], W["w2_sf"][e], W["gs_w2"][e] = q.quantize(w2)
    return W


def dev(a, dtype=None, device="cuda"):
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def bf16_dev(x_f32, device="cuda"):
    """fp32 values already on the BF16 grid -> BF16 device tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(x_f32, np.float32)).to(torch.bfloat16).to(device)


def cosine(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


def assert_layer_close(got, ref, what=""):
    """The layer tolerance: |gpu - oracle| <= 1e-2 * max|oracle| per element and
    cosine >= 0.9999, on identical quantised inputs."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    cos = cosine(got, ref) if scale > 0 else 1.0
    assert err <= 1e-2 * scale, f"{what}: max|err| {err:.4g} > 1e-2 * {scale:.4g}"
    assert cos >= 0.9999, f"{what}: cosine {cos:.6f}"
    return err, cos
