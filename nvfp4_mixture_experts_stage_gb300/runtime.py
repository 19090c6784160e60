"""Device-side set-up around the C ABI: expert weights resident in HBM, the
workspace, and one call of the whole layer.

Nothing here computes: weight quantisation and scale rearrangement run in the
library's kernels (moe_stage_activation, moe_prepare_weights), the layer runs
in moe_forward.  PyTorch only allocates device memory and supplies streams.
"""

from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B


@dataclass
class Layer:
    """One rank's expert weights in the layout the grouped GEMMs read."""
    K: int
    I: int
    E: int
    topk: int
    expert_offset: int
    w1_fp4: torch.Tensor      # [E, 2I, K/2] uint8
    w1_sf: torch.Tensor       # prepared (MOE_PREP_W1), E*2I*K/16 bytes
    gs_w1_gate: torch.Tensor  # [E] fp32
    gs_w1_up: torch.Tensor    # [E] fp32
    w2_fp4: torch.Tensor      # [E, K, I/2] uint8
    w2_sf: torch.Tensor       # prepared (MOE_PREP_W2)
    gs_w2: torch.Tensor       # [E] fp32
    w1_sf_rowmajor: torch.Tensor = None  # [E, 2I, K/16] (kept for checks)
    w2_sf_rowmajor: torch.Tensor = None  # [E, K, I/16]

    def weights_struct(self):
        return B.make_weights(self.w1_fp4, self.w1_sf, self.gs_w1_gate, self.gs_w1_up,
                              self.w2_fp4, self.w2_sf, self.gs_w2)

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in
                   (self.w1_fp4, self.w1_sf, self.w2_fp4, self.w2_sf))


def _prepare(layer, stream=None):
    E, I, K = layer.E, layer.I, layer.K
    dev = layer.w1_fp4.device
    layer.w1_sf = torch.empty(E * 2 * I * K // 16, dtype=torch.uint8, device=dev)
    layer.w2_sf = torch.empty(E * K * I // 16, dtype=torch.uint8, device=dev)
    B.moe_prepare_weights(layer.w1_sf_rowmajor, layer.w1_sf, E, 2 * I, K, B.MOE_PREP_W1, stream)
    B.moe_prepare_weights(layer.w2_sf_rowmajor, layer.w2_sf, E, K, I, B.MOE_PREP_W2, stream)
    return layer


def layer_from_nvfp4(w1_codes, w1_sf, gs_w1_gate, gs_w1_up, w2_codes, w2_sf, gs_w2, topk, expert_offset,
                     device="cuda"):
    """Upload already-quantised weights (row-major (N, K_sf) scales, as in a
    checkpoint) and rearrange their scales on the device."""
    t = lambda a, dt: torch.as_tensor(np.ascontiguousarray(a)).to(device=device, dtype=dt)
    E, N2, K2 = w1_codes.shape
    layer = Layer(K=K2 * 2, I=N2 // 2, E=E, topk=topk, expert_offset=expert_offset,
                  w1_fp4=t(w1_codes, torch.uint8), w1_sf=None,
                  gs_w1_gate=t(gs_w1_gate, torch.float32), gs_w1_up=t(gs_w1_up, torch.float32),
                  w2_fp4=t(w2_codes, torch.uint8), w2_sf=None, gs_w2=t(gs_w2, torch.float32),
                  w1_sf_rowmajor=t(w1_sf, torch.uint8), w2_sf_rowmajor=t(w2_sf, torch.uint8))
    return _prepare(layer)


def quantize_weights_on_device(wl, expert_w1, expert_w2, device="cuda", keep_rowmajor=False):
    """Quantise BF16 expert weights to NVFP4 with the library's own quantiser
    (gate and up of each expert with separate global scales, the down
    projection with one), then rearrange the scales.

    expert_w1(e) -> [2I, K] BF16 CPU tensor; expert_w2(e) -> [K, I]."""
    E, I, K = wl.E, wl.I, wl.K
    f = lambda *s, dt=torch.uint8: torch.empty(*s, dtype=dt, device=device)
    w1_fp4, w1_sfr = f(E, 2 * I, K // 2), f(E, 2 * I, K // 16)
    w2_fp4, w2_sfr = f(E, K, I // 2), f(E, K, I // 16)
    gs = f(3, E, dt=torch.float32)
    ws = f(B.moe_stage_workspace_size())
    for e in range(E):
        w1 = expert_w1(e).to(device)
        w2 = expert_w2(e).to(device)
        B.moe_stage_activation(w1[:I], w1_fp4[e, :I], w1_sfr[e, :I], B.MOE_SF_ROWMAJOR, gs[0, e:e + 1], ws=ws)
        B.moe_stage_activation(w1[I:], w1_fp4[e, I:], w1_sfr[e, I:], B.MOE_SF_ROWMAJOR, gs[1, e:e + 1], ws=ws)
        B.moe_stage_activation(w2, w2_fp4[e], w2_sfr[e], B.MOE_SF_ROWMAJOR, gs[2, e:e + 1], ws=ws)
    layer = Layer(K=K, I=I, E=E, topk=wl.topk, expert_offset=wl.expert_offset,
                  w1_fp4=w1_fp4, w1_sf=None, gs_w1_gate=gs[0].clone(), gs_w1_up=gs[1].clone(),
                  w2_fp4=w2_fp4, w2_sf=None, gs_w2=gs[2].clone(),
                  w1_sf_rowmajor=w1_sfr, w2_sf_rowmajor=w2_sfr)
    _prepare(layer)
    if not keep_rowmajor:
        torch.cuda.current_stream().synchronize()
        layer.w1_sf_rowmajor = layer.w2_sf_rowmajor = None
    return layer


class Forward:
    """Pre-allocated buffers for repeated calls of the layer at a fixed T (so the
    call can be captured into a CUDA graph)."""

    def __init__(self, layer: Layer, T, gs_h_mode=B.MOE_GS_DYNAMIC, device="cuda"):
        self.layer = layer
        self.T = T
        self.gs_h_mode = gs_h_mode
        self.ws = torch.empty(B.moe_workspace_size(T, layer.K, layer.I, layer.E, layer.topk),
                              dtype=torch.uint8, device=device)
        self.out = torch.empty(T, layer.K, dtype=torch.bfloat16, device=device)
        self.gs_h = torch.zeros(1, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.wstruct = layer.weights_struct()

    def __call__(self, x, topk_ids, topk_w, gs_x_fixed=None, stream=None, events=None, out=None):
        """The layer on x; writes `out` ([T, K] BF16 on the device) if given, else the
        object's own output buffer, and returns it."""
        L = self.layer
        o = self.out if out is None else out
        if events is None:
            B.moe_forward(x, topk_ids, topk_w, L.E, L.I, L.expert_offset, self.wstruct, self.gs_h_mode,
                          self.gs_h, o, self.ws, gs_x_fixed=gs_x_fixed, dev_status=self.status,
                          stream=stream)
        else:
            B.moe_forward_traced(x, topk_ids, topk_w, L.E, L.I, L.expert_offset, self.wstruct, self.gs_h_mode,
                                 self.gs_h, o, self.ws, events, gs_x_fixed=gs_x_fixed,
                                 dev_status=self.status, stream=stream)
        return o


def run_forward(layer, x, topk_ids, topk_w, gs_h_mode=B.MOE_GS_DYNAMIC, gs_h=None, gs_x_fixed=None):
    """One call of the layer; returns (out [T, K] BF16, gs_h)."""
    fw = Forward(layer, x.shape[0], gs_h_mode, device=x.device)
    if gs_h is not None:
        fw.gs_h.fill_(float(gs_h))
    out = fw(x, topk_ids, topk_w, gs_x_fixed=gs_x_fixed)
    return out, fw.gs_h
