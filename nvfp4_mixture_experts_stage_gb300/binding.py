"""Thin ctypes binding of libmoe_stage.so (include/moe_stage.h).

Argument marshalling only: every function takes torch tensors (device memory,
or pinned host memory where noted by the caller), passes their data pointers
and the current CUDA stream to the C entry point of the same name, and raises
:class:`MoeError` on a non-zero status.  Every step of the layer runs in the
library's CUDA kernels; there is no Python or CPU fallback.  If the shared
library is missing the import of this module fails.
"""

import ctypes
import os

import torch

from .build import LIB

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_INDEX = 6

MOE_TILE_M = 128
MOE_SF_ROWMAJOR, MOE_SF_SWIZZLED = 0, 1
MOE_PREP_W1, MOE_PREP_W2 = 0, 1
MOE_L1_GATEUP_BF16, MOE_L1_SILU_BF16, MOE_L1_SILU_REQUANT = 0, 1, 2
MOE_L2_ROWS_BF16, MOE_L2_SCATTER = 0, 1
MOE_GS_DYNAMIC, MOE_GS_FIXED = 0, 1

#: Every symbol include/moe_stage.h declares.
EXPORTS = (
    "moe_status_string", "moe_slot_capacity", "moe_route_workspace_size",
    "moe_stage_workspace_size", "moe_workspace_size", "moe_prepare_weights",
    "moe_stage_activation", "moe_stage_activation_to_slots", "moe_route",
    "moe_grouped_gemm_l1", "moe_requant", "moe_grouped_gemm_l2",
    "moe_cast_output", "moe_forward", "moe_forward_traced", "moe_route_static_scratch",
    "moe_set_gemm_policy", "moe_combine_rows", "moe_selftest_bounded_wait", "moe_fold_gate_up_scales",
    "moe_quantize_weights_workspace_size", "moe_quantize_weights", "moe_selftest_codecs",
    "moe_selftest_silu",
)

MOE_GEMM_AUTO, MOE_GEMM_TILED, MOE_GEMM_STREAMING = 0, 1, 2
MOE_GEMM_STREAMING_N32, MOE_GEMM_STREAMING_N64, MOE_GEMM_TILED_1CTA, MOE_GEMM_TILED_PAIR = 3, 4, 5, 6

MOE_ROUTE_STATIC_TABLE_INTS = 262144

MOE_TRACE_EVENTS = 7


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {_lib.moe_status_string(status).decode()} (status {status})")


class MoeWeights(ctypes.Structure):
    _fields_ = [("w1_fp4", ctypes.c_void_p), ("w1_sf", ctypes.c_void_p),
                ("gs_w1_gate", ctypes.c_void_p), ("gs_w1_up", ctypes.c_void_p),
                ("w2_fp4", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p),
                ("gs_w2", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB):
        raise ImportError(f"{LIB} is not built; run nvfp4_mixture_experts_stage_gb300.build.build()")
    lib = ctypes.CDLL(LIB)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "moe_status_string": (ctypes.c_char_p, [I32]),
        "moe_slot_capacity": (I64, [I64, I32, I32]),
        "moe_route_workspace_size": (SZ, [I64, I32, I32]),
        "moe_stage_workspace_size": (SZ, []),
        "moe_workspace_size": (SZ, [I64, I32, I32, I32, I32]),
        "moe_prepare_weights": (I32, [P, P, I32, I32, I32, I32, P]),
        "moe_stage_activation": (I32, [P, I64, I32, I64, P, P, I32, P, P, P, SZ, P, P]),
        "moe_stage_activation_to_slots": (I32, [P, I64, I32, I64, P, I32, I64, P, P, P, P, P, SZ, P, P]),
        "moe_route": (I32, [P, P, I64, I32, I32, I32, P, P, P, P, P, P, I64, P, SZ, P]),
        "moe_route_static_scratch": (I32, [P, P, I64, I32, I32, I32, P, P, P, P, P, P, I64, P]),
        "moe_grouped_gemm_l1": (I32, [P, P, P, P, P, I32, I64, I32, I32, P, P, P, P, I32, P, P, P, P, P, P, P]),
        "moe_requant": (I32, [P, I64, I32, P, P, P, P, P, P, P]),
        "moe_grouped_gemm_l2": (I32, [P, P, P, P, P, I32, I64, I32, I32, P, P, P, I32, P, P, P, P, I64, P, P]),
        "moe_cast_output": (I32, [P, P, I64, I32, P]),
        "moe_combine_rows": (I32, [P, I64, P, P, I64, I32, I32, I64, P, P, P]),
        "moe_selftest_bounded_wait": (I32, [P, P, P]),
        "moe_selftest_codecs": (I32, [ctypes.c_uint32, I64, P, P, P]),
        "moe_selftest_silu": (I32, [P, I64, P, P]),
        "moe_fold_gate_up_scales": (I32, [P, P, P, P, I32, I32, I32, P]),
        "moe_quantize_weights_workspace_size": (ctypes.c_size_t, [I32, I32, I32]),
        "moe_quantize_weights": (I32, [P, P, I32, I32, I32, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]),
        "moe_set_gemm_policy": (I32, [I32]),
        "moe_forward": (I32, [P, I64, I32, I32, I32, P, P, I32, I32, ctypes.POINTER(MoeWeights), P, I32, P, P,
                              P, P, SZ, P]),
        "moe_forward_traced": (I32, [P, I64, I32, I32, I32, P, P, I32, I32, ctypes.POINTER(MoeWeights), P, I32,
                                     P, P, P, P, SZ, ctypes.POINTER(ctypes.c_void_p), P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def library():
    """The loaded ctypes.CDLL (for symbol checks)."""
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)


# ----------------------------------------------------------------- queries

def moe_slot_capacity(T, topk, E):
    return _lib.moe_slot_capacity(T, topk, E)


def moe_route_workspace_size(T, topk, E):
    return _lib.moe_route_workspace_size(T, topk, E)


def moe_stage_workspace_size():
    return _lib.moe_stage_workspace_size()


def moe_workspace_size(T_max, K, I, E, topk):
    return _lib.moe_workspace_size(T_max, K, I, E, topk)


def moe_set_gemm_policy(policy):
    """Select the grouped-GEMM kernels (MOE_GEMM_AUTO / _TILED / _TILED_1CTA /
    _TILED_PAIR / _STREAMING / _STREAMING_N32 / _STREAMING_N64); returns the
    previous policy."""
    r = _lib.moe_set_gemm_policy(policy)
    if r < 0:
        raise MoeError("moe_set_gemm_policy", MOE_ERR_INVALID_ARG)
    return r


def moe_status_string(s):
    return _lib.moe_status_string(s).decode()


# ----------------------------------------------------------------- calls

def moe_prepare_weights(sf_rowmajor, sf_prepared, E, N, K, kind, stream=None):
    _check("moe_prepare_weights", _lib.moe_prepare_weights(
        _p(sf_rowmajor), _p(sf_prepared), E, N, K, kind, _stream(stream)))


def moe_stage_activation(x, x_fp4, x_sf, sf_layout, gs_out, gs_fixed=None, ws=None, dev_status=None,
                         stream=None):
    T, K = x.shape
    _check("moe_stage_activation", _lib.moe_stage_activation(
        _p(x), T, K, x.stride(0), _p(x_fp4), _p(x_sf), sf_layout, _p(gs_out), _p(gs_fixed),
        _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(dev_status), _stream(stream)))


def moe_stage_activation_to_slots(x, pair_slot, topk, capacity, a_fp4, a_sf, gs_out, gs_fixed=None, ws=None,
                                  dev_status=None, stream=None):
    T, K = x.shape
    _check("moe_stage_activation_to_slots", _lib.moe_stage_activation_to_slots(
        _p(x), T, K, x.stride(0), _p(pair_slot), topk, capacity, _p(a_fp4), _p(a_sf), _p(gs_out),
        _p(gs_fixed), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _p(dev_status),
        _stream(stream)))


def moe_route(topk_ids, topk_w, E, expert_offset, counts, offsets, padded_offsets, slot_token, slot_weight,
              pair_slot, ws, stream=None):
    T, topk = topk_ids.shape
    _check("moe_route", _lib.moe_route(
        _p(topk_ids), _p(topk_w), T, topk, E, expert_offset, _p(counts), _p(offsets), _p(padded_offsets),
        _p(slot_token), _p(slot_weight), _p(pair_slot), slot_token.numel(), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_static_scratch(topk_ids, topk_w, E, expert_offset, counts, offsets, padded_offsets, slot_token,
                             slot_weight, pair_slot, stream=None):
    """moe_route without a workspace (its scratch is a fixed device array inside
    the library; see include/moe_stage.h for the size limit and the rules)."""
    T, topk = topk_ids.shape
    _check("moe_route_static_scratch", _lib.moe_route_static_scratch(
        _p(topk_ids), _p(topk_w), T, topk, E, expert_offset, _p(counts), _p(offsets), _p(padded_offsets),
        _p(slot_token), _p(slot_weight), _p(pair_slot), slot_token.numel(), _stream(stream)))


def moe_grouped_gemm_l1(a_fp4, a_sf, gs_a, offsets, padded_offsets, E, K, I, w1_fp4, w1_sf, gs_w1_gate,
                        gs_w1_up, epilogue, out_bf16=None, h_amax=None, h_fp4=None, h_sf=None, gs_h=None,
                        dev_status=None, stream=None):
    capacity = a_fp4.shape[0]
    _check("moe_grouped_gemm_l1", _lib.moe_grouped_gemm_l1(
        _p(a_fp4), _p(a_sf), _p(gs_a), _p(offsets), _p(padded_offsets), E, capacity, K, I, _p(w1_fp4),
        _p(w1_sf), _p(gs_w1_gate), _p(gs_w1_up), epilogue, _p(out_bf16), _p(h_amax), _p(h_fp4), _p(h_sf),
        _p(gs_h), _p(dev_status), _stream(stream)))


def moe_requant(h, slot_token, h_amax, gs_h_out, h_fp4, h_sf, dev_status=None, stream=None):
    capacity, I = h.shape
    _check("moe_requant", _lib.moe_requant(
        _p(h), capacity, I, _p(slot_token), _p(h_amax), _p(gs_h_out), _p(h_fp4), _p(h_sf), _p(dev_status),
        _stream(stream)))


def moe_grouped_gemm_l2(h_fp4, h_sf, gs_h, offsets, padded_offsets, E, I, K, w2_fp4, w2_sf, gs_w2, epilogue,
                        y_rows=None, slot_token=None, slot_weight=None, out32=None, T=0, dev_status=None,
                        stream=None):
    capacity = h_fp4.shape[0]
    _check("moe_grouped_gemm_l2", _lib.moe_grouped_gemm_l2(
        _p(h_fp4), _p(h_sf), _p(gs_h), _p(offsets), _p(padded_offsets), E, capacity, I, K, _p(w2_fp4),
        _p(w2_sf), _p(gs_w2), epilogue, _p(y_rows), _p(slot_token), _p(slot_weight), _p(out32), T,
        _p(dev_status), _stream(stream)))


def moe_cast_output(out32, out_bf16, stream=None):
    T, K = out32.shape
    _check("moe_cast_output", _lib.moe_cast_output(_p(out32), _p(out_bf16), T, K, _stream(stream)))


def moe_quantize_weights_workspace_size(E, I, K):
    return int(_lib.moe_quantize_weights_workspace_size(E, I, K))


def moe_quantize_weights(w1, w2, w1_fp4, w1_sf, gs_w1_gate, gs_w1_up, w2_fp4, w2_sf, gs_w2, ws, stream=None):
    """BF16 expert weights w1 [E, 2I, K], w2 [E, K, I] -> NVFP4 codes, prepared scales and
    global scales (see include/moe_stage.h)."""
    E, N2, K = w1.shape
    _check("moe_quantize_weights", _lib.moe_quantize_weights(
        _p(w1), _p(w2), E, N2 // 2, K, _p(w1_fp4), _p(w1_sf), _p(gs_w1_gate), _p(gs_w1_up), _p(w2_fp4),
        _p(w2_sf), _p(gs_w2), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_fold_gate_up_scales(w1_sf, gs_gate, gs_up, gs_common, stream=None):
    """Fold W1's two global scales into one (see include/moe_stage.h): w1_sf [E, 2I, K/16]
    uint8 row-major, folded in place; gs_common [E] written."""
    E, N2, k_sf = w1_sf.shape
    _check("moe_fold_gate_up_scales", _lib.moe_fold_gate_up_scales(
        _p(w1_sf), _p(gs_gate), _p(gs_up), _p(gs_common), E, N2 // 2, k_sf * 16, _stream(stream)))


def moe_selftest_bounded_wait(dev_status, dev_result, stream=None):
    """Failure-reporting self-test (see include/moe_stage.h): about one second of device
    time; afterwards dev_status holds MOE_ERR_TIMEOUT and dev_result (2 int32) [1, 1]."""
    _check("moe_selftest_bounded_wait", _lib.moe_selftest_bounded_wait(_p(dev_status), _p(dev_result),
                                                                       _stream(stream)))


def moe_selftest_codecs(first_pattern, e2m1_codes, e4m3_bytes, stream=None):
    """Encoder self-test (see include/moe_stage.h): for the fp32 bit patterns
    first_pattern .. first_pattern + n - 1 (n = e2m1_codes.numel()), the device's E2M1
    code and UE4M3 byte of each value, written to the two uint8 device tensors."""
    n = e2m1_codes.numel()
    assert e4m3_bytes.numel() == n
    _check("moe_selftest_codecs", _lib.moe_selftest_codecs(first_pattern, n, _p(e2m1_codes), _p(e4m3_bytes),
                                                           _stream(stream)))


def moe_selftest_silu(g, silu_out, stream=None):
    """SiLU self-test (see include/moe_stage.h): silu_out[i] = the L1 epilogue's fp32
    SiLU of g[i] (both fp32 device tensors of the same size)."""
    n = g.numel()
    assert silu_out.numel() == n and g.dtype == torch.float32 and silu_out.dtype == torch.float32
    _check("moe_selftest_silu", _lib.moe_selftest_silu(_p(g), n, _p(silu_out), _stream(stream)))


def moe_combine_rows(y_rows, pair_slot, topk_w, out_bf16, capacity=None, dev_status=None, stream=None):
    """out_bf16[t] = bf16(sum_j w[t, j] * y_rows[pair_slot[t, j]]) (include/moe_stage.h)."""
    T, topk = topk_w.shape
    K = out_bf16.shape[1]
    cap = y_rows.shape[0] if capacity is None else capacity
    _check("moe_combine_rows", _lib.moe_combine_rows(
        _p(y_rows), y_rows.stride(0), _p(pair_slot), _p(topk_w), T, topk, K, cap, _p(out_bf16), _p(dev_status),
        _stream(stream)))


def make_weights(w1_fp4, w1_sf, gs_w1_gate, gs_w1_up, w2_fp4, w2_sf, gs_w2):
    """A moe_weights struct pointing at device tensors (the caller keeps them alive)."""
    return MoeWeights(*(t.data_ptr() for t in (w1_fp4, w1_sf, gs_w1_gate, gs_w1_up, w2_fp4, w2_sf, gs_w2)))


def moe_forward(x, topk_ids, topk_w, E, I, expert_offset, weights, gs_h_mode, gs_h, out, ws, gs_x_fixed=None,
                dev_status=None, stream=None):
    T, K = x.shape
    topk = topk_ids.shape[1]
    _check("moe_forward", _lib.moe_forward(
        _p(x), T, K, I, E, _p(topk_ids), _p(topk_w), topk, expert_offset, ctypes.byref(weights),
        _p(gs_x_fixed), gs_h_mode, _p(gs_h), _p(out), _p(dev_status), _p(ws), ws.numel() * ws.element_size(),
        _stream(stream)))


def moe_forward_traced(x, topk_ids, topk_w, E, I, expert_offset, weights, gs_h_mode, gs_h, out, ws, events,
                       gs_x_fixed=None, dev_status=None, stream=None):
    """moe_forward that records MOE_TRACE_EVENTS torch.cuda.Event objects (timing
    enabled, already created by one record()) at the stage boundaries; None
    entries are skipped."""
    T, K = x.shape
    topk = topk_ids.shape[1]
    arr = (ctypes.c_void_p * MOE_TRACE_EVENTS)(*[None if ev is None else ev.cuda_event for ev in events])
    _check("moe_forward_traced", _lib.moe_forward_traced(
        _p(x), T, K, I, E, _p(topk_ids), _p(topk_w), topk, expert_offset, ctypes.byref(weights),
        _p(gs_x_fixed), gs_h_mode, _p(gs_h), _p(out), _p(dev_status), _p(ws), ws.numel() * ws.element_size(),
        arr, _stream(stream)))
