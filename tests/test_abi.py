"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host-side logic (size queries, argument checks) behaves."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_stage.h")


@pytest.fixture(scope="module")
def B():
    from nvfp4_mixture_experts_stage_gb300 import build
    build.build()
    from nvfp4_mixture_experts_stage_gb300 import binding
    return binding


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_all_exported(B):
    names = _declared()
    assert set(names) == set(B.EXPORTS)
    for n in names:
        assert hasattr(B.library(), n), n


def test_status_strings(B):
    for s in range(7):
        assert B.moe_status_string(s)
    assert "workspace" in B.moe_status_string(B.MOE_ERR_WORKSPACE)


def test_slot_capacity(B):
    assert B.moe_slot_capacity(16, 2, 8) == 1152           # 32 + 127*8 = 1048 -> 9*128
    assert B.moe_slot_capacity(0, 1, 1) == 128
    assert B.moe_slot_capacity(8192, 8, 48) % 128 == 0
    assert B.moe_slot_capacity(8192, 8, 48) >= 8192 * 8 + 127 * 48
    assert B.moe_slot_capacity(-1, 1, 1) == -1


def test_gemm_policy_values(B):
    """Every documented policy is accepted and returned as the previous one; others fail."""
    old = B.moe_set_gemm_policy(B.MOE_GEMM_AUTO)
    try:
        for pol in (B.MOE_GEMM_TILED, B.MOE_GEMM_STREAMING, B.MOE_GEMM_STREAMING_N32, B.MOE_GEMM_STREAMING_N64,
                    B.MOE_GEMM_TILED_1CTA, B.MOE_GEMM_TILED_PAIR, B.MOE_GEMM_AUTO):
            prev = B.moe_set_gemm_policy(pol)
            assert B.moe_set_gemm_policy(pol) == pol
            assert prev != pol or pol == B.MOE_GEMM_AUTO
        for bad in (-1, 7):
            with pytest.raises(B.MoeError):
                B.moe_set_gemm_policy(bad)
    finally:
        B.moe_set_gemm_policy(old)


def test_workspace_sizes(B):
    assert B.moe_stage_workspace_size() >= 4
    assert B.moe_route_workspace_size(256, 8, 48) >= 2 * 8 * 48 * 4
    small = B.moe_workspace_size(16, 256, 128, 8, 2)
    big = B.moe_workspace_size(8192, 4096, 3072, 48, 8)
    assert 0 < small < big
    # unsupported shapes give 0
    assert B.moe_workspace_size(16, 100, 128, 8, 2) == 0
    assert B.moe_workspace_size(16, 256, 100, 8, 2) == 0
    assert B.moe_workspace_size(16, 256, 128, 300, 2) == 0


def test_argument_checks_fail_before_any_device_work(B):
    lib = B.library()
    null = ctypes.c_void_p(0)
    # null pointers / bad enums / bad shapes are rejected on the host
    assert lib.moe_route(null, null, 4, 2, 8, 0, null, null, null, null, null, null, 1024, null, 0, null) \
        == B.MOE_ERR_INVALID_ARG
    assert lib.moe_route(null, null, 4, 64, 8, 0, null, null, null, null, null, null, 1024, null, 0, null) \
        == B.MOE_ERR_UNSUPPORTED_SHAPE
    assert lib.moe_prepare_weights(null, null, 1, 128, 64, 0, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_gemm_l1(null, null, null, null, null, 1, 128, 256, 128, null, null, null, null, 0,
                                   null, null, null, null, null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_cast_output(null, null, 4, 7, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_codecs(0, 16, null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_codecs(0, -1, null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_codecs(0xFFFFFFF0, 17, 8, 8, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_codecs(0, 0, null, null, null) == B.MOE_OK
    assert lib.moe_quantize_weights(null, null, 2, 128, 256, null, null, null, null, null, null, null, null, 0,
                                    null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_fold_gate_up_scales(null, null, null, null, 2, 128, 256, null) == B.MOE_ERR_INVALID_ARG
    assert B.moe_quantize_weights_workspace_size(2, 128, 256) >= 2 * 256 * 16 + 2 * 256 * 8
    assert lib.moe_combine_rows(null, 8, null, null, 4, 2, 7, 16, null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_rows(null, 8, null, null, 4, 2, 8, 16, null, null, null) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_combine_rows(null, 8, null, null, 0, 2, 8, 16, null, null, null) == B.MOE_OK  # nothing to do
    w = B.MoeWeights()
    assert lib.moe_forward(null, 4, 256, 100, 8, null, null, 2, 0, ctypes.byref(w), null, 0, null, null, null,
                           null, 0, null) in (B.MOE_ERR_INVALID_ARG, B.MOE_ERR_UNSUPPORTED_SHAPE)


def test_bench_traffic_is_keyed_by_workload_policy_and_kernel_sources():
    """The ncu DRAM figure belongs to one kernel on one workload: other workloads,
    policies or stages get none, and an edit to the kernel's sources drops it."""
    import bench
    for (wl, pol, stage), tr in bench.NCU_TRAFFIC.items():
        other_wl = "skew_top8" if wl != "skew_top8" else "prefill"
        assert (other_wl, pol, stage) not in bench.NCU_TRAFFIC
        assert bench.ncu_traffic(other_wl, pol, stage) is None
        assert bench.ncu_traffic(wl, "tiled1", stage) is None
        assert bench.ncu_traffic(wl, pol, "route") is None
        saved = dict(tr)
        try:
            tr["sources_sha256_16"] = bench.kernel_sources_hash(tr["kernel_sources"])
            assert bench.ncu_traffic(wl, pol, stage) == tr["bytes"]
            tr["sources_sha256_16"] = "0" * 16
            assert bench.ncu_traffic(wl, pol, stage) is None
        finally:
            tr.clear()
            tr.update(saved)


def test_bench_rejects_throttled_or_locked_clocks():
    """A timed region is re-measured once if its clock samples saw a hardware or thermal
    slowdown, or SM clocks well below their maximum with no reason (a leftover lock);
    the power cap alone is kept."""
    import bench
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected({**ok, "sm_mhz": 1900.0, "reasons": ["sw_power_cap"]})
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({**ok, "reasons": [r]})
    assert bench.clocks_rejected({**ok, "sm_mhz": 1000.0})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]})
