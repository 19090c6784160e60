"""Device-side error reporting: malformed routing tables and out-of-range slot or token
indices are reported in the status word (MOE_ERR_DEVICE_INDEX), and the kernels do no
work with them (nothing is written outside the caller's buffers or for the bad rows)."""

import numpy as np
import pytest
import torch

from oracle import nvfp4 as q
from tests.helpers import dev

pytestmark = pytest.mark.gpu

B = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global B
    from nvfp4_mixture_experts_stage_gb300 import binding
    B = binding


@pytest.fixture(params=["tiled", "tiled1", "tiledp", "stream32"])
def policy(request, _lib):
    pol = {"tiled": B.MOE_GEMM_TILED, "tiled1": B.MOE_GEMM_TILED_1CTA, "tiledp": B.MOE_GEMM_TILED_PAIR,
           "stream32": B.MOE_GEMM_STREAMING_N32}[request.param]
    old = B.moe_set_gemm_policy(pol)
    yield request.param
    B.moe_set_gemm_policy(old)


E, K, I, CAP = 3, 256, 128, 512
GOOD_OFFSETS = [0, 10, 20, 30]
GOOD_POFF = [0, 128, 256, 384]
BAD_TABLES = {
    "unaligned": (GOOD_OFFSETS, [0, 100, 256, 384]),
    "past_capacity": (GOOD_OFFSETS, [0, 128, 256, CAP + 128]),
    "count_above_range": ([0, 200, 210, 220], GOOD_POFF),
    "decreasing": (GOOD_OFFSETS, [0, 256, 128, 384]),
    "negative": (GOOD_OFFSETS, [-128, 128, 256, 384]),
}


def _operands(rows, kdim, seed):
    r = np.random.default_rng(seed)
    codes = r.integers(0, 256, (rows, kdim // 2)).astype(np.uint8)
    sf = np.full((rows, kdim // 16), 0x38, np.uint8)
    return codes, sf


@pytest.mark.parametrize("bad", sorted(BAD_TABLES))
def test_l1_bad_routing_tables_are_reported_and_skipped(policy, bad):
    offs, poff = BAD_TABLES[bad]
    a, asf = _operands(CAP, K, 1)
    w1, w1s = _operands(E * 2 * I, K, 2)
    d_wsf = torch.empty(w1s.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(dev(w1s.reshape(E, 2 * I, K // 16)), d_wsf, E, 2 * I, K, B.MOE_PREP_W1)
    out = torch.full((CAP, 2 * I), 7.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    one = dev(np.ones(E, np.float32))
    B.moe_grouped_gemm_l1(dev(a), dev(q.swizzle(asf)), dev(np.ones(1, np.float32)), dev(np.array(offs, np.int32)),
                          dev(np.array(poff, np.int32)), E, K, I, dev(w1.reshape(E, 2 * I, K // 2)), d_wsf, one, one,
                          B.MOE_L1_GATEUP_BF16, out_bf16=out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == B.MOE_ERR_DEVICE_INDEX
    assert bool((out == 7.0).all())                      # no tile ran


@pytest.mark.parametrize("bad", ["unaligned", "past_capacity"])
def test_l2_bad_routing_tables_are_reported_and_skipped(policy, bad):
    offs, poff = BAD_TABLES[bad]
    h, hsf = _operands(CAP, I, 3)
    w2, w2s = _operands(E * K, I, 4)
    d_wsf = torch.empty(w2s.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(dev(w2s.reshape(E, K, I // 16)), d_wsf, E, K, I, B.MOE_PREP_W2)
    y = torch.full((CAP, K), 7.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_l2(dev(h), dev(q.swizzle(hsf)), dev(np.ones(1, np.float32)), dev(np.array(offs, np.int32)),
                          dev(np.array(poff, np.int32)), E, I, K, dev(w2.reshape(E, K, I // 2)), d_wsf,
                          dev(np.ones(E, np.float32)), B.MOE_L2_ROWS_BF16, y_rows=y, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == B.MOE_ERR_DEVICE_INDEX
    assert bool((y == 7.0).all())


def test_l2_scatter_token_out_of_range_is_reported_and_dropped(policy):
    """One slot names token T (one past the output): its row is dropped, the status is
    set, the other slots still land."""
    T = 40
    h, hsf = _operands(CAP, I, 5)
    w2, w2s = _operands(E * K, I, 6)
    d_wsf = torch.empty(w2s.size, dtype=torch.uint8, device="cuda")
    B.moe_prepare_weights(dev(w2s.reshape(E, K, I // 16)), d_wsf, E, K, I, B.MOE_PREP_W2)
    st_tok = np.full(CAP, -1, np.int32)
    sw = np.zeros(CAP, np.float32)
    for e in range(E):
        st_tok[GOOD_POFF[e]:GOOD_POFF[e] + 10] = np.arange(10) + 10 * e
        sw[GOOD_POFF[e]:GOOD_POFF[e] + 10] = 1.0
    st_tok[GOOD_POFF[1] + 3] = T                         # out of range
    out32 = torch.zeros(T, K, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_grouped_gemm_l2(dev(h), dev(q.swizzle(hsf)), dev(np.ones(1, np.float32)),
                          dev(np.array(GOOD_OFFSETS, np.int32)), dev(np.array(GOOD_POFF, np.int32)), E, I, K,
                          dev(w2.reshape(E, K, I // 2)), d_wsf, dev(np.ones(E, np.float32)), B.MOE_L2_SCATTER,
                          slot_token=dev(st_tok), slot_weight=dev(sw), out32=out32, T=T, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == B.MOE_ERR_DEVICE_INDEX
    got = out32.cpu().numpy()
    assert not got[13].any()                             # the dropped slot's token got nothing
    assert np.abs(got[12]).sum() > 0 and np.abs(got[0]).sum() > 0


@pytest.mark.parametrize("topk", [4, 9])
def test_stage_to_slots_slot_out_of_range_is_reported_and_not_written(topk):
    """A pair_slot entry at or past the capacity is flagged and not written: the rows
    after the capacity (a guard region of the same buffer) stay zero."""
    T, Kx, cap = 20, 512, 256
    r = np.random.default_rng(7)
    x = q.bf16_round(r.standard_normal((T, Kx)).astype(np.float32))
    ps = r.permutation(cap)[:T * topk].astype(np.int32)
    ps[5] = cap                                          # just past the capacity
    ps[9] = cap + 100
    guard = 128
    a = torch.zeros(cap + guard, Kx // 2, dtype=torch.uint8, device="cuda")
    asf = torch.zeros((cap + guard) * Kx // 16, dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(B.moe_stage_workspace_size(), dtype=torch.uint8, device="cuda")
    B.moe_stage_activation_to_slots(torch.from_numpy(x).to(torch.bfloat16).cuda(), dev(ps), topk, cap, a, asf, gs,
                                    ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == B.MOE_ERR_DEVICE_INDEX
    assert not a[cap:].any().item()
    assert not asf[cap * Kx // 16:].any().item()
    # the valid pairs were still written
    rc, _, _ = q.quantize(x)
    got = a.cpu().numpy()
    for i in (0, 1, 2, 30):
        assert np.array_equal(got[ps[i]], rc[i // topk])


def test_stage_to_slots_code_buffer_aligned_to_4_bytes_only():
    """The API accepts a code buffer aligned to 4 bytes; such a buffer takes the general
    kernel (the run kernel's 16-byte stores need 16-byte alignment) with the same bytes."""
    T, Kx, cap, topk = 16, 256, 128, 2
    r = np.random.default_rng(8)
    x = q.bf16_round(r.standard_normal((T, Kx)).astype(np.float32))
    ps = r.permutation(cap)[:T * topk].astype(np.int32)
    xd = torch.from_numpy(x).to(torch.bfloat16).cuda()
    ws = torch.empty(B.moe_stage_workspace_size(), dtype=torch.uint8, device="cuda")
    outs = []
    for shift in (0, 4):
        base = torch.zeros(cap * Kx // 2 + 64, dtype=torch.uint8, device="cuda")
        a = base[shift:shift + cap * Kx // 2].view(cap, Kx // 2)
        asf = torch.zeros(cap * Kx // 16, dtype=torch.uint8, device="cuda")
        gs = torch.zeros(1, dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.moe_stage_activation_to_slots(xd, dev(ps), topk, cap, a, asf, gs, ws=ws, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0
        outs.append((a.cpu().numpy().copy(), asf.cpu().numpy().copy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    rc, _, _ = q.quantize(x)
    for i in range(T * topk):
        assert np.array_equal(outs[1][0][ps[i]], rc[i // topk])


def test_bounded_wait_gives_up_reports_timeout_and_leaves_the_context_usable():
    """A wait on a barrier nothing completes ends after the library's limit with
    MOE_ERR_TIMEOUT; a second waiter returns through the abort flag; the next call works."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    B.moe_selftest_bounded_wait(st, res)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert st.item() == B.MOE_ERR_TIMEOUT
    assert res.cpu().tolist() == [1, 1]
    assert 0.9 < dt < 10.0
    # the context still runs work
    x = q.bf16_round(np.random.default_rng(9).standard_normal((4, 64)).astype(np.float32))
    codes = torch.zeros(4, 32, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(4 * 4, dtype=torch.uint8, device="cuda")
    gs = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(B.moe_stage_workspace_size(), dtype=torch.uint8, device="cuda")
    B.moe_stage_activation(torch.from_numpy(x).to(torch.bfloat16).cuda(), codes, sf, B.MOE_SF_ROWMAJOR, gs, ws=ws)
    torch.cuda.synchronize()
    rc, rs, rg = q.quantize(x)
    assert np.array_equal(codes.cpu().numpy(), rc) and np.float32(gs.item()) == rg
