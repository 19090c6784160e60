"""Pins for the oracle's tensor quantisation and scale layout (CPU only)."""

import os

import numpy as np
import pytest

from oracle import nvfp4 as q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(tok):
    """A decimal or hex-float (0x1p-130) literal."""
    return float.fromhex(tok) if "0x" in tok else float(tok)


def _golden_blocks():
    out = []
    for line in open(os.path.join(GOLDEN, "quant_blocks.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, gs, xs, sb, nibs, bts = [f.strip() for f in line.split("|")]
        out.append((name, None if gs == "data" else _num(gs),
                    np.array([_num(v) for v in xs.split()], np.float32),
                    int(sb, 16), [int(v) for v in nibs.split()],
                    [int(v, 16) for v in bts.split()]))
    return out


@pytest.mark.parametrize("case", _golden_blocks(), ids=lambda c: c[0])
def test_quantize_hand_derived_blocks(case):
    name, gs, x, sb, nibs, bts = case
    codes, sf, g = q.quantize(x[None, :], gs)
    assert sf[0, 0] == sb
    assert list(q.unpack_nibbles(codes)[0]) == nibs
    assert list(codes[0]) == bts
    if gs is None:
        assert g == np.float32(1.0)


def test_global_scale_divisor_is_6_times_448():
    # "global scale" commit: amax / (6 * 448); 6 * 448 = 2688
    assert q.GLOBAL_SCALE_DIVISOR == np.float32(2688.0)
    assert q.global_scale(np.float32(2688.0)) == np.float32(1.0)


def _rand_bf16(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    x = (r.standard_normal(shape) * scale).astype(np.float32)
    return q.bf16_round(x)


@pytest.mark.parametrize("amax", [1.0, 1e4, 1e30, 3e-30])
def test_block_scales_never_exceed_448(amax):
    """The "global scale" commit's promise: normalising by amax/2688 keeps every
    block scale within UE4M3 range, and the largest block reaches it."""
    x = _rand_bf16((64, 512), 5)
    x = q.bf16_round(x * np.float32(amax / np.abs(x).max()))
    codes, sf, gs = q.quantize(x)
    assert np.all(sf <= q.E4M3_MAX_BYTE)          # sign 0, finite, <= 448
    assert np.all(q.e4m3_decode(sf) <= 448.0)
    # the block holding amax gets a scale near 448 (within e4m3 rounding)
    top = q.e4m3_decode(sf).max()
    assert 448.0 / 1.0625 <= top <= 448.0
    # and dequantised magnitudes reproduce amax to within one e4m3/e2m1 step
    deq = q.dequantize(codes, sf) * float(gs)
    assert abs(np.abs(deq).max() - np.abs(x).max()) <= 0.125 * np.abs(x).max()


def test_all_zero_tensor_gives_zero_scale_and_sign_only_codes():
    x = np.zeros((3, 32), np.float32)
    x[1, :] = -0.0
    codes, sf, gs = q.quantize(x)
    assert gs == 0 and np.all(sf == 0)
    nib = q.unpack_nibbles(codes)
    assert np.all(nib[0] == 0) and np.all(nib[1] == 8) and np.all(nib[2] == 0)


def test_single_nonzero_codes_to_six():
    """A block with one nonzero +-a and zeros elsewhere: the scale is a/6 in
    normalised units; when that is an exact e4m3 value the element is +-6."""
    for a, gs in [(3.0, 1.0), (-96.0, 2.0), (0.375, 0.125)]:
        x = np.zeros((1, 16), np.float32)
        x[0, 5] = a
        codes, sf, _ = q.quantize(x, gs)
        nib = q.unpack_nibbles(codes)[0]
        assert nib[5] == (15 if a < 0 else 7)
        assert np.all(np.delete(nib, 5) == 0)
        assert q.e4m3_decode(sf[0, 0]) == abs(a) / gs / 6.0


def test_constant_block_of_six_times_scale_is_index_7():
    for b in [0x08, 0x20, 0x38, 0x50, 0x7E]:
        s = q.e4m3_decode(np.uint8(b))
        x = np.full((1, 16), 6.0 * s, np.float32)
        codes, sf, _ = q.quantize(x, 1.0)
        assert sf[0, 0] == b
        assert np.all(q.unpack_nibbles(codes) == 7)


def test_every_code_is_the_nearest_grid_point_of_its_block():
    """Brute force: for each element, the chosen dequantised value must be a
    nearest point (ties allowed either way) of that block's grid
    {+-m * scale * gs}, unless the value lies past the top of the grid (then
    the top is chosen).  Checked in fp64 with a small slack for the fp32
    rounding of the scaled value."""
    x = _rand_bf16((48, 256), 6, 3.0)
    codes, sf, gs = q.quantize(x)
    sd = q.e4m3_decode(sf).astype(np.float64)
    grid = np.asarray(q.E2M1_MAGNITUDES)
    nib = q.unpack_nibbles(codes).reshape(48, 16, 16)
    xb = np.abs(x.astype(np.float64)).reshape(48, 16, 16)
    unit = (sd * float(gs))[:, :, None]
    chosen = grid[nib & 7] * unit
    dist = np.abs(xb[..., None] - grid[None, None, None, :] * unit[..., None])
    best = dist.min(axis=-1)
    slack = 1e-6 * unit
    assert np.all(np.abs(xb - chosen) <= best + slack)
    # sign: bit 3 is the sign bit of x
    assert np.array_equal((nib >> 3).astype(bool), np.signbit(x).reshape(48, 16, 16))


def test_fixed_global_scale_saturates_codes_and_scales():
    x = np.full((1, 16), 3000.0, np.float32)
    codes, sf, gs = q.quantize(x, 1.0)      # 3000/6 = 500 > 448
    assert sf[0, 0] == 0x7E and np.all(q.unpack_nibbles(codes) == 7) and gs == 1.0


def _load_layout():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "scale_layout.txt"))
            if l.strip() and not l.startswith("#")]
    return [tuple(int(v) for v in r) for r in rows]


@pytest.mark.parametrize("m,k,ksf,off", _load_layout())
def test_swizzle_offsets_match_hand_computed(m, k, ksf, off):
    assert q.swizzle_offset(m, k, ksf) == off


def test_swizzle_is_a_permutation_and_roundtrips():
    R, ksf = 384, 16
    offs = q.swizzle_offset(*np.meshgrid(np.arange(R), np.arange(ksf), indexing="ij"), ksf)
    assert np.array_equal(np.sort(offs.ravel()), np.arange(R * ksf))
    sf = np.random.default_rng(7).integers(0, 127, (300, 8)).astype(np.uint8)
    flat = q.swizzle(sf)
    assert flat.size == 384 * 8
    assert np.array_equal(q.unswizzle(flat, 300, 8), sf)
