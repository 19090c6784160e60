"""Pins for the oracle's codecs (CPU only).

Each test ties the oracle to something other than itself: torch's float8 /
bfloat16 implementations (independent library code), brute-force nearest
search, hand-derived fixtures under tests/golden, or exhaustive round trips.
"""

import os

import numpy as np
import pytest
import torch

from oracle import nvfp4 as q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32_neighbours(vals, n_ulps=4):
    """fp32 values within n_ulps of each value (both sides), non-negative."""
    v = np.asarray(vals, np.float32).view(np.int32).astype(np.int64)
    d = np.arange(-n_ulps, n_ulps + 1)
    out = (v[:, None] + d[None, :]).reshape(-1)
    out = out[(out >= 0) & (out < 0x7F800000)]
    return out.astype(np.int32).view(np.float32)


# ---------------------------------------------------------------- UE4M3 ----

def test_e4m3_decode_matches_torch_bit_view_all_bytes():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = q.e4m3_decode(b)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    # signed zero: 0x80 is -0.0
    assert np.signbit(got[0x80]) and got[0x80] == 0.0


def test_byte_0x3f_is_a_bit_view_not_a_value_conversion():
    """The "0x3F" commit (src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py commits):
    scale bytes must be unpacked by a bit view, which is the inverse of the
    packing view; converting the integer 63 to float8 is a different thing.
    The page's "~0.984" for the view is not what e4m3fn gives: 0x3F is
    sign 0, exponent 0111, mantissa 111 -> 1.875 (recorded as a page error)."""
    assert q.e4m3_decode(np.uint8(0x3F)) == 1.875
    # value conversion of 63.0 lands on 64.0 = 2**6 = byte 0x68, not 0x3F
    conv = torch.tensor([63.0]).to(torch.float8_e4m3fn)
    assert conv.view(torch.uint8).item() == 0x68 and conv.float().item() == 64.0
    assert q.e4m3_decode(np.uint8(0x68)) == 64.0
    # pack (bytes -> uint32 words) and unpack are exact inverses on every byte
    allb = np.arange(256, dtype=np.uint8)
    words = q.pack_scale_bytes(allb.reshape(-1, 4))
    assert np.array_equal(q.unpack_scale_words(words).reshape(-1), allb)
    # little-endian: the first scale of a row is the low byte of the word
    assert q.pack_scale_bytes(np.array([[0x3F, 0, 0, 0]], np.uint8))[0, 0] == 0x3F


def test_e4m3_encode_roundtrips_every_finite_nonnegative_byte():
    b = np.arange(0x7F, dtype=np.uint8)  # 0x00..0x7E
    vals = q.e4m3_decode(b).astype(np.float32)
    assert np.array_equal(q.e4m3_encode_satfinite(vals), b)


def _torch_e4m3_bytes(f):
    return torch.from_numpy(np.asarray(f, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_rne_near_every_midpoint():
    """torch's float8_e4m3fn cast rounds to nearest even; below 448 it never
    overflows, so it is an independent reference for the rounding."""
    grid = q.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2.0  # exact in fp64; all fp32-representable
    probe = np.concatenate([_f32_neighbours(mids, 6), _f32_neighbours(grid, 3)])
    probe = probe[probe < 448.0]
    assert np.array_equal(q.e4m3_encode_satfinite(probe), _torch_e4m3_bytes(probe))


def test_e4m3_encode_matches_torch_on_all_bf16_patterns_and_random_fp32():
    bf = (np.arange(0, 0x43E0, dtype=np.uint32) << 16).view(np.float32)  # [0, 448)
    rnd = np.random.default_rng(1).uniform(0, 448, 2_000_000).astype(np.float32)
    tiny = np.random.default_rng(2).uniform(0, 2 ** -5, 500_000).astype(np.float32)
    for probe in (bf, rnd, tiny):
        probe = probe[probe < 448.0]
        assert np.array_equal(q.e4m3_encode_satfinite(probe), _torch_e4m3_bytes(probe))


def test_e4m3_encode_saturates_at_448():
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(q.e4m3_encode_satfinite(big) == 0x7E)
    # tiny values: 2**-10 is the tie between 0 and the smallest subnormal -> 0
    assert q.e4m3_encode_satfinite(np.float32(2.0 ** -10)) == 0
    assert q.e4m3_encode_satfinite(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 1


# ---------------------------------------------------------------- E2M1 -----

def _load_grid():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_grid.txt"))
            if l.strip() and not l.startswith("#")]
    return {int(a): float(b) for a, b in rows}


def test_e2m1_nibble_table_matches_golden():
    grid = _load_grid()
    got = q.e2m1_decode_nibble(np.arange(16, dtype=np.uint8))
    for n, v in grid.items():
        assert got[n] == v and np.signbit(got[n]) == np.signbit(v), n


def _brute_nearest_index(v):
    """Nearest of the 8 magnitudes by distance; ties to the even index;
    values past 6 -> index 7."""
    g = np.asarray(q.E2M1_MAGNITUDES, np.float64)
    d = np.abs(np.asarray(v, np.float64)[:, None] - g[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates pick an even index if one exists
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return pick.astype(np.uint8)


def test_e2m1_index_matches_brute_force_nearest():
    g = np.asarray(q.E2M1_MAGNITUDES, np.float32)
    mids = (g[:-1] + g[1:]) / 2
    probe = np.concatenate([
        _f32_neighbours(mids, 8), _f32_neighbours(g, 3),
        np.random.default_rng(3).uniform(0, 7, 1_000_000).astype(np.float32),
        (np.arange(0, 0x40E0, dtype=np.uint32) << 16).view(np.float32),  # bf16 grid to 7
    ])
    probe = probe[probe <= 6.0]
    assert np.array_equal(q.e2m1_index(probe), _brute_nearest_index(probe))
    # saturation past the largest magnitude
    assert np.all(q.e2m1_index(np.array([6.0001, 7, 100, 3e38, np.inf], np.float32)) == 7)
    # the grid itself maps to its own index
    assert np.array_equal(q.e2m1_index(g), np.arange(8))


def test_nibble_pack_unpack_are_inverses():
    b = np.arange(256, dtype=np.uint8)
    assert np.array_equal(q.pack_nibbles(q.unpack_nibbles(b[None, :]))[0], b)
    lo, hi = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    pairs = np.stack([lo.ravel(), hi.ravel()], axis=1).astype(np.uint8)
    packed = q.pack_nibbles(pairs)
    assert np.array_equal(q.unpack_nibbles(packed), pairs)
    # even-K element in the low nibble
    assert q.pack_nibbles(np.array([[0x1, 0xF]], np.uint8))[0, 0] == 0xF1


# ---------------------------------------------------------------- BF16 -----

def test_bf16_round_matches_torch():
    r = np.random.default_rng(4)
    x = np.concatenate([
        r.standard_normal(1_000_000).astype(np.float32) * np.float32(100),
        (r.integers(0, 2 ** 31, 1_000_000, dtype=np.uint64).astype(np.uint32)
         & np.uint32(0x7F7FFFFF)).view(np.float32),  # random finite bit patterns
        # exact ties: low half-word 0x8000
        ((r.integers(0, 0x7F00, 10000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
    ])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = q.bf16_round(x)
    assert np.array_equal(ref.view(np.uint32), got.view(np.uint32))
