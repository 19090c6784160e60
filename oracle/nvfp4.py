"""NVFP4 encoding, restated on the CPU (oracle; test infrastructure only).

Sources, all on the nvfp4-megamoe-kernel commit pages:

* commits of ``src/nvfp4_megamoe_kernel/nvfp4_mega_moe.py``:
  - the "three bugs fixed" commit that introduced ``_quantize_to_e2m1``:
    E2M1 codes are sign-magnitude nibbles (bit 3 = sign, bits 2..0 = index
    of the magnitude in {0, 0.5, 1, 1.5, 2, 3, 4, 6}); the stored block scale
    is block_max / 6 (the dequantisation factor); each value snaps to the
    nearest E2M1 magnitude;
  - the "global scale" commit: gs = amax / (6 * 448) and the tensor is
    normalised by it before block quantisation so every block scale stays at
    or below the UE4M3 maximum 448;
  - the "0x3F" commit: packing and unpacking of scale bytes are bit views, not
    value conversions, and must be exact inverses;
  - the "global scale as alpha" commit: the global scale is not folded into
    the block scales; it is applied later as the GEMM epilogue alpha.
* commits of ``tests``: the "float4_e2m1fn_x2" commit -- two codes per byte,
  packed along K.
* commits of ``src``: the "scale-factor layout" commits -- the block-scaled
  MMA wants its scales in 128-row x 4-column atoms with
  m = f0 + 32*f1 + 128*f2 and k_sf = f4 + 4*f5.

Readings where the pages are silent (each also listed in the design notes):

* rounding: UE4M3 and E2M1 both round to nearest, ties to even encoding,
  saturating to the largest finite value (448 and 6);
* fp32 order of operations: gs = amax / 2688; rg = 1 / gs (saturated to the
  largest finite fp32); block scale s = (bm * rg) / 6; code value
  v = (|x| * rg) * (1 / decode(e4m3(s)));
* a block whose scale encodes to 0 gets sign-only nibbles; gs == 0 gives all
  zero scales and sign-only nibbles;
* the sign nibble bit is the IEEE sign bit of x (so -0.0 and small negatives
  that round to zero code as 0x8);
* the even-K element sits in the low nibble of each byte.
"""

import numpy as np

F32 = np.float32
FLT_MAX = F32(np.finfo(np.float32).max)

#: E2M1 magnitudes, indexed by the low three bits of a nibble.
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)

#: Largest finite UE4M3 value and its byte.
E4M3_MAX = 448.0
E4M3_MAX_BYTE = 0x7E

#: gs = amax / (6 * 448): the largest code magnitude times the largest scale.
GLOBAL_SCALE_DIVISOR = F32(6.0 * 448.0)  # 2688

BLOCK = 16  # elements per block scale


# --------------------------------------------------------------------------
# UE4M3 / E4M3 codec (bit-level)
# --------------------------------------------------------------------------

def e4m3_decode(b):
    """Value of each byte read as float8 e4m3fn (1 sign, 4 exponent, 3 mantissa
    bits, bias 7; exponent 0 is subnormal m * 2**-9; 0x7F/0xFF are NaN).

    This is the bit view the "0x3F" commit insists on: the byte pattern *is*
    the number.  Returns float64 (every e4m3 value is exact there)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode_satfinite(f):
    """Encode non-negative fp32 values as UE4M3 bytes: round to nearest, ties to
    even mantissa, saturate at 448 (0x7E).  Sign bit is always 0.

    Subnormal range (f < 2**-6): the byte is the nearest integer q of f * 2**9
    (q == 8 is exactly the smallest normal, byte 0x08).  Normal range: split
    f = (1 + q/8) * 2**e and round q."""
    f = np.asarray(f, dtype=np.float32).astype(np.float64)
    if np.any(f < 0) or np.any(np.isnan(f)):
        raise ValueError("e4m3_encode_satfinite takes non-negative, non-NaN input")
    out = np.zeros(f.shape, dtype=np.int64)
    sub = f < 2.0 ** -6
    q_sub = np.rint(f * 512.0)  # np.rint: round half to even
    out = np.where(sub, q_sub, out)
    with np.errstate(divide="ignore", invalid="ignore"):
        mant, ex = np.frexp(np.where(sub, 1.0, np.minimum(f, 1e6)))  # f = mant * 2**ex, mant in [0.5, 1)
    e = ex - 1
    q = np.rint((mant * 2.0 - 1.0) * 8.0)  # exact: mant*2-1 has <= 24 bits
    carry = q == 8
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 0, q)
    byte = (e + 7) * 8 + q
    byte = np.where(byte > E4M3_MAX_BYTE, E4M3_MAX_BYTE, byte)
    out = np.where(sub, out, byte)
    return out.astype(np.uint8)


# --------------------------------------------------------------------------
# E2M1 codec
# --------------------------------------------------------------------------

def e2m1_index(v):
    """Magnitude index (0..7) of the E2M1 value nearest to each non-negative
    fp32 v; ties go to the even index (the even encoding); values past 6
    saturate to index 7.  The tie points are the midpoints 0.25, 0.75, 1.25,
    1.75, 2.5, 3.5 and 5."""
    v = np.asarray(v, dtype=np.float32)
    idx = ((v > F32(0.25)).astype(np.uint8)
           + (v >= F32(0.75)) + (v > F32(1.25)) + (v >= F32(1.75))
           + (v > F32(2.5)) + (v >= F32(3.5)) + (v > F32(5.0)))
    return idx.astype(np.uint8)


def e2m1_decode_nibble(n):
    """Signed value of a 4-bit code (bit 3 sign, bits 2..0 magnitude index)."""
    n = np.asarray(n, dtype=np.uint8)
    mag = np.asarray(E2M1_MAGNITUDES)[n & 7]
    return np.where((n >> 3) & 1, -mag, mag)


def pack_nibbles(nib):
    """[..., C] nibbles -> [..., C/2] bytes; element 2i in the low nibble."""
    nib = np.asarray(nib, dtype=np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    """Inverse of :func:`pack_nibbles`."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pack_scale_bytes(sf_bytes):
    """Four consecutive scale bytes of a row -> one little-endian uint32 (the
    packed activation-scale form); a bit view, no value conversion."""
    sf = np.ascontiguousarray(np.asarray(sf_bytes, dtype=np.uint8))
    return sf.view(np.uint32)


def unpack_scale_words(words):
    """Inverse of :func:`pack_scale_bytes` (a bit view again)."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.uint32))
    return w.view(np.uint8)


# --------------------------------------------------------------------------
# Tensor quantisation
# --------------------------------------------------------------------------

def global_scale(amax):
    """gs = amax / (6 * 448) in fp32."""
    return F32(F32(amax) / GLOBAL_SCALE_DIVISOR)


def reciprocal_global_scale(gs):
    """rg = 1 / gs in fp32, saturated to the largest finite fp32 (gs so small
    that 1/gs overflows)."""
    gs = F32(gs)
    with np.errstate(divide="ignore", over="ignore"):
        rg = F32(F32(1.0) / gs)
    if not np.isfinite(rg):
        rg = FLT_MAX
    return rg


def quantize(x, gs=None):
    """Quantise a 2-D tensor to NVFP4.

    x: [R, C] float32 (BF16 values widened exactly), C % 16 == 0.
    gs: None -> computed from the tensor (amax / 2688); else the fixed fp32
        global scale to use (the calibrated mode of the vllm/nvfp4_cutedsl.py
        commits).

    Returns (codes [R, C/2] uint8, sf [R, C/16] uint8 row-major, gs float32).
    """
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    if C % BLOCK:
        raise ValueError("C must be a multiple of 16")
    ax = np.abs(x)
    if gs is None:
        amax = F32(ax.max()) if ax.size else F32(0.0)
        gs = global_scale(amax)
    gs = F32(gs)
    sign = np.signbit(x).astype(np.uint8) << 3
    if gs == 0:
        return pack_nibbles(sign), np.zeros((R, C // BLOCK), np.uint8), gs
    rg = reciprocal_global_scale(gs)
    blocks = ax.reshape(R, C // BLOCK, BLOCK)
    bm = blocks.max(axis=2)
    with np.errstate(over="ignore"):
        s = (bm * rg) / F32(6.0)                      # fp32, two roundings
    sb = e4m3_encode_satfinite(s)                      # [R, C/16]
    sd = e4m3_decode(sb).astype(np.float32)
    with np.errstate(divide="ignore"):
        rb = np.where(sd > 0, F32(1.0) / np.where(sd > 0, sd, F32(1.0)), F32(0.0)).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        v = (blocks * rg) * rb[:, :, None]             # (|x| * rg) * rb, fp32
    idx = e2m1_index(v)
    idx = np.where((sd > 0)[:, :, None], idx, 0).astype(np.uint8)
    nib = sign | idx.reshape(R, C)
    return pack_nibbles(nib), sb, gs


def dequantize(codes, sf):
    """Exact float64 values of an NVFP4 tensor (without the global scale):
    E2M1 value times the decoded block scale."""
    nib = unpack_nibbles(codes)
    R, C = nib.shape
    vals = e2m1_decode_nibble(nib).reshape(R, C // BLOCK, BLOCK)
    return (vals * e4m3_decode(sf)[:, :, None]).reshape(R, C)


# --------------------------------------------------------------------------
# Block-scale swizzle for the block-scaled MMA
# --------------------------------------------------------------------------

ATOM_ROWS = 128
ATOM_COLS = 4
ATOM_BYTES = ATOM_ROWS * ATOM_COLS


def swizzle_offset(m, k, k_sf):
    """Byte offset of scale (row m, scale column k) in the swizzled layout of a
    tensor with k_sf scale columns (k_sf % 4 == 0).

    Within an atom of 128 rows x 4 scale columns (512 bytes), writing
    m = f0 + 32 f1 + 128 f2 (f0 < 32, f1 < 4) and k = f4 + 4 f5 (f4 < 4):
    offset = 16 f0 + 4 f1 + f4.  Atoms are stored row-block major:
    atom index = f2 * (k_sf / 4) + f5."""
    m = np.asarray(m, dtype=np.int64)
    k = np.asarray(k, dtype=np.int64)
    f0, f1, f2 = m % 32, (m // 32) % 4, m // 128
    f4, f5 = k % 4, k // 4
    return (f2 * (k_sf // 4) + f5) * ATOM_BYTES + f0 * 16 + f1 * 4 + f4


def swizzle(sf):
    """[R, k_sf] row-major scale bytes -> swizzled flat array.  R is padded up
    to a multiple of 128 with zero scales; k_sf must be a multiple of 4."""
    sf = np.asarray(sf, dtype=np.uint8)
    R, k_sf = sf.shape
    if k_sf % ATOM_COLS:
        raise ValueError("scale columns must be a multiple of 4")
    Rp = -(-R // ATOM_ROWS) * ATOM_ROWS
    out = np.zeros(Rp * k_sf, dtype=np.uint8)
    m, k = np.meshgrid(np.arange(R), np.arange(k_sf), indexing="ij")
    out[swizzle_offset(m, k, k_sf)] = sf
    return out


def unswizzle(flat, R, k_sf):
    """Inverse of :func:`swizzle` (first R rows)."""
    flat = np.asarray(flat, dtype=np.uint8)
    m, k = np.meshgrid(np.arange(R), np.arange(k_sf), indexing="ij")
    return flat[swizzle_offset(m, k, k_sf)]


# --------------------------------------------------------------------------
# BF16
# --------------------------------------------------------------------------

def bf16_round(f):
    """Round fp32 to the nearest BF16 (ties to even) and return it as fp32.
    Inputs are finite."""
    u = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (r.astype(np.uint32) << 16).view(np.float32)


def bf16_bits(f):
    """BF16 bit patterns (uint16) of fp32 values already on the BF16 grid, or
    rounded to it first."""
    return (bf16_round(f).view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(b):
    """fp32 values of BF16 bit patterns."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
