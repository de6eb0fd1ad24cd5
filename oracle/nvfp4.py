"""NVFP4 number formats for the CPU oracle (float64, exact).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline may import this package; the product path never does.

Formats (the weight value is E2M1 code x UE4M3 scale of its 16-group):

* E2M1 (4-bit codes with a UE4M3 scale for every group of 16 weights, per the
  header constants of "moe_sel_census.rs"; "moe_union_probe.rs" counts a row as
  in_f/2 code bytes plus in_f/16 UE4M3 scale bytes).  4-bit code c: sign s = c>>3, exponent e =
  (c>>1)&3, mantissa m = c&1; value (-1)^s * (m/2 if e == 0 else (1+m/2)*2^(e-1)).
  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; code 8 is -0.
* UE4M3 scale byte b (bit 7 must be 0, 0x7F is NaN and rejected): e = (b>>3)&15,
  m = b&7; value (m/8)*2^-6 if e == 0 else (1+m/8)*2^(e-7).  Max 0x7E = 448.
* Packing (a reading; the pages are silent): two codes per byte, the low
  nibble holds the even element, the high nibble the odd one.

The activation quantiser Q is a reading too (the pages never quantise
activations to FP4; a block-scaled FP4 x FP4 tensor-core product needs it):

* row exponent s = the smallest integer with amax_row <= 6 * 448 * 2^s (0 for a
  zero row);
* block scale sb = UE4M3 value nearest to amax_16 / (6 * 2^s), ties to the even
  encoding;
* code = E2M1 value nearest to v / (sb * 2^s), saturating at 6, ties to the
  even encoding, sign bit set iff v < 0; a block with sb == 0 is all zero codes.

Every decision is an exact comparison of |v| * 2^-s against products of a
midpoint and a scale, all of which are exact in float64 (and in float32), so a
float32 implementation takes the same decisions bit for bit.
"""
from __future__ import annotations

import numpy as np

E2M1_MAG_CODES = 8


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code (closed form)."""
    if not 0 <= code < 16:
        raise ValueError("E2M1 code out of range")
    s, e, m = code >> 3, (code >> 1) & 3, code & 1
    mag = 0.5 * m if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


# The exact 16-entry table, indexed by code.
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def ue4m3_value(b: int) -> float:
    """Value of one unsigned E4M3 scale byte (closed form); bit 7 and 0x7F are invalid."""
    if not 0 <= b <= 0x7E:
        raise ValueError(f"invalid UE4M3 scale byte 0x{b:02x}")
    e, m = (b >> 3) & 15, b & 7
    return (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Values of the 127 valid encodings 0x00..0x7E, increasing with the code.
UE4M3_TABLE = np.array([ue4m3_value(b) for b in range(0x7F)], dtype=np.float64)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64, exactly."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def check_scales(scales: np.ndarray) -> None:
    s = np.asarray(scales)
    if np.any(s > 0x7E):
        raise ValueError("UE4M3 scale with bit 7 set or NaN encoding")


def dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode planar NVFP4 rows to float64.

    codes u8 [..., n/2] (low nibble = even element), scales u8 [..., n/16];
    returns float64 [..., n] = E2M1(code) * UE4M3(scale of the element's 16-group).
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    check_scales(scales)
    n = codes.shape[-1] * 2
    if scales.shape[-1] * 16 != n:
        raise ValueError("scale plane does not match code plane")
    nib = np.empty(codes.shape[:-1] + (n,), dtype=np.uint8)
    nib[..., 0::2] = codes & 0x0F
    nib[..., 1::2] = codes >> 4
    vals = E2M1_TABLE[nib]
    sc = np.repeat(UE4M3_TABLE[scales], 16, axis=-1)
    return vals * sc


# ---------------------------------------------------------------------------
# Quantiser Q (reading; see module docstring)
# ---------------------------------------------------------------------------

ROW_LIMIT = 6.0 * 448.0            # largest magnitude one block can hold at s = 0
# Midpoints between consecutive UE4M3 values, times 6 (exact in float64).
_UE4M3_MID6 = 6.0 * 0.5 * (UE4M3_TABLE[:-1] + UE4M3_TABLE[1:])
# Midpoints between consecutive E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
_E2M1_MAGS = E2M1_TABLE[:8]
_E2M1_MIDS = 0.5 * (_E2M1_MAGS[:-1] + _E2M1_MAGS[1:])   # .25 .75 1.25 1.75 2.5 3.5 5


def row_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer s with amax <= 6*448*2^s, elementwise (0 where amax == 0)."""
    amax = np.asarray(amax, dtype=np.float64)
    s = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    if np.any(nz):
        _, e = np.frexp(amax[nz] / ROW_LIMIT)
        e = e.astype(np.int64)
        a = amax[nz]
        # exact fix-ups: enforce amax <= L*2^e and amax > L*2^(e-1)
        for _ in range(3):
            up = a > np.ldexp(ROW_LIMIT, e)
            e = e + up
            down = a <= np.ldexp(ROW_LIMIT, e - 1)
            e = e - down
        s[nz] = e
    return s


def nearest_even(keys: np.ndarray, mids: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value for sorted grid midpoints, ties to the even index.

    The grid values are increasing; ``mids[j]`` separates grid values j and j+1.
    """
    left = np.searchsorted(mids, keys, side="left")          # number of mids < key
    tie = np.zeros(keys.shape, dtype=bool)
    inb = left < mids.shape[0]
    tie[inb] = mids[left[inb]] == keys[inb]
    up = tie & ((left + 1) % 2 == 0)
    return left + up


def block_scale_codes(bamax_scaled: np.ndarray) -> np.ndarray:
    """UE4M3 encoding nearest to r = bamax_scaled / 6 (ties to the even encoding).

    ``bamax_scaled`` is a block's amax times 2^-s; it is compared with 6 x the
    midpoints between consecutive UE4M3 values, all exact products.
    """
    return nearest_even(np.asarray(bamax_scaled, dtype=np.float64), _UE4M3_MID6).astype(np.uint8)


def e2m1_magnitude_codes(keys: np.ndarray, sb: np.ndarray) -> np.ndarray:
    """E2M1 magnitude code (0..7) nearest to keys / sb, saturating at 6, ties to the even code.

    keys [nb, m] are |v| * 2^-s, sb [nb] the block scale values; the comparison
    is against midpoint * sb, exact in float64.
    """
    keys = np.asarray(keys, dtype=np.float64)
    thr = _E2M1_MIDS[None, :] * np.asarray(sb, dtype=np.float64).reshape(-1, 1)   # [nb, 7]
    mag = np.zeros(keys.shape, dtype=np.uint8)
    for j in range(7):
        t = thr[:, j:j + 1]
        above = keys > t
        tie = (keys == t) & (j % 2 == 1)                    # upper neighbour even for odd j
        mag += (above | tie).astype(np.uint8)
    return mag


def quantize(v: np.ndarray):
    """Q over the last axis (length a multiple of 16).

    v: float64 array [..., n] of finite values.  Returns (codes u8 [..., n/2],
    scales u8 [..., n/16], s int64 [...]) in the same planar layout as the weights.
    """
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % 16:
        raise ValueError("row length must be a multiple of 16")
    if not np.all(np.isfinite(v)):
        raise ValueError("Q needs finite input")
    lead = v.shape[:-1]
    a = np.abs(v)
    s = row_exponent(a.max(axis=-1) if n else np.zeros(lead))
    a_s = np.ldexp(a, -s[..., None])                       # |v| * 2^-s, exact
    keys = a_s.reshape(-1, 16)
    sb_code = block_scale_codes(keys.max(axis=1))          # <= 0x7E by choice of s
    sb = UE4M3_TABLE[sb_code]
    mag = e2m1_magnitude_codes(keys, sb)
    neg = v.reshape(-1, 16) < 0
    code = mag | (neg.astype(np.uint8) << 3)
    code[sb == 0, :] = 0                                    # a zero-scale block is all zero codes
    code = code.reshape(lead + (n,))
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, sb_code.reshape(lead + (n // 16,)), s


def dequant_q(codes: np.ndarray, scales: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Value of a Q result: E2M1(code) * UE4M3(scale) * 2^s."""
    return np.ldexp(dequant(codes, scales), np.asarray(s)[..., None])


def from_interleaved(blob: np.ndarray, in_f: int):
    """Planar (codes, scales) of rows stored as 36-byte blocks per 64 weights.

    The pages' own banks use this storage: `mk_bank` in `fn main` of "moe_sk_repro.rs"
    sizes a row at 36 bytes for every 64 weights (row bytes in_f / 64 * 36), and the
    `BLK` constant of "moe_sel_census.rs" splits such a block into four UE4M3 scale bytes
    and thirty-two code bytes.  Reading
    of the order the pages leave open: the block's 4 scale bytes come first (scale i
    covers weights 16i .. 16i+15 of the block), then its 32 code bytes (two codes per
    byte, low nibble = even weight, as in the planar layout).

    blob: uint8 [..., in_f / 64 * 36].  Returns codes uint8 [..., in_f / 2] and scales
    uint8 [..., in_f / 16].
    """
    blob = np.asarray(blob, dtype=np.uint8)
    if in_f % 64:
        raise ValueError("in_f must be a multiple of 64")
    nblk = in_f // 64
    if blob.shape[-1] != nblk * 36:
        raise ValueError("row length must be in_f / 64 * 36 bytes")
    b = blob.reshape(blob.shape[:-1] + (nblk, 36))
    scales = b[..., :4].reshape(blob.shape[:-1] + (in_f // 16,))
    codes = b[..., 4:].reshape(blob.shape[:-1] + (in_f // 2,))
    return codes.copy(), scales.copy()
