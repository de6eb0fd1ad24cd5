"""Pins for the oracle's number formats and quantiser (CPU only).

The E2M1 table is pinned to the OCP MX specification's value table, the UE4M3
decoder to PyTorch's float8_e4m3fn decoder, and the quantiser Q to a brute-force
nearest-value search written with exact rationals.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4


def test_e2m1_table_matches_ocp_mx_values(golden_dir):
    rows = [l.split() for l in open(os.path.join(golden_dir, "e2m1_values.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        got = nvfp4.E2M1_TABLE[code]
        assert got == val
        assert np.signbit(got) == np.signbit(val), code       # code 8 is -0


def test_ue4m3_matches_torch_float8_e4m3fn():
    b = torch.arange(0x7F, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(nvfp4.UE4M3_TABLE, ref)
    assert nvfp4.UE4M3_TABLE[0x7E] == 448.0
    assert nvfp4.UE4M3_TABLE[1] == 2.0 ** -9
    assert nvfp4.UE4M3_TABLE[0x08] == 2.0 ** -6 and nvfp4.UE4M3_TABLE[0x30] == 0.5
    with pytest.raises(ValueError):
        nvfp4.ue4m3_value(0x7F)
    with pytest.raises(ValueError):
        nvfp4.dequant(np.zeros((1, 8), np.uint8), np.array([[0x80]], np.uint8))


def test_dequant_nibble_order_and_groups():
    # byte 0x21: element 0 = code 1 (0.5), element 1 = code 2 (1.0)
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x21
    codes[0, 8] = 0xF7                      # element 16 = code 7 (6), element 17 = code 15 (-6)
    scales = np.array([[0x38, 0x30]], np.uint8)   # 1.0 then 0.5
    v = nvfp4.dequant(codes, scales)[0]
    assert v[0] == 0.5 and v[1] == 1.0
    assert v[16] == 3.0 and v[17] == -3.0
    assert np.all(v[2:16] == 0)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]              # finite patterns only
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = nvfp4.bf16_to_f64(bits)
    fin = np.isfinite(t)
    assert np.array_equal(got[fin], t[fin])


# ---------------------------------------------------------------------------
# Quantiser Q against brute force
# ---------------------------------------------------------------------------

UE = [Fraction(v) for v in nvfp4.UE4M3_TABLE]
MAGS = [Fraction(v) for v in nvfp4.E2M1_TABLE[:8]]


def nearest_index(target: Fraction, grid):
    best = None
    for i, g in enumerate(grid):
        d = abs(target - g)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def q_brute(row):
    vals = [Fraction(float(x)) for x in row]
    amax = max(abs(v) for v in vals)
    s = 0
    if amax > 0:
        s = -300
        while amax > 6 * 448 * Fraction(2) ** s:
            s += 1
    codes, scales = [], []
    for b in range(len(vals) // 16):
        blk = vals[16 * b:16 * b + 16]
        bm = max(abs(v) for v in blk)
        sbc = nearest_index(bm / (6 * Fraction(2) ** s), UE)
        scales.append(sbc)
        sb = UE[sbc]
        for v in blk:
            if sb == 0:
                codes.append(0)
                continue
            m = nearest_index(min(abs(v) / (sb * Fraction(2) ** s), Fraction(6)), MAGS)
            codes.append(m | (8 if v < 0 else 0))
    return codes, scales, s


def unpack(packed):
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def test_quantize_matches_brute_force_random_rows():
    rng = np.random.default_rng(1)
    rows = []
    for i in range(120):
        scale = 2.0 ** rng.integers(-30, 30)
        r = rng.standard_normal(32) * scale
        if i % 7 == 0:
            r[:16] *= 2.0 ** -20                 # tiny block next to a big one
        if i % 11 == 0:
            r[5] = 0.0
        rows.append(r.astype(np.float32).astype(np.float64))
    rows.append(np.zeros(32))
    rows.append(np.full(32, -0.0))
    # exact ties: values on E2M1 and UE4M3 midpoints
    tie = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4, dtype=np.float64)
    rows.append(tie)
    rows.append(-tie)
    v = np.stack(rows)
    c, sc, s = nvfp4.quantize(v)
    c = unpack(c)
    for i, r in enumerate(rows):
        bc, bs, bexp = q_brute(r)
        assert int(s[i]) == bexp, i
        assert list(sc[i]) == bs, i
        assert list(c[i]) == bc, i


def test_e2m1_codes_exhaustive_over_bf16_and_scales():
    """Every finite bf16 magnitude x every nonzero UE4M3 scale: nearest E2M1, ties even."""
    bits = np.arange(0, 0x7F80, dtype=np.uint16)             # finite non-negative bf16
    vals = nvfp4.bf16_to_f64(bits)
    mags = nvfp4.E2M1_TABLE[:8]
    for sbc in range(1, 0x7F):
        sb = nvfp4.UE4M3_TABLE[sbc]
        keys = vals
        got = nvfp4.e2m1_magnitude_codes(keys[None, :], np.array([sb]))[0]
        # brute force: distance to each grid point (exact here: few significant bits,
        # only keys within 2^+-60 of the scale are compared, others are trivially 0 or 7)
        d = np.abs(np.minimum(keys, 6.0 * sb)[:, None] - mags[None, :] * sb)
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        # among equal distances prefer the even code
        even = cand & (np.arange(8)[None, :] % 2 == 0)
        ref = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        inr = (keys == 0) | ((keys > sb * 2.0 ** -60) & (keys < sb * 2.0 ** 60))
        assert np.array_equal(got[inr], ref[inr]), sbc
        assert np.all(got[keys >= 6 * sb] == 7)
        assert np.all(got[(keys > 0) & (keys < 0.25 * sb)] == 0)


def test_block_scale_codes_exhaustive():
    """Block amax over all finite bf16 magnitudes: nearest UE4M3 to amax/6, ties even."""
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    a = nvfp4.bf16_to_f64(bits)
    a = a[a <= 6 * 448]
    got = nvfp4.block_scale_codes(a)
    grid = nvfp4.UE4M3_TABLE
    d = np.abs(a[:, None] / 6.0 - grid[None, :])   # /6 may round; check ties exactly below
    ref = d.argmin(axis=1)
    # resolve near-ties with exact rational arithmetic
    srt = np.sort(d, axis=1)
    close = np.nonzero(srt[:, 1] - srt[:, 0] <= 1e-12 * np.maximum(srt[:, 0], 1e-300))[0]
    for i in close:
        ref[i] = nearest_index(Fraction(float(a[i])) / 6, UE)
    assert np.array_equal(got, ref)


def test_row_exponent_edges():
    L = 6.0 * 448.0
    a = np.array([0.0, L, L * (1 + 2 ** -20), L / 2, L / 2 * (1 + 2 ** -20), 1.0, 1e-30, 3e38])
    s = nvfp4.row_exponent(a)
    for ai, si in zip(a, s):
        if ai == 0:
            assert si == 0
            continue
        assert ai <= L * 2.0 ** si and ai > L * 2.0 ** (si - 1)


def test_quantize_roundtrip_error_bound():
    """|deq(Q(v)) - v| <= half an E2M1 gap at the block's scale, plus saturation."""
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 256)) * 30
    c, sc, s = nvfp4.quantize(v)
    d = nvfp4.dequant_q(c, sc, s)
    unit = np.repeat(np.ldexp(nvfp4.UE4M3_TABLE[sc], s[:, None]), 16, axis=1)
    assert np.all(np.abs(d - v) <= 1.0 * unit + 1e-300)
    # scaling a row by a power of two leaves codes and block scales unchanged
    c2, sc2, s2 = nvfp4.quantize(v * 2.0 ** 7)
    assert np.array_equal(c, c2) and np.array_equal(sc, sc2) and np.array_equal(s2, s + 7)


def test_interleaved_block_import_matches_hand_written_fixture(golden_dir):
    """The pages' 36-byte blocks (4 scales + 32 code bytes per 64 weights) become the planar
    code and scale rows written out by hand, and dequantise to the values the block means."""
    rows = {}
    for line in open(os.path.join(golden_dir, "interleaved_block.txt")):
        if line.strip() and not line.startswith("#"):
            f = line.split()
            rows[f[0]] = np.frombuffer(bytes.fromhex("".join(f[1:])), np.uint8)
    assert rows["interleaved"].size == 2 * 36
    codes, scales = nvfp4.from_interleaved(rows["interleaved"], 128)
    assert np.array_equal(codes, rows["codes"])
    assert np.array_equal(scales, rows["scales"])
    w = nvfp4.dequant(codes[None, None, :], scales[None, None, :])[0, 0]
    # block 0: code w%16 times scales 1, 0.5, 0.25, 0.125 per 16 weights
    assert w[0] == 0.0 and w[7] == 6.0 and w[15] == -6.0 and w[17] == 0.25 and w[33] == 0.125 and w[40] == 0.0
    # block 1: even weights 0.5, odd weights 1.0, times 2^-6, 2^-5, 2^-4, 448
    assert w[64] == 0.5 / 64 and w[65] == 1.0 / 64 and w[80] == 0.5 / 32 and w[127] == 448.0
    with pytest.raises(ValueError):
        nvfp4.from_interleaved(rows["interleaved"][:70], 128)


def test_quantize_power_of_two_and_sign_invariance():
    """Q commutes with exact rescaling and negation: Q(2^j v) has v's codes and block scales
    and row exponent s + j (the row scale is a power of two, so every decision is the same
    comparison); Q(-v) flips exactly the sign bit of every code of a nonzero value."""
    rng = np.random.default_rng(17)
    v = rng.standard_normal((6, 64)) * np.exp2(rng.integers(-30, 30, size=(6, 1)))
    v[0, :16] = 0.0                                         # a zero block
    c0, s0, e0 = nvfp4.quantize(v)
    for j in (-40, -3, 1, 7, 60):
        c, s, e = nvfp4.quantize(np.ldexp(v, j))
        assert np.array_equal(c, c0) and np.array_equal(s, s0) and np.array_equal(e, e0 + j)
    cn, sn, en = nvfp4.quantize(-v)
    assert np.array_equal(sn, s0) and np.array_equal(en, e0)
    lo, hi = c0 & 0xF, c0 >> 4
    nlo, nhi = cn & 0xF, cn >> 4
    nz_lo, nz_hi = v[:, 0::2] != 0, v[:, 1::2] != 0
    assert np.array_equal(nlo[nz_lo], lo[nz_lo] ^ 8) and np.array_equal(nhi[nz_hi], hi[nz_hi] ^ 8)
