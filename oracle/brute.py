"""Pure-Python brute force of the routed-MoE FFN for tiny shapes.

TEST INFRASTRUCTURE: used only by the tests to pin the vectorised oracle.

It shares nothing with ``oracle.moe``/``oracle.nvfp4`` except the definitions
it restates independently: NVFP4 values are decoded bit field by bit field with
``fractions.Fraction`` (no table), the gate/up dot products are exact rational
sums, routing is a Python ``sorted`` and grouping is a list of buckets.  Only
SiLU (an exponential) and the down projection run in Python floats.
"""
from __future__ import annotations

import math
from fractions import Fraction


def e2m1(code: int) -> Fraction:
    sign = -1 if code & 0x8 else 1
    exp_field = (code >> 1) & 0x3
    man = code & 0x1
    if exp_field == 0:                       # subnormal: 0 or 0.5
        return sign * Fraction(man, 2)
    return sign * (1 + Fraction(man, 2)) * Fraction(2) ** (exp_field - 1)


def ue4m3(b: int) -> Fraction:
    assert 0 <= b < 0x7F
    exp_field = (b >> 3) & 0xF
    man = b & 0x7
    if exp_field == 0:
        return Fraction(man, 8) * Fraction(1, 64)
    return (1 + Fraction(man, 8)) * Fraction(2) ** (exp_field - 7)


def bf16(bits: int) -> Fraction:
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(m, 128) * Fraction(2) ** -126
    return sign * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def weight(codes_row, scales_row, c: int) -> Fraction:
    byte = int(codes_row[c // 2])
    nib = (byte >> 4) if (c % 2) else (byte & 0xF)
    return e2m1(nib) * ue4m3(int(scales_row[c // 16]))


def route(logits_row, k: int):
    E = len(logits_row)
    order = sorted(range(E), key=lambda e: (-float(logits_row[e]), e))[:k]
    sel = [float(logits_row[e]) for e in order]
    m = sel[0]
    ex = [math.exp(v - m) for v in sel]
    tot = sum(ex)
    return order, [v / tot for v in ex]


def moe_ffn(x_bits, logits, gate_up, down, k: int, ids=None, w=None):
    """y[t][r] as Python floats for a tiny workload (decode semantics)."""
    T = len(x_bits)
    H = len(x_bits[0])
    E = gate_up.codes.shape[0]
    F = gate_up.codes.shape[1] // 2
    if ids is None:
        ids, w = [], []
        for t in range(T):
            o, ww = route(logits[t], k)
            ids.append(o)
            w.append(ww)
    buckets = [[] for _ in range(E)]
    for p in range(T * k):
        buckets[int(ids[p // k][p % k])].append(p)
    z = {}
    for e in range(E):
        for p in buckets[e]:
            t = p // k
            a = [bf16(int(b)) for b in x_bits[t]]
            h = []
            for i in range(F):
                g = sum(weight(gate_up.codes[e][i], gate_up.scales[e][i], c) * a[c] for c in range(H))
                u = sum(weight(gate_up.codes[e][F + i], gate_up.scales[e][F + i], c) * a[c]
                        for c in range(H))
                gf, uf = float(g), float(u)
                h.append(gf / (1.0 + math.exp(-gf)) * uf)
            zr = []
            for r in range(H):
                acc = 0.0
                for i in range(F):
                    acc += float(weight(down.codes[e][r], down.scales[e][r], i)) * h[i]
                zr.append(acc)
            z[p] = zr
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            zr = z[t * k + j]
            wj = float(w[t][j])
            for r in range(H):
                y[t][r] += wj * zr[r]
    return ids, w, y
