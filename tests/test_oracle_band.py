"""Pins for the prefill quantisation band (oracle.h_band, oracle.qh_ambiguity), CPU only.

The band bounds how far a device float32 h = silu(g) * u can sit from the oracle's float64
value when g and u come from a tensor-core accumulation in 64-element K-steps.  It is
pinned here against a float32 emulation of that accumulation, written independently of the
band's formula: each step's exact sum of products added into a float32 accumulator (round
to nearest), and a harsher variant whose step sums are first truncated to float32; the
epilogue (SiLU, product) then runs in numpy float32.  The emulated h must stay inside the
band with a factor-of-two margin, and each term of the band must be needed: without the
accumulation term the emulation leaves it, and without the underflow floor a row whose
float32 SiLU underflows (g < -88.7) leaves it.
"""
import numpy as np
import pytest

import synth
import oracle
from oracle import nvfp4


def _rz32(x):
    """Round float64 values to float32 toward zero."""
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f[over] = np.nextafter(f[over], np.float32(0))
    return f


def _emulate_h(a, wgu, F, variant):
    """Device-style float32 h for one activation row a [K] against gate/up rows wgu [2F, K]."""
    K = a.shape[0]
    S = (a[None, :] * wgu).reshape(2 * F, K // 64, 64).sum(axis=2)   # exact step sums
    acc = np.zeros(2 * F, np.float32)
    for j in range(K // 64):
        s = S[:, j] if variant == "rn" else _rz32(S[:, j]).astype(np.float64)
        acc = (acc.astype(np.float64) + s).astype(np.float32)
    g32, u32 = acc[:F], acc[F:]
    with np.errstate(over="ignore"):
        silu32 = g32 / (np.float32(1) + np.exp(-g32))
    return (silu32 * u32).astype(np.float64)


def _emulated_ratios(wl, tokens, band):
    ids = wl.ids
    k, F = wl.k, wl.F
    res = oracle.ffn(wl.x_bits, ids, wl.weights.astype(np.float64), wl.gate_up, wl.down,
                     mode="prefill", tokens=tokens)
    x = nvfp4.bf16_to_f64(wl.x_bits)
    out = {"rn": [], "rz": []}
    for t in tokens:
        a = nvfp4.dequant_q(*nvfp4.quantize(x[t]))
        for j in range(k):
            p = t * k + j
            wgu = nvfp4.dequant(wl.gate_up.codes[ids[t, j]], wl.gate_up.scales[ids[t, j]])
            for variant in out:
                h32 = _emulate_h(a, wgu, F, variant)
                out[variant].append(np.abs(h32 - res.h[p]) / band(res)[p])
    return {v: np.concatenate(r) for v, r in out.items()}


@pytest.mark.parametrize("H", [256, 2560, 4096])
def test_band_covers_float32_accumulation(H):
    wl = synth.prefill(seed=H, T=4, H=H, F=128, E=8, k=2)
    r = _emulated_ratios(wl, np.arange(wl.T), oracle.h_band)
    for variant, ratio in r.items():
        assert ratio.max() <= 0.5, f"{variant}: emulated h leaves half the band ({ratio.max():.3g})"


def _cancelling_workload():
    """One token (all ones), one expert whose gate row 0 runs four K-steps of 64: weights
    6 * 448, then 0.5 * 2^-9, then -6 * 448, then 0.  The float32 running sum after the
    second step (about 177408) cannot hold the small step's sum (0.0645) exactly, and the
    third step cancels the large part: g = 0.064453125 exactly, 0.0625 in float32.
    Up row 0 is 1.0 * 2^-6 everywhere (u = 4.125)."""
    base = synth.prefill(seed=5, T=1, H=256, F=64, E=2, k=1)
    x_bits = synth.f32_to_bf16_bits(np.ones((1, 256), np.float32))
    gu = synth.Bank(base.gate_up.codes.copy(), base.gate_up.scales.copy())
    gu.codes[0, 0, 0:32], gu.scales[0, 0, 0:4] = 0x77, 0x7E      # +6 x 448
    gu.codes[0, 0, 32:64], gu.scales[0, 0, 4:8] = 0x11, 0x01     # +0.5 x 2^-9
    gu.codes[0, 0, 64:96], gu.scales[0, 0, 8:12] = 0xFF, 0x7E    # -6 x 448
    gu.codes[0, 0, 96:128], gu.scales[0, 0, 12:16] = 0x00, 0x08  # 0
    gu.codes[0, 64, :], gu.scales[0, 64, :] = 0x22, 0x08         # up row: 1.0 x 2^-6
    return synth.Workload("cancel", 1, 256, 64, 2, 1, x_bits, gu, base.down,
                          ids=np.zeros((1, 1), np.int32), weights=np.ones((1, 1), np.float32))


def test_accumulation_term_is_needed_and_enough():
    """A row whose float32 running sum loses a small step to a large one: the accumulation
    term of the band covers the error, and without it the band does not."""
    wl = _cancelling_workload()
    res = oracle.ffn(wl.x_bits, wl.ids, wl.weights.astype(np.float64), wl.gate_up, wl.down,
                     mode="prefill")
    assert res.g[0, 0] == 0.064453125 and res.u[0, 0] == 4.125
    x = nvfp4.bf16_to_f64(wl.x_bits)
    a = nvfp4.dequant_q(*nvfp4.quantize(x[0]))
    wgu = nvfp4.dequant(wl.gate_up.codes[0], wl.gate_up.scales[0])
    h32 = _emulate_h(a, wgu, wl.F, "rn")
    err = abs(h32[0] - res.h[0, 0])
    assert err > 1e-3 * abs(res.h[0, 0])                 # the float32 sum really is off
    assert err <= 0.5 * oracle.h_band(res)[0, 0]                       # enough
    assert err > oracle.h_band(res, widen=0.0)[0, 0]                   # needed


def _underflow_workload():
    """One token, one expert: gate row 0 gives g = -99 (float32 SiLU underflows to -0),
    up row 0 gives u = 4.125; the other rows are random."""
    base = synth.prefill(seed=7, T=1, H=256, F=64, E=2, k=1)
    x_bits = synth.f32_to_bf16_bits(np.ones((1, 256), np.float32))
    gu = synth.Bank(base.gate_up.codes.copy(), base.gate_up.scales.copy())
    gu.codes[0, 0, :] = 0x99            # every weight -0.5 (E2M1 code 9)
    gu.scales[0, 0, :] = 0x34           # UE4M3 0.75
    gu.codes[0, 64, :] = 0x22           # every weight 1.0 (E2M1 code 2)
    gu.scales[0, 64, :] = 0x08          # UE4M3 2^-6
    return synth.Workload("underflow", 1, 256, 64, 2, 1, x_bits, gu, base.down,
                          ids=np.zeros((1, 1), np.int32), weights=np.ones((1, 1), np.float32))


def test_underflow_floor_is_needed_and_enough():
    wl = _underflow_workload()
    res = oracle.ffn(wl.x_bits, wl.ids, wl.weights.astype(np.float64), wl.gate_up, wl.down,
                     mode="prefill")
    assert res.g[0, 0] == -99.0 and res.u[0, 0] == 4.125
    x = nvfp4.bf16_to_f64(wl.x_bits)
    a = nvfp4.dequant_q(*nvfp4.quantize(x[0]))
    wgu = nvfp4.dequant(wl.gate_up.codes[0], wl.gate_up.scales[0])
    h32 = _emulate_h(a, wgu, wl.F, "rn")
    assert h32[0] == 0.0 and res.h[0, 0] != 0.0          # float32 SiLU underflow
    err = abs(h32[0] - res.h[0, 0])
    band = oracle.h_band(res)[0, 0]
    floor = 2.0 ** -120 * abs(res.u[0, 0]) + 2.0 ** -140
    assert err <= band                                   # enough
    assert err > band - floor                            # needed
    # the element is a zero code whose sign the band leaves open, not a value flip
    amb = oracle.qh_ambiguity(res, np.array([0]))
    assert amb.zero_sign[0, 0] and not amb.flagged[0, 0]


def test_flagged_share_is_small_on_prefill_data():
    """On prefill-shaped data almost no Q(h) decision changes value inside the band."""
    wl = synth.prefill(seed=2, T=64)
    toks = np.arange(0, 64, 8)
    res = oracle.ffn(wl.x_bits, wl.ids, wl.weights.astype(np.float64), wl.gate_up, wl.down,
                     mode="prefill", tokens=toks)
    pairs = (toks[:, None] * wl.k + np.arange(wl.k)).reshape(-1)
    amb = oracle.qh_ambiguity(res, pairs)
    assert amb.flagged[pairs].mean() < 1e-3
    # the allowance only widens the rows of tokens with a flagged element
    extra = oracle.prefill_allowance(res, amb, wl.down, wl.ids, wl.weights, toks)
    widened = np.nonzero(extra[toks].max(axis=1) > 0)[0]
    has_flag = np.nonzero(amb.flagged[pairs].reshape(len(toks), -1).any(axis=1))[0]
    assert np.array_equal(widened, has_flag) and len(has_flag) < len(toks)


def test_down_combine_equals_the_ffn_steps():
    """The oracle's standalone down projection and combine, given the h the FFN fed to its
    down projection, reproduce the FFN's y and tolerance scale."""
    wl = synth.tiny(seed=6)
    ids, w = oracle.route_topk(wl.logits, wl.k)
    for mode in ("decode", "prefill"):
        res = oracle.ffn(wl.x_bits, ids, w, wl.gate_up, wl.down, mode=mode)
        y, tsum = oracle.down_combine(res.h_used, ids, w, wl.down, np.arange(wl.T))
        assert np.allclose(y, res.y, rtol=1e-12, atol=1e-12)
        assert np.allclose(tsum, res.tsum, rtol=1e-12, atol=0)
