"""GPU parity of the prefill path (Q(x) -> tcgen05 block-scaled gate/up -> Q(h) ->
tcgen05 down -> combine) against the CPU oracle, stage by stage, through the C ABI.

Stages: (i) Q(x) is bit-exact; (ii) h is within the accumulation tolerance of the
oracle's h from the same Q(x) and within the quantisation band the oracle assumes;
(iii) Q(h) is bit-exact wherever the oracle's decision is not within that band;
(iv) the down projection and combine, fed the oracle's own h, match the oracle within
2e-3 * sum|w * terms| + 1e-5 and reproduce Q(h) bit-exactly; (v) end to end, y is within
that tolerance plus the allowance of the flagged Q(h) decisions.
"""
import hashlib

import numpy as np
import pytest
import torch

import synth
import oracle
from oracle import nvfp4
import nvfp4_grouped_gemm_gb300 as moe
from gpu_util import run_layer, h_tolerance, assert_within, device_banks, qh_scale_pitch

pytestmark = pytest.mark.gpu
PF = moe.PATH_PREFILL


def _unpack(packed):
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def _routing(wl):
    if wl.logits is not None:
        return oracle.route_topk(wl.logits, wl.k)
    return wl.ids, wl.weights.astype(np.float64)


def _stages(wl, run, tokens):
    ids, w = _routing(wl)
    P, H, F, k = wl.P, wl.H, wl.F, wl.k
    toks = np.asarray(tokens)
    pairs = (toks[:, None] * k + np.arange(k)).reshape(-1)
    pairs = pairs[run.pair_pos[pairs] >= 0]
    pos = run.pair_pos[pairs]
    # (i) Q(x), bit-exact, for every token (cheap) at its CSR rows
    x = nvfp4.bf16_to_f64(wl.x_bits)
    cx, sx, ex = nvfp4.quantize(x)
    g_c = run.region("qx_codes", P * H // 2, np.uint8, (P, H // 2))
    g_s = run.region("qx_scales", P * H // 16, np.uint8, (P, H // 16))
    g_e = run.region("qx_exp", P * 4, np.int32, (P,))
    allp = np.nonzero(run.pair_pos >= 0)[0]
    allpos = run.pair_pos[allp]
    assert np.array_equal(g_c[allpos], cx[allp // k]), "Q(x) codes"
    assert np.array_equal(g_s[allpos], sx[allp // k]), "Q(x) scales"
    assert np.array_equal(g_e[allpos], ex[allp // k]), "Q(x) row exponents"
    # oracle in prefill mode on the sampled tokens
    res = oracle.ffn(wl.x_bits, ids, w, wl.gate_up, wl.down, mode="prefill", tokens=toks)
    # (ii) h
    h_gpu = run.region("h", P * F * 4, np.float32, (P, F))[pos].astype(np.float64)
    assert_within(h_gpu, res.h[pairs], h_tolerance(res)[pairs], "h")
    amb = oracle.qh_ambiguity(res, pairs)
    ratio = np.abs(h_gpu - res.h[pairs]) / amb.band[pairs]
    band_ratio = float(np.max(ratio))
    gscale = res.g_abs[pairs]
    print(f"h error / band: max {band_ratio:.3g} p99 {np.percentile(ratio, 99):.3g} "
          f"median {np.median(ratio):.3g}; |h_gpu-h|/|h| max "
          f"{np.max(np.abs(h_gpu - res.h[pairs]) / (np.abs(res.h[pairs]) + 1e-30)):.3g}")
    assert band_ratio <= 1.0, f"h error exceeds the quantisation band by {band_ratio:.3g}x"
    # (iii) Q(h) where the decision is not ambiguous
    q_c = _unpack(run.region("qh_codes", P * F // 2, np.uint8, (P, F // 2))[pos])
    S = qh_scale_pitch(F)
    q_s = run.region("qh_scales", P * S, np.uint8, (P, S))[pos, :F // 16]
    q_e = run.region("qh_exp", P * 4, np.int32, (P,))[pos]
    r_c = _unpack(res.qh[0][pairs])
    flagged = amb.flagged[pairs]
    assert np.array_equal(q_c[~flagged], r_c[~flagged]), "Q(h) codes outside the band"
    blk_flag = flagged.reshape(len(pairs), F // 16, 16).any(axis=2)
    assert np.array_equal(q_s[~blk_flag], res.qh[1][pairs][~blk_flag]), "Q(h) block scales"
    row_flag = flagged.all(axis=1)
    assert np.array_equal(q_e[~row_flag], res.qh[2][pairs][~row_flag]), "Q(h) row exponents"
    # (v) end to end
    extra = oracle.prefill_allowance(res, amb, wl.down, ids, w, toks)
    worst = assert_within(run.y[toks], res.y[toks], oracle.tolerance(res.tsum, extra)[toks], "y")
    return res, {"flagged_frac": float(flagged.mean()), "band_ratio": float(band_ratio),
                 "y_worst": worst}


def _down_from_oracle_h(wl, run, res, tokens):
    """(iv): overwrite the workspace's h with the oracle's h, rerun down+combine."""
    layer = run.layer
    b = layer.buffers(wl.T, PF)
    ws = b["ws"]
    P, F, H, k = wl.P, wl.F, wl.H, wl.k
    toks = np.asarray(tokens)
    pairs = (toks[:, None] * k + np.arange(k)).reshape(-1)
    pairs = pairs[run.pair_pos[pairs] >= 0]
    pos = run.pair_pos[pairs]
    h_all = run.region("h", P * F * 4, np.float32, (P, F)).copy()
    h_all[pos] = res.h[pairs].astype(np.float32)
    off = run.ws["h"]
    ws[off:off + P * F * 4].copy_(torch.from_numpy(h_all.view(np.uint8).reshape(-1)).cuda())
    ids, w = _routing(wl)
    w_t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    y = torch.zeros(wl.T, H, dtype=torch.float32, device="cuda")
    moe.moe_grouped_down_combine_nvfp4(layer.down, b["csr"], w_t, wl.T, H, F, k, y, ws, PF)
    torch.cuda.synchronize()
    wsn = ws.cpu().numpy()
    L = run.ws
    q_c = wsn[L["qh_codes"]:L["qh_codes"] + P * F // 2].reshape(P, F // 2)[pos]
    S = qh_scale_pitch(F)
    q_s = wsn[L["qh_scales"]:L["qh_scales"] + P * S].reshape(P, S)[pos, :F // 16]
    assert np.array_equal(q_c, res.qh[0][pairs]), "Q(oracle h) codes"
    assert np.array_equal(q_s, res.qh[1][pairs]), "Q(oracle h) scales"
    yy = y.cpu().numpy()
    return assert_within(yy[toks], res.y[toks], oracle.tolerance(res.tsum)[toks], "y from oracle h")


def test_tiny_prefill():
    wl = synth.tiny()
    run = run_layer(wl, path=PF)
    assert run.err == 0
    res, info = _stages(wl, run, np.arange(wl.T))
    _down_from_oracle_h(wl, run, res, np.arange(wl.T))


@pytest.mark.parametrize("seed", [0, 1])
def test_prefill_small(seed):
    wl = synth.prefill(seed=seed, T=256)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    from test_gpu_decode import _check_csr
    _check_csr(run, wl.ids, wl.E)
    toks = np.arange(0, 256, 37)
    res, info = _stages(wl, run, toks)
    _down_from_oracle_h(wl, run, res, toks)


@pytest.mark.parametrize("T", [1, 8])
def test_prefill_numerics_at_decode_sizes(T):
    """The PREFILL path (NVFP4 x and h, FP4 x FP4 tensor-core GEMMs) chosen explicitly at
    decode batch sizes: one T sweep can keep the prefill semantics across the AUTO switch,
    checked stage by stage like the large cases."""
    wl = synth.decode(T)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    res, info = _stages(wl, run, np.arange(T))


def test_prefill_per_expert_alpha():
    """Prefill with a per-expert second-level scale alpha on both banks (down's <= 2)."""
    wl = synth.prefill(seed=3, T=256)
    rng = np.random.default_rng(13)
    wl.gate_up.alpha = rng.uniform(0.25, 1.75, size=wl.E).astype(np.float32)
    wl.down.alpha = rng.uniform(0.25, 1.75, size=wl.E).astype(np.float32)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    _stages(wl, run, np.arange(0, 256, 41))


def test_prefill_full_size_sampled():
    """The prefill workload at full size (4096 tokens, 32768 pairs, 288 experts)."""
    wl = synth.prefill()
    run = run_layer(wl, path=PF)
    assert run.err == 0
    from test_gpu_decode import _check_csr
    _check_csr(run, wl.ids, wl.E)
    toks = np.array([0, 1, 777, 2048, 4095])
    res, info = _stages(wl, run, toks)
    _down_from_oracle_h(wl, run, res, toks)


def test_prefill_replays_bit_identical():
    wl = synth.prefill(T=512)
    gu, dn = device_banks(wl)
    layer = moe.MoeLayer(gu, dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(wl.ids).cuda()
    w = torch.from_numpy(wl.weights).cuda()
    hashes = set()
    for _ in range(5):
        y = layer.forward(x, ids=ids, w=w, path=PF)
        torch.cuda.synchronize()
        hashes.add(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
    assert len(hashes) == 1


def test_auto_path_switch():
    th = moe.prefill_min_pairs()
    assert moe.resolve_path(th // 8, 8) == moe.PATH_PREFILL
    assert moe.resolve_path(th // 8 - 1, 8) == moe.PATH_DECODE


def _crafted_rows(H):
    """Activation rows that sit exactly on Q's decision boundaries."""
    rows = []
    # block 0 sets sb = 448 at s = 0 (amax 2688); the rest hit every E2M1 midpoint exactly
    r = np.zeros(H)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]) * 448
    r[0] = 2688.0
    r[1:8] = mids
    r[8:15] = -mids
    r[15] = -0.0
    # block 1: amax exactly on UE4M3 thresholds 3 * (v(j) + v(j+1)) for a few j
    r[16] = 3.0 * (0.5 + 0.5625)          # between 0x30 and 0x31
    r[17:32] = 0.1
    r[32] = 3.0 * (0.015625 + 0.017578125)  # between 0x08 and 0x09
    r[48] = 3.0 * (0.001953125 * 1 + 0.001953125 * 2)   # subnormal encodings 1 and 2
    r[64:80] = 1e-30                        # far below the row scale: zero block scale
    r[80:96] = -7.5e3                        # saturates against the row exponent
    rows.append(r)
    rows.append(np.zeros(H))                # all-zero row
    rng = np.random.default_rng(5)
    rows.append(rng.standard_normal(H) * 2.0 ** 40)
    rows.append(rng.standard_normal(H) * 2.0 ** -40)
    bits = synth.f32_to_bf16_bits(np.stack(rows).astype(np.float32))
    return bits


def test_quantiser_decision_boundaries():
    base = synth.tiny(seed=2)
    x_bits = _crafted_rows(base.H)
    wl = synth.Workload("edges", 4, base.H, base.F, base.E, base.k, x_bits, base.gate_up,
                        base.down, ids=np.array([[0, 1], [2, 3], [4, 5], [6, 7]], np.int32),
                        weights=np.full((4, 2), 0.5, np.float32))
    run = run_layer(wl, path=PF)
    x = nvfp4.bf16_to_f64(x_bits)
    cx, sx, ex = nvfp4.quantize(x)
    P, H, k = wl.P, wl.H, wl.k
    g_c = run.region("qx_codes", P * H // 2, np.uint8, (P, H // 2))
    g_s = run.region("qx_scales", P * H // 16, np.uint8, (P, H // 16))
    g_e = run.region("qx_exp", P * 4, np.int32, (P,))
    p = np.arange(P)
    assert np.array_equal(g_e[run.pair_pos[p]], ex[p // k])
    assert np.array_equal(g_s[run.pair_pos[p]], sx[p // k])
    assert np.array_equal(g_c[run.pair_pos[p]], cx[p // k])
