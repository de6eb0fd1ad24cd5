"""GPU parity of the prefill path (Q(x) -> tcgen05 block-scaled gate/up -> Q(h) ->
tcgen05 down -> combine) against the CPU oracle, stage by stage, through the C ABI.

Stages: (i) Q(x) is bit-exact; (ii) h is within the accumulation tolerance of the
oracle's h from the same Q(x), and within the float32 accumulation band the oracle
models (oracle.h_band); (iii) Q(h) equals the oracle's Q applied to the GPU's own h, bit
for bit (both take every decision on the same float32 values), and equals the oracle's
Q of its own h wherever that decision is outside the band (the flagged share is bounded);
(iv) y equals the oracle's down projection and combine of the GPU's Q(h) within
2e-3 * sum|w * terms| + 1e-5, and, fed the oracle's own h, the GPU reproduces Q(h) bit for
bit and y within the same bound; (v) end to end, y is within that bound plus the
allowance of the flagged Q(h) decisions (the share inside the plain bound is reported and
bounded).
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


# Largest share of Q(h) elements whose value-changing decision may lie within the band
# (0.1%), or four blocks' worth of elements in small samples, where one ambiguous block
# scale alone flags its 16 elements.
FLAG_CEILING = 1e-3
FLAG_FLOOR_ELEMENTS = 64
# Smallest share of y elements within the plain end-to-end bound (no allowance).
PLAIN_SHARE_FLOOR = 0.999


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
    h32 = run.region("h", P * F * 4, np.float32, (P, F))[pos]
    h_gpu = h32.astype(np.float64)
    assert_within(h_gpu, res.h[pairs], h_tolerance(res)[pairs], "h")
    amb = oracle.qh_ambiguity(res, pairs)
    ratio = np.abs(h_gpu - res.h[pairs]) / amb.band[pairs]
    band_ratio = float(np.max(ratio))
    print(f"h error / band: max {band_ratio:.3g} p99 {np.percentile(ratio, 99):.3g} "
          f"median {np.median(ratio):.3g}")
    assert band_ratio <= 1.0, f"h error exceeds the accumulation band by {band_ratio:.3g}x"
    # (iii) Q(h): against the oracle's Q of the GPU's own h, everywhere ...
    q_packed = run.region("qh_codes", P * F // 2, np.uint8, (P, F // 2))[pos]
    S = qh_scale_pitch(F)
    q_s = run.region("qh_scales", P * S, np.uint8, (P, S))[pos, :F // 16]
    q_e = run.region("qh_exp", P * 4, np.int32, (P,))[pos]
    own_c, own_s, own_e = nvfp4.quantize(h_gpu)
    assert np.array_equal(q_packed, own_c), "Q(h) codes vs the oracle's Q of the GPU's h"
    assert np.array_equal(q_s, own_s), "Q(h) scales vs the oracle's Q of the GPU's h"
    assert np.array_equal(q_e, own_e), "Q(h) exponents vs the oracle's Q of the GPU's h"
    # ... and against the oracle's Q of its own h outside the band
    q_c = _unpack(q_packed)
    r_c = _unpack(res.qh[0][pairs])
    flagged = amb.flagged[pairs]
    zsign = amb.zero_sign[pairs]
    exact = ~flagged & ~zsign
    assert np.array_equal(q_c[exact], r_c[exact]), "Q(h) codes outside the band"
    assert np.array_equal(q_c[zsign] & 7, r_c[zsign] & 7), "Q(h) zero codes (magnitude)"
    blk_flag = flagged.reshape(len(pairs), F // 16, 16).any(axis=2)
    assert np.array_equal(q_s[~blk_flag], res.qh[1][pairs][~blk_flag]), "Q(h) block scales"
    row_flag = flagged.all(axis=1)
    assert np.array_equal(q_e[~row_flag], res.qh[2][pairs][~row_flag]), "Q(h) row exponents"
    flagged_frac = float(flagged.mean())
    print(f"flagged Q(h) share {flagged_frac:.3g} ({int(flagged.sum())} of {flagged.size}), "
          f"sign-only zero codes {float(zsign.mean()):.3g}")
    assert flagged.sum() <= max(FLAG_CEILING * flagged.size, FLAG_FLOOR_ELEMENTS), \
        f"flagged Q(h) share {flagged_frac:.3g}"
    # (iv) y from the GPU's own Q(h): the oracle's down projection and combine of it
    hq = np.zeros((P, F))
    hq[pairs] = nvfp4.dequant_q(q_packed, q_s, q_e.astype(np.int64))
    y4, tsum4 = oracle.down_combine(hq, ids, w, wl.down, toks)
    assert_within(run.y[toks], y4[toks], oracle.tolerance(tsum4)[toks], "y from the GPU's Q(h)")
    # (v) end to end
    plain = oracle.tolerance(res.tsum)[toks]
    extra = oracle.prefill_allowance(res, amb, wl.down, ids, w, toks)[toks]
    worst = assert_within(run.y[toks], res.y[toks], plain + extra, "y")
    share = float(np.mean(np.abs(run.y[toks] - res.y[toks]) <= plain))
    print(f"y end to end: worst err/tol {worst:.3g}; share within the plain bound {share:.6f}; "
          f"allowance/plain tolerance max {float(np.max(extra / plain)):.3g}")
    assert share >= PLAIN_SHARE_FLOOR, f"only {share:.6f} of y within the plain bound"
    return res, {"flagged_frac": flagged_frac, "band_ratio": band_ratio, "y_worst": worst,
                 "plain_share": share}


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


@pytest.mark.parametrize("F", [768, 832, 1152])
def test_prefill_ff_widths(F):
    """The down GEMM's forms across F: the Q(h) tile held in shared memory for up to three
    k-stages (F = 768, all three full) and re-read every stage beyond that (F = 832 with a
    half-empty last stage, F = 1152); two M-tiles per expert, every token checked."""
    wl = synth.logits_workload(f"prefill_F{F}", 256, 512, F, 4, 4, seed=5)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    toks = np.arange(wl.T)
    res, info = _stages(wl, run, toks)
    _down_from_oracle_h(wl, run, res, toks)


def test_prefill_largest_ff_and_hidden():
    """The prefill path at its largest F and H (F = H = 4096): Q(h) of 256 blocks per row
    and the general down GEMM over 16 k-stages; every token checked."""
    wl = synth.logits_workload("prefill_F4096", 32, 4096, 4096, 16, 4, seed=29)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    toks = np.arange(wl.T)
    res, info = _stages(wl, run, toks)
    _down_from_oracle_h(wl, run, res, toks)


def test_prefill_per_expert_alpha():
    """Prefill with a per-expert second-level scale alpha on both banks (down's <= 2)."""
    wl = synth.prefill(seed=3, T=256)
    rng = np.random.default_rng(13)
    wl.gate_up.alpha = rng.uniform(0.25, 1.75, size=wl.E).astype(np.float32)
    wl.down.alpha = rng.uniform(0.25, 1.75, size=wl.E).astype(np.float32)
    run = run_layer(wl, path=PF)
    assert run.err == 0
    _stages(wl, run, np.arange(0, 256, 41))


def _tile_probe_tokens(ids, E, k, hottest=3, ragged=24, extra=24, seed=0):
    """Tokens whose pairs land on chosen rows of the 128-row M-tiles: the first and last row
    of every tile of the `hottest` experts, the last row of the last (ragged) tile of
    `ragged` more experts, plus `extra` random tokens."""
    csr = oracle.build_expert_csr(ids, E)
    counts = np.diff(csr.offsets.astype(np.int64))
    order = np.argsort(-counts, kind="stable")
    rows = []
    for e in order[:hottest]:
        off, m = int(csr.offsets[e]), int(counts[e])
        for t0 in range(0, m, 128):
            rows += [off + t0, off + min(t0 + 127, m - 1)]
    rag = [e for e in order[hottest:] if counts[e] % 128 not in (0, 1)][:ragged]
    rows += [int(csr.offsets[e + 1]) - 1 for e in rag]
    toks = set(int(csr.pair_ids[r]) // k for r in rows)
    rng = np.random.default_rng(seed)
    toks |= set(rng.choice(ids.shape[0], size=extra, replace=False).tolist())
    while len(toks) < 64:
        toks.add(int(rng.integers(ids.shape[0])))
    return np.array(sorted(toks)), rows, rag


def test_prefill_full_size_sampled():
    """The prefill workload at full size (4096 tokens, 32768 pairs, 288 experts): checked
    rows in every M-tile of the three hottest experts (first and last row of each) and in
    the last, ragged tile of 24 more experts."""
    wl = synth.prefill()
    run = run_layer(wl, path=PF)
    assert run.err == 0
    from test_gpu_decode import _check_csr
    _check_csr(run, wl.ids, wl.E)
    toks, rows, rag = _tile_probe_tokens(wl.ids, wl.E, wl.k)
    assert len(toks) >= 64 and len(rag) >= 20
    hot_tiles = sum((int(c) + 127) // 128 for c in np.sort(np.bincount(wl.ids.reshape(-1), minlength=wl.E))[-3:])
    assert hot_tiles >= 9                       # the hottest experts span several M-tiles
    res, info = _stages(wl, run, toks)
    _down_from_oracle_h(wl, run, res, toks)


def test_prefill_invalid_ids_and_empty_tokens():
    """Out-of-range expert ids on the prefill path: the pairs are skipped and flagged, a
    token with some invalid pairs combines the rest, and a token with none valid gets a
    zero row (no pair arrives to write it)."""
    wl = synth.prefill(seed=4, T=256)
    ids = wl.ids.copy()
    ids[3, :] = wl.E + 1                     # every pair of token 3 invalid
    ids[10, 2] = -1
    ids[77, 0] = wl.E
    ids[200, 5:] = -7
    bad = synth.Workload("prefill_bad", wl.T, wl.H, wl.F, wl.E, wl.k, wl.x_bits, wl.gate_up,
                         wl.down, ids=ids, weights=wl.weights)
    gu, dn = device_banks(bad)
    layer = moe.MoeLayer(gu, dn, bad.k)
    b = layer.buffers(bad.T, PF)
    b["y"].fill_(7.0)                       # stale values where the row must become zero
    run = run_layer(bad, path=PF, layer=layer)
    assert run.err & moe.DEVERR_EXPERT_ID
    assert np.all(run.y[3] == 0.0)
    _stages(bad, run, np.array([3, 10, 77, 200, 201]))


def test_prefill_replays_bit_identical():
    wl = synth.prefill(T=512)
    gu, dn = device_banks(wl)
    layer = moe.MoeLayer(gu, dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.from_numpy(wl.ids).cuda()
    w = torch.from_numpy(wl.weights).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, ids=ids, w=w, path=PF, stream=s)     # allocate buffers, warm up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        y = layer.forward(x, ids=ids, w=w, path=PF, stream=s)
    hashes = set()
    for _ in range(10):
        g.replay()
        torch.cuda.synchronize()
        hashes.add(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
    assert len(hashes) == 1
    y2 = layer.forward(x, ids=ids, w=w, path=PF).cpu().numpy()
    assert hashlib.sha256(y2.tobytes()).hexdigest() in hashes


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
