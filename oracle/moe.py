"""The routed-MoE FFN, written out plainly in float64 (CPU oracle).

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline may import this package; the product path never does.

Steps, in the order the pages run them:

1. ``route_topk``  -- per token, the k largest router logits (ties to the lower
   expert id), weights = softmax over the selected logits (equal to the full
   softmax renormalised over the selection).  The pages' probes start from
   already-routed pairs; this is the router that produces them.
2. ``build_expert_csr`` -- pairs p = t*k + j bucketed by expert in ascending p
   ("moe_sk_repro.rs", fn main: buckets, ex_ids, ex_off, ex_pairs); the token of
   a pair is p / k (csr_tok there).
3. ``ffn`` -- per pair (t, j) with expert e: g = W_gate[e] a, u = W_up[e] a,
   h = silu(g) * u, z = W_down[e] h ("moe_union_probe.rs": fused gate_up bank
   [E, 2*ff, hidden], gate rows first, down bank [E, hidden, ff]; "moe_sk_repro.rs":
   three grouped projections per layer), then the routing-weighted combine
   y[t] = sum_j w[t, j] * z[t*k + j] in j order.

``mode='decode'`` uses the exact bf16 activations and float64 h; ``mode='prefill'``
quantises x and h with Q (oracle.nvfp4.quantize) before their projections, h
being rounded to float32 first because that is the precision the quantiser
sees on the device.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from . import nvfp4

TOL_REL = 2e-3
TOL_ABS = 1e-5


# ---------------------------------------------------------------------------
# 1. routing
# ---------------------------------------------------------------------------

def route_topk(logits: np.ndarray, k: int):
    """Top-k experts per token by logit (descending, ties to the lower id) and their weights.

    Returns ids int32 [T, k] in (logit desc, id asc) order and w float64 [T, k]
    = softmax over the k selected logits.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    expert = np.arange(E)
    for t in range(T):
        l = logits[t].astype(np.float64)
        order = np.lexsort((expert, -l))        # primary: logit descending; then id ascending
        sel = order[:k]
        ids[t] = sel
        ex = np.exp(l[sel] - l[sel[0]])
        w[t] = ex / ex.sum()
    return ids, w


# ---------------------------------------------------------------------------
# 2. expert-first CSR
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class CSR:
    counts: np.ndarray          # int64 [E]
    offsets: np.ndarray         # int32 [E+1]
    pair_ids: np.ndarray        # int32 [n_valid] pairs ordered by (expert, p)
    active: np.ndarray          # int32 [n_active] experts with at least one pair, ascending
    n_active: int
    pair_pos: np.ndarray        # int32 [P] CSR position of each pair, -1 if its id is invalid


def build_expert_csr(ids: np.ndarray, E: int) -> CSR:
    """Counting sort of the P = T*k pairs by expert, stable in the pair index p."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    P = flat.shape[0]
    valid = (flat >= 0) & (flat < E)
    counts = np.zeros(E, dtype=np.int64)
    for e in flat[valid]:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    pair_ids = np.empty(int(offsets[-1]), dtype=np.int32)
    pair_pos = np.full(P, -1, dtype=np.int32)
    for p in range(P):                         # ascending p: stable placement
        if valid[p]:
            e = flat[p]
            pair_ids[cursor[e]] = p
            pair_pos[p] = cursor[e]
            cursor[e] += 1
    active = np.nonzero(counts)[0].astype(np.int32)
    return CSR(counts, offsets.astype(np.int32), pair_ids, active, int(active.shape[0]), pair_pos)


# ---------------------------------------------------------------------------
# 3. the FFN
# ---------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


@dataclasses.dataclass
class FFNResult:
    y: np.ndarray               # float64 [T, H]
    tsum: np.ndarray            # float64 [T, H]  sum_j |w| * sum_i |D h|  (tolerance scale)
    z: np.ndarray               # float64 [P, H]  per-pair down projections (pair order)
    s_abs: np.ndarray           # float64 [P, H]  sum_i |D[r, i] h_i| per pair
    h: np.ndarray               # float64 [P, F]  h per pair (pair order), before any Q
    g: np.ndarray               # float64 [P, F]
    u: np.ndarray               # float64 [P, F]
    g_abs: np.ndarray           # float64 [P, F]  sum_c |Wg a| (accumulation scale)
    u_abs: np.ndarray           # float64 [P, F]
    qx: Optional[tuple] = None  # prefill: Q(x) per token (codes, scales, s)
    qh: Optional[tuple] = None  # prefill: Q(f32(h)) per pair (codes, scales, s)
    h_used: Optional[np.ndarray] = None  # the h fed to the down projection, [P, F]


def _expert_weights(bank, e: int) -> np.ndarray:
    """Expert e's weights in float64: E2M1(code) x UE4M3(scale), times the bank's per-expert
    second-level scale alpha[e] when it has one.  Page 4's setup runs ModelOpt NVFP4
    checkpoints with 16-weight groups, whose weights carry such a float32 scale per tensor;
    the pages never print it, so a bank without alpha means alpha = 1."""
    wt = nvfp4.dequant(bank.codes[e], bank.scales[e])
    alpha = getattr(bank, "alpha", None)
    return wt if alpha is None else wt * float(np.float32(alpha[e]))


def ffn(x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray, gate_up, down,
        mode: str = "decode", tokens: Optional[np.ndarray] = None,
        qh_override: Optional[tuple] = None) -> FFNResult:
    """Routed FFN in float64.

    x_bits uint16 [T, H] bf16 bits; ids int [T, k]; w float [T, k];
    gate_up/down: objects with ``codes``/``scales`` planes [E, rows, in/2], [E, rows, in/16].
    ``tokens`` restricts the computation to a subset of tokens (rows of y for
    the others stay zero).  ``qh_override`` (prefill only) replaces Q(h) by a
    given (codes, scales, s) triple in pair order, to check the down projection
    alone.
    """
    if mode not in ("decode", "prefill"):
        raise ValueError(mode)
    T, H = x_bits.shape
    k = ids.shape[1]
    F = gate_up.codes.shape[1] // 2
    E = gate_up.codes.shape[0]
    P = T * k
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, dtype=np.int64)
    x = nvfp4.bf16_to_f64(x_bits)
    qx = None
    if mode == "prefill":
        cx, sx, ex = nvfp4.quantize(x[tokens])
        a_tok = np.zeros_like(x)
        a_tok[tokens] = nvfp4.dequant_q(cx, sx, ex)
        full_cx = np.zeros((T, H // 2), np.uint8)
        full_sx = np.zeros((T, H // 16), np.uint8)
        full_ex = np.zeros(T, np.int64)
        full_cx[tokens], full_sx[tokens], full_ex[tokens] = cx, sx, ex
        qx = (full_cx, full_sx, full_ex)
    else:
        a_tok = x

    pairs = (tokens[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    flat_ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    z = np.zeros((P, H))
    s_abs = np.zeros((P, H))
    hh = np.zeros((P, F))
    gg = np.zeros((P, F))
    uu = np.zeros((P, F))
    ga = np.zeros((P, F))
    ua = np.zeros((P, F))
    h_used = np.zeros((P, F))
    qh_c = np.zeros((P, F // 2), np.uint8)
    qh_s = np.zeros((P, F // 16), np.uint8)
    qh_e = np.zeros(P, np.int64)
    sel = pairs[(flat_ids[pairs] >= 0) & (flat_ids[pairs] < E)]
    for e in np.unique(flat_ids[sel]):
        pe = sel[flat_ids[sel] == e]                       # this expert's pairs, ascending p
        a = a_tok[pe // k]                                  # [m, H]
        wgu = _expert_weights(gate_up, e)                           # [2F, H]
        wg, wu = wgu[:F], wgu[F:]
        g = a @ wg.T
        u = a @ wu.T
        gg[pe], uu[pe] = g, u
        ga[pe] = np.abs(a) @ np.abs(wg).T
        ua[pe] = np.abs(a) @ np.abs(wu).T
        h = silu(g) * u
        hh[pe] = h
        if mode == "prefill":
            if qh_override is not None:
                c, s, ex = (qh_override[0][pe], qh_override[1][pe], qh_override[2][pe])
            else:
                h32 = h.astype(np.float32).astype(np.float64)
                c, s, ex = nvfp4.quantize(h32)
            qh_c[pe], qh_s[pe], qh_e[pe] = c, s, ex
            hq = nvfp4.dequant_q(c, s, ex)
        else:
            hq = h
        h_used[pe] = hq
        wd = _expert_weights(down, e)                               # [H, F]
        z[pe] = hq @ wd.T
        s_abs[pe] = np.abs(hq) @ np.abs(wd).T
    y = np.zeros((T, H))
    tsum = np.zeros((T, H))
    wf = np.asarray(w, dtype=np.float64)
    valid = (flat_ids >= 0) & (flat_ids < E)
    for t in tokens:
        for j in range(k):                                 # fixed j order
            p = t * k + j
            if valid[p]:
                y[t] += wf[t, j] * z[p]
                tsum[t] += abs(wf[t, j]) * s_abs[p]
    return FFNResult(y, tsum, z, s_abs, hh, gg, uu, ga, ua, qx=qx,
                     qh=(qh_c, qh_s, qh_e) if mode == "prefill" else None, h_used=h_used)


def tolerance(tsum: np.ndarray, extra: Optional[np.ndarray] = None) -> np.ndarray:
    """Per-element bound |y_gpu - y| <= 2e-3 * sum_j |w_j * terms| + 1e-5 (+ extra)."""
    tol = TOL_REL * tsum + TOL_ABS
    if extra is not None:
        tol = tol + extra
    return tol


def unique_expert_bytes(H: int, F: int) -> int:
    """NVFP4 bytes of one expert: gate+up 2F rows of H/2 + H/16, down H rows of F/2 + F/16
    ("moe_union_probe.rs", per-expert bytes from the row arithmetic)."""
    return 2 * F * (H // 2 + H // 16) + H * (F // 2 + F // 16)


def useful_flops(P: int, H: int, F: int) -> int:
    """Useful FLOPs of one layer: P pairs x 2 x (2F*H + H*F) ("moe_sk_repro.rs",
    n_pairs * out_f * in_f * 2 per grouped call, summed over gate, up and down)."""
    return P * 2 * (2 * F * H + H * F)


# ---------------------------------------------------------------------------
# Prefill: which Q(h) decisions a float32 device accumulation may take either way
# ---------------------------------------------------------------------------

# Bound on the relative error of a float32 accumulation of K products that a
# tensor core performs in K/64 steps, one rounding of the running sum per step:
# (K/64) * 2^-24 with K <= 4096 gives 2^-18; twice that leaves room for one more
# rounding per step inside the instruction.
H_BAND = 2.0 ** -17


@dataclasses.dataclass
class QAmbiguity:
    flagged: np.ndarray        # bool [P, F]: some Q decision for the element lies within the band
    delta: np.ndarray          # float64 [P, F]: bound on |deq(Q(h')) - deq(Q(h))| where flagged
    band: np.ndarray           # float64 [P, F]: the error band eps_i assumed for h_i


def _silu_prime(g):
    sg = 1.0 / (1.0 + np.exp(-g))
    return sg * (1.0 + g * (1.0 - sg))


def qh_ambiguity(res: FFNResult, pairs: np.ndarray, beta: float = H_BAND) -> QAmbiguity:
    """Flag the elements of Q(h) whose code could differ for an h within the band.

    The band for h_i is eps_i = beta * (|silu'(g)| |u| G_abs + |silu(g)| U_abs)
    + 2^-22 |h_i| + 2^-26 amax_row, G_abs/U_abs being the sums of absolute products of
    the gate and up dot products.  The last term covers values far below every
    decision of their row: a float32 SiLU underflows to 0 for g below about -88, where
    the float64 value is ~1e-38; no threshold of Q lies below 2^-22 amax_row except the
    zero-scale one near 2^-19 amax_row, so the floor cannot hide a decision.  An element is flagged if its row exponent, its block scale
    or its own code changes between the two ends of the band.  A flagged
    element's dequantised value then moves by at most
    |deq' - h'| + |h' - h| + |h - deq| <= 1.375 unit' + eps + 1.375 unit, a
    rounding error being at most half the largest E2M1 gap (1 unit) plus the
    saturation overshoot (3/8 unit); with unit' <= unit_hi this is bounded by
    3 unit_hi + eps, unit_hi being the block's unit at the upper end of the band
    (twice that when the row exponent itself may move).
    """
    P, F = res.h.shape
    g, u = res.g, res.u
    eps = beta * (np.abs(_silu_prime(g)) * np.abs(u) * res.g_abs + np.abs(silu(g)) * res.u_abs)
    eps = eps + 2.0 ** -22 * np.abs(res.h)
    eps = eps + 2.0 ** -26 * np.abs(res.h).max(axis=1, keepdims=True)
    flagged = np.zeros((P, F), dtype=bool)
    delta = np.zeros((P, F))
    mids6 = nvfp4._UE4M3_MID6
    for p in pairs:
        v = res.h[p].astype(np.float32).astype(np.float64)
        a = np.abs(v)
        e = eps[p]
        emax = e.max()
        s = nvfp4.row_exponent(np.array([a.max()]))[0]
        s_lo = nvfp4.row_exponent(np.array([max(a.max() - emax, 0.0)]))[0]
        s_hi = nvfp4.row_exponent(np.array([a.max() + emax]))[0]
        row_amb = (s_lo != s) or (s_hi != s)
        ab = np.ldexp(a, -s).reshape(-1, 16)
        eb = np.ldexp(e, -s).reshape(-1, 16)
        bmax = ab.max(axis=1)
        bemax = eb.max(axis=1)
        sb_c = nvfp4.nearest_even(bmax, mids6)
        sb_lo = nvfp4.nearest_even(np.maximum(bmax - bemax, 0.0), mids6)
        sb_hi = nvfp4.nearest_even(bmax + bemax, mids6)
        blk_amb = (sb_lo != sb_c) | (sb_hi != sb_c)
        sbv = nvfp4.UE4M3_TABLE[sb_c][:, None]
        thr = nvfp4._E2M1_MIDS[None, None, :] * sbv[..., None]        # [nb, 1, 7]
        def mag(x):
            return ((x[..., None] > thr) | ((x[..., None] == thr) &
                    (np.arange(7) % 2 == 1))).sum(axis=-1)
        el_amb = (mag(np.maximum(ab - eb, 0.0)) != mag(ab + eb))
        # a code of magnitude 0 may take either sign
        el_amb |= (ab <= eb) & (sbv > 0)
        unit = np.ldexp(nvfp4.UE4M3_TABLE[np.minimum(sb_hi, 0x7E)], s)[:, None] * np.ones((1, 16))
        f = el_amb | blk_amb[:, None]
        if row_amb:
            f[:] = True
            unit = unit * 2.0
        flagged[p] = f.reshape(-1)
        delta[p] = np.where(f, 3.0 * unit + e.reshape(-1, 16), 0.0).reshape(-1)
    return QAmbiguity(flagged, delta, eps)


def prefill_allowance(res: FFNResult, amb: QAmbiguity, down, ids: np.ndarray,
                      w: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """Extra tolerance on y from flagged Q(h) decisions: sum_j |w| sum_i |D[r,i]| delta_i."""
    T, H = res.y.shape
    k = ids.shape[1]
    E = down.codes.shape[0]
    extra = np.zeros((T, H))
    for t in tokens:
        for j in range(k):
            p = t * k + j
            e = int(ids[t, j])
            if not 0 <= e < E or not amb.flagged[p].any():
                continue
            idx = np.nonzero(amb.flagged[p])[0]
            wd = np.abs(_expert_weights(down, e))[:, idx]
            extra[t] += abs(float(w[t, j])) * (wd @ amb.delta[p, idx])
    return extra
