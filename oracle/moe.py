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
    g_acc: Optional[np.ndarray] = None   # prefill: float64 [P, F] accumulation scale of g
    u_acc: Optional[np.ndarray] = None   # prefill: float64 [P, F] accumulation scale of u


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
    g_acc = np.zeros((P, F)) if mode == "prefill" else None
    u_acc = np.zeros((P, F)) if mode == "prefill" else None
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
            acc = accumulation_scale(a, wgu)
            g_acc[pe], u_acc[pe] = acc[:, :F], acc[:, F:]
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
                     qh=(qh_c, qh_s, qh_e) if mode == "prefill" else None, h_used=h_used,
                     g_acc=g_acc, u_acc=u_acc)


def down_combine(h_used: np.ndarray, ids: np.ndarray, w: np.ndarray, down,
                 tokens: np.ndarray):
    """Steps 4-6 alone: z_p = W_down[e] h_used[p], y[t] = sum_j w[t, j] z_{t*k+j} in j order,
    and the tolerance scale tsum, for given per-pair down-projection inputs h_used [P, F]
    (pair order).  Returns (y, tsum), both float64 [T, H] (rows of other tokens zero)."""
    T, k = ids.shape
    E, H = down.codes.shape[0], down.codes.shape[1]
    y = np.zeros((T, H))
    tsum = np.zeros((T, H))
    wd = {}
    for t in np.asarray(tokens, dtype=np.int64):
        for j in range(k):                                 # fixed j order
            e = int(ids[t, j])
            if not 0 <= e < E:
                continue
            if e not in wd:
                wd[e] = _expert_weights(down, e)
            hp = h_used[t * k + j]
            y[t] += float(w[t, j]) * (wd[e] @ hp)
            tsum[t] += abs(float(w[t, j])) * (np.abs(wd[e]) @ np.abs(hp))
    return y, tsum


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

# The block-scaled FP4 tensor-core product consumes K in steps of 64 elements (one
# instruction: four 16-element groups, each with its pair of UE4M3 scales) and adds each
# step's sum into a float32 accumulator.  The products themselves are exact in float32
# (an E2M1 x UE4M3 operand has at most 6 significant bits, a product of two at most 12).
ACC_STEP = 64
# Roundings charged per step: one of the step's own sum and one of the running sum, each at
# most 2^-24 of the rounded magnitude (round to nearest).  This is an assumption about the
# device's arithmetic; the tests pin it against a float32 emulation of the accumulation and
# check the device's h against it.
ACC_ROUNDINGS = 2
UNIT_ROUNDOFF = 2.0 ** -24


def accumulation_scale(a: np.ndarray, w: np.ndarray, step: int = ACC_STEP) -> np.ndarray:
    """Sum over the K-steps of |S_j| + |A_j| for every dot product a[m] . w[n].

    S_j is the exact sum of step j's products and A_j = S_1 + ... + S_j the exact running
    sum after it.  A float32 accumulation that rounds each S_j and each A_j once (round to
    nearest) is off the exact dot product by at most 2^-24 times this scale, to first order.
    a [m, K], w [n, K] (float64, exact operand values), K a multiple of `step`; returns
    [m, n].
    """
    m, K = a.shape
    n = w.shape[0]
    if K % step:
        raise ValueError("K must be a multiple of the accumulation step")
    J = K // step
    # S[j] = a[:, step j] @ w[:, step j].T, one matrix product per step
    S = np.matmul(a.reshape(m, J, step).transpose(1, 0, 2), w.reshape(n, J, step).transpose(1, 2, 0))
    A = np.cumsum(S, axis=0)
    return np.abs(S).sum(axis=0) + np.abs(A).sum(axis=0)


@dataclasses.dataclass
class QAmbiguity:
    flagged: np.ndarray        # bool [P, F]: some Q decision for the element lies within the band
    delta: np.ndarray          # float64 [P, F]: bound on |deq(Q(h')) - deq(Q(h))| where flagged
    band: np.ndarray           # float64 [P, F]: the error band eps_i assumed for h_i
    zero_sign: np.ndarray = None   # bool [P, F]: a zero code whose sign bit may differ


def _silu_prime(g):
    sg = 1.0 / (1.0 + np.exp(-g))
    return sg * (1.0 + g * (1.0 - sg))


def h_band(res: FFNResult, widen: float = 1.0) -> np.ndarray:
    """Error band eps_i of a device float32 h_i = silu(g_i) * u_i around the exact value.

    eps = widen * ACC_ROUNDINGS * 2^-24 * (|silu'(g)| |u| g_acc + |silu(g)| u_acc)
          + 2^-22 |h| + 2^-120 |u| + 2^-140.
    The first term propagates the accumulation bound of g and u (accumulation_scale) to h
    to first order; the second covers the float32 epilogue (exp, divide, multiplies: a few
    roundings of h).  The last two cover float32 underflow, where relative bounds fail: a
    float32 SiLU is 0 for g below about -88.7 (exp(-g) overflows), while the exact
    |silu(g)| = |g| e^g there is below 2^-121; results below 2^-126 are subnormal, with an
    absolute error of at most 2^-150 per operation.
    """
    if res.g_acc is None:
        raise ValueError("the band needs a prefill-mode result (accumulation scales)")
    g, u = res.g, res.u
    eps = widen * ACC_ROUNDINGS * UNIT_ROUNDOFF * (np.abs(_silu_prime(g)) * np.abs(u) * res.g_acc
                                                   + np.abs(silu(g)) * res.u_acc)
    eps = eps + 2.0 ** -22 * np.abs(res.h)
    eps = eps + 2.0 ** -120 * np.abs(u) + 2.0 ** -140
    return eps


def qh_ambiguity(res: FFNResult, pairs: np.ndarray, widen: float = 1.0) -> QAmbiguity:
    """Flag the elements of Q(h) whose decisions could differ for any h' with
    |h'_i - h_i| <= eps_i (h_band).

    The row exponent follows the row's largest magnitude, which for such h' lies in
    [max_i (|h_i| - eps_i), max_i (|h_i| + eps_i)]; a block scale likewise follows its
    block's largest magnitude.  An element is flagged if its row exponent, its block scale
    or its own E2M1 magnitude code changes inside these intervals.  A flagged element's
    dequantised value moves by at most |deq' - h'| + |h' - h| + |h - deq| <= 1.375 unit'
    + eps + 1.375 unit, a rounding error being at most half the largest E2M1 gap (1 unit)
    plus the saturation overshoot (3/8 unit); with unit' <= unit_hi this is bounded by
    3 unit_hi + eps, unit_hi being the block's unit at the upper end of the interval
    (twice that when the row exponent itself may move).

    Separately, ``zero_sign`` marks elements whose code has magnitude 0 at both ends but
    whose sign may differ (|h_i| <= eps_i): the sign bit of a zero code follows the sign
    of h', which the band does not fix, and the value (+0 or -0) is the same either way.
    """
    P, F = res.h.shape
    eps = h_band(res, widen)
    flagged = np.zeros((P, F), dtype=bool)
    zero_sign = np.zeros((P, F), dtype=bool)
    delta = np.zeros((P, F))
    mids6 = nvfp4._UE4M3_MID6
    for p in pairs:
        v = res.h[p].astype(np.float32).astype(np.float64)
        a = np.abs(v)
        e = eps[p]
        lo = np.maximum(a - e, 0.0)
        hi = a + e
        s = nvfp4.row_exponent(np.array([a.max()]))[0]
        s_lo = nvfp4.row_exponent(np.array([lo.max()]))[0]
        s_hi = nvfp4.row_exponent(np.array([hi.max()]))[0]
        row_amb = (s_lo != s) or (s_hi != s)
        ab = np.ldexp(a, -s).reshape(-1, 16)
        lob = np.ldexp(lo, -s).reshape(-1, 16)
        hib = np.ldexp(hi, -s).reshape(-1, 16)
        sb_c = nvfp4.nearest_even(ab.max(axis=1), mids6)
        sb_lo = nvfp4.nearest_even(lob.max(axis=1), mids6)
        sb_hi = nvfp4.nearest_even(hib.max(axis=1), mids6)
        blk_amb = (sb_lo != sb_c) | (sb_hi != sb_c)
        sbv = nvfp4.UE4M3_TABLE[sb_c][:, None]
        thr = nvfp4._E2M1_MIDS[None, None, :] * sbv[..., None]        # [nb, 1, 7]

        def mag(x):
            return ((x[..., None] > thr) | ((x[..., None] == thr) &
                    (np.arange(7) % 2 == 1))).sum(axis=-1)
        m_lo, m_hi = mag(lob), mag(hib)
        el_amb = m_lo != m_hi
        unit = np.ldexp(nvfp4.UE4M3_TABLE[np.minimum(sb_hi, 0x7E)], s)[:, None] * np.ones((1, 16))
        f = el_amb | blk_amb[:, None]
        if row_amb:
            f[:] = True
            unit = unit * 2.0
        flagged[p] = f.reshape(-1)
        zero_sign[p] = (~f & (m_hi == 0) & (lob == 0.0)).reshape(-1)
        delta[p] = np.where(f, 3.0 * unit + e.reshape(-1, 16), 0.0).reshape(-1)
    return QAmbiguity(flagged, delta, eps, zero_sign)


def prefill_allowance(res: FFNResult, amb: QAmbiguity, down, ids: np.ndarray,
                      w: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """Extra tolerance on y from flagged Q(h) decisions: sum_j |w| sum_i |D[r,i]| delta_i."""
    T, H = res.y.shape
    k = ids.shape[1]
    E = down.codes.shape[0]
    extra = np.zeros((T, H))
    absd = {}
    for t in tokens:
        for j in range(k):
            p = t * k + j
            e = int(ids[t, j])
            if not 0 <= e < E or not amb.flagged[p].any():
                continue
            if e not in absd:
                absd[e] = np.abs(_expert_weights(down, e))
            idx = np.nonzero(amb.flagged[p])[0]
            extra[t] += abs(float(w[t, j])) * (absd[e][:, idx] @ amb.delta[p, idx])
    return extra
