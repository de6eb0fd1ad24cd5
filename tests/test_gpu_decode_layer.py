"""GPU parity of the one-kernel decode layer (moe_decode_layer_nvfp4).

Its picks and routing weights must equal the routing call's bit for bit, and h and y must
sit within the oracle's tolerances (y: |y_gpu - y| <= 2e-3 * sum_j |w_j * terms| + 1e-5).
Every step runs the arithmetic of the per-call TMA-fed decode kernels (the f16 prescales,
each unit's K order, the combine in ascending j), so where the four-call layer runs those
kernels (from 8 units per SM in both projections) h and y must also equal its h and y bit
for bit; below that the per-call path's CTA kernels sum K in another order.  Graph replays
must agree bit for bit.
"""
import hashlib

import numpy as np
import pytest
import torch

import synth
import oracle
import nvfp4_grouped_gemm_gb300 as moe
from gpu_util import run_layer, assert_within, device_banks, ws_view, h_tolerance

pytestmark = pytest.mark.gpu


def _x(wl):
    return torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)


def _fused(wl, banks, ids=None, w=None):
    """Run the layer through moe_decode_layer_nvfp4; return y, picks, weights, h, error."""
    gu, dn = banks
    layer = moe.MoeLayer(gu, dn, wl.k)
    x = _x(wl)
    if wl.logits is not None and ids is None:
        y = layer.forward_fused(x, logits=torch.from_numpy(wl.logits).cuda())
    else:
        ids_t = torch.from_numpy(np.ascontiguousarray(wl.ids if ids is None else ids, np.int32)).cuda()
        w_t = torch.from_numpy(np.ascontiguousarray(wl.weights if w is None else w, np.float32)).cuda()
        y = layer.forward_fused(x, ids=ids_t, w=w_t)
    torch.cuda.synchronize()
    b = layer.buffers(wl.T, moe.PATH_DECODE)
    L = moe.workspace_layout(wl.T, wl.H, wl.F, wl.E, wl.k, moe.PATH_DECODE)
    h = ws_view(b["ws"], L["h"], 4 * wl.P * wl.F, torch.float32).view(wl.P, wl.F).cpu().numpy()
    err = moe.get_device_error(b["ws"])
    return (y.cpu().numpy().copy(), b["ids"].cpu().numpy(), b["w"].cpu().numpy(), h, err)


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def _per_call_runs_tma_kernels(wl):
    """Whether both projections of the four-call layer run the TMA-fed kernels (at least 8
    units per SM: min(P, E) * F/8 gate/up units, min(P, E) * H/16 down units)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m = min(wl.P, wl.E)
    return m * (wl.F // 8) >= 8 * sms and m * (wl.H // 16) >= 8 * sms


def _same_as_per_call(wl, ids=None, w=None, expect_err=0):
    """Run both forms; check picks, weights, h and y against the four-call layer and the
    oracle.  Returns y and the four-call run."""
    assert moe.decode_layer_supported(wl.T, wl.H, wl.F, wl.E, wl.k)
    banks = device_banks(wl)
    ref = run_layer(wl, banks=banks, ids=ids, w=w)
    y, f_ids, f_w, h, err = _fused(wl, banks, ids=ids, w=w)
    assert err == expect_err and ref.err == expect_err
    if wl.logits is not None and ids is None:
        assert np.array_equal(f_ids, ref.ids), "picks differ from the routing call"
        assert np.array_equal(_bits(f_w), _bits(ref.w)), "routing weights differ"
        o_ids, o_w = oracle.route_topk(wl.logits, wl.k)
    else:
        o_ids = wl.ids if ids is None else ids
        o_w = (wl.weights if w is None else w).astype(np.float64)
    res = oracle.ffn(wl.x_bits, o_ids, np.asarray(o_w, np.float64), wl.gate_up, wl.down)
    # h in CSR order: the kernel's CSR is the CSR call's (checked bit-exact in the decode tests)
    valid = np.flatnonzero(ref.pair_pos >= 0)
    assert_within(h[ref.pair_pos[valid]], res.h[valid], h_tolerance(res)[valid], "h")
    assert_within(y, res.y, oracle.tolerance(res.tsum), "y")
    if _per_call_runs_tma_kernels(wl):
        n_valid = int(ref.offsets[-1])
        assert np.array_equal(_bits(h[:n_valid]), _bits(ref.h_csr[:n_valid])), "h rows differ"
        assert np.array_equal(_bits(y), _bits(ref.y)), "y differs from the four-call layer"
    return y, ref


@pytest.mark.parametrize("name", ["decode_T1", "decode_T2", "decode_T4", "decode_T8",
                                  "union_U10", "union_U30", "union_U60", "verify_T16"])
def test_layer_kernel_equals_four_calls_and_oracle(name):
    wl = synth.by_name(name)
    _same_as_per_call(wl)


@pytest.mark.parametrize("T,H,F,E,k", [(3, 256, 128, 16, 4),       # small, one K-box chunks
                                       (5, 768, 384, 40, 6),       # nb = 1 boxes, F = 384
                                       (4, 4096, 256, 1024, 32),   # largest E, k and H
                                       (25, 512, 256, 64, 10)])    # 250 pairs, 25 tokens
def test_layer_kernel_shapes(T, H, F, E, k):
    wl = synth.logits_workload(f"layer_{T}_{H}_{F}_{E}_{k}", T, H, F, E, k, seed=31)
    _same_as_per_call(wl)


def test_layer_kernel_many_pairs_per_expert():
    """An expert with 120 pairs (15 groups of eight: each unit streamed 15 times), given
    picks instead of logits."""
    T, k, E = 24, 10, 32
    wl = synth.logits_workload("layer_hot", T, 512, 256, E, k, seed=32)
    rng = np.random.default_rng(33)
    # tokens 0..11 pick among experts 6..31; tokens 12..23 name expert 5 in all k slots
    ids = np.stack([6 + rng.permutation(E - 6)[:k] for _ in range(T)]).astype(np.int32)
    ids[12:, :] = 5
    w = rng.uniform(0.0, 1.0, size=(T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    _, ref = _same_as_per_call(wl, ids=ids, w=w)
    assert int(np.diff(ref.offsets)[5]) == 120


def test_layer_kernel_invalid_ids_flagged_and_left_out():
    """Given picks with ids outside [0, E): the error word says so and those pairs add
    nothing, exactly as on the four-call path."""
    T, k, E = 6, 4, 16
    wl = synth.logits_workload("layer_bad", T, 256, 128, E, k, seed=34)
    rng = np.random.default_rng(35)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[1, 2] = E
    ids[4, 0] = -3
    w = np.full((T, k), 0.25, np.float32)
    _same_as_per_call(wl, ids=ids, w=w, expect_err=moe.DEVERR_EXPERT_ID)


def test_layer_kernel_alpha_banks():
    """Per-expert second-level scales on both banks."""
    wl = synth.decode(4)
    rng = np.random.default_rng(36)
    for bank in (wl.gate_up, wl.down):
        bank.alpha = rng.uniform(0.25, 1.75, size=bank.E).astype(np.float32)
    _same_as_per_call(wl)


def test_layer_kernel_graph_replays_bit_identical():
    """Ten CUDA-graph replays of the one-kernel layer give one hash, equal to an eager call
    and to the four-call layer."""
    wl = synth.decode(8)
    banks = device_banks(wl)
    layer = moe.MoeLayer(*banks, wl.k)
    x = _x(wl)
    logits = torch.from_numpy(wl.logits).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward_fused(x, logits=logits, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        y = layer.forward_fused(x, logits=logits, stream=s)
    hashes = set()
    for _ in range(10):
        g.replay()
        torch.cuda.synchronize()
        hashes.add(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
    assert len(hashes) == 1
    eager = layer.forward_fused(x, logits=logits).cpu().numpy()
    assert hashlib.sha256(eager.tobytes()).hexdigest() in hashes
    assert _per_call_runs_tma_kernels(wl)
    ref = run_layer(wl, banks=banks, fetch=False).y
    assert hashlib.sha256(ref.tobytes()).hexdigest() in hashes


def test_layer_kernel_two_layers_back_to_back():
    """Layers through the call one after another: the sync words of each workspace keep
    counting from call to call (a fresh layer's start at zero), and results repeat."""
    a, b = synth.decode(2, seed=1), synth.decode(8, seed=2)
    ya, _ = _same_as_per_call(a)
    yb, _ = _same_as_per_call(b)
    ya2, _ = _same_as_per_call(a)
    assert np.array_equal(_bits(ya), _bits(ya2))


def test_layer_kernel_wait_runs_out_then_reports_until_zeroed():
    """The kernel's bounded waits, made to run out without a fault: the workspace's call
    counter is set far ahead of the barrier counters (as in a workspace left by another
    run), so no count the grid reaches satisfies a wait. The waits give up after their 2 s
    budget, the call sets MOE_DEVERR_TIMEOUT and marks the sync words, the next call only
    reports it, and after the workspace is zero-filled again the layer is back to normal."""
    import time
    wl = synth.decode(1)
    banks = device_banks(wl)
    layer = moe.MoeLayer(*banks, wl.k)
    x = _x(wl)
    lg = torch.from_numpy(wl.logits).cuda()
    y_ok = layer.forward_fused(x, logits=lg).cpu().numpy().copy()
    b = layer.buffers(wl.T, moe.PATH_DECODE)
    assert moe.get_device_error(b["ws"]) == 0
    L = moe.workspace_layout(wl.T, wl.H, wl.F, wl.E, wl.k, moe.PATH_DECODE)
    sync = b["ws"][L["sync"]:L["sync"] + 48].view(torch.int64)
    assert int(sync[0]) == 1                       # one completed call: the epoch advanced
    sync[0] = 1000                                 # barrier targets no count can reach
    t0 = time.time()
    layer.forward_fused(x, logits=lg)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert moe.get_device_error(b["ws"]) & moe.DEVERR_TIMEOUT
    assert int(sync[5]) != 0                       # the sync words are marked
    t0 = time.time()
    layer.forward_fused(x, logits=lg)              # reports it without waiting
    torch.cuda.synchronize()
    assert time.time() - t0 < 1.0
    assert moe.get_device_error(b["ws"]) & moe.DEVERR_TIMEOUT
    b["ws"].zero_()
    y = layer.forward_fused(x, logits=lg).cpu().numpy()
    assert moe.get_device_error(b["ws"]) == 0
    assert np.array_equal(_bits(y), _bits(y_ok))
