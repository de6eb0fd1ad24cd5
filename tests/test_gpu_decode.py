"""GPU parity of the decode path against the CPU oracle, through the C ABI.

Integer outputs (expert ids, CSR offsets, pair order, active list, n_active) must be
bit-exact; floating point must satisfy |y_gpu - y| <= 2e-3 * sum_j |w_j * terms| + 1e-5
per element, and replays must be bit-identical.
"""
import hashlib

import numpy as np
import pytest
import torch

import synth
import oracle
import nvfp4_grouped_gemm_gb300 as moe
from gpu_util import run_layer, h_tolerance, assert_within, device_banks

pytestmark = pytest.mark.gpu


def _check_csr(run, ids, E):
    ref = oracle.build_expert_csr(ids, E)
    n_valid = int(ref.offsets[-1])
    assert np.array_equal(run.offsets, ref.offsets)
    assert np.array_equal(run.pair_ids[:n_valid], ref.pair_ids)
    assert run.n_active == ref.n_active
    assert np.array_equal(run.active[:ref.n_active], ref.active)
    assert np.array_equal(run.pair_pos, ref.pair_pos)
    return ref


def _check_layer(wl, run, tokens=None, check_h=True):
    if wl.logits is not None:
        ids, w = oracle.route_topk(wl.logits, wl.k)
        assert np.array_equal(run.ids, ids), "routing ids differ"
        assert np.allclose(run.w, w, rtol=2e-6, atol=1e-7), "routing weights differ"
    else:
        ids, w = wl.ids, wl.weights.astype(np.float64)
    _check_csr(run, ids, wl.E)
    res = oracle.ffn(wl.x_bits, ids, w, wl.gate_up, wl.down, tokens=tokens)
    toks = np.arange(wl.T) if tokens is None else np.asarray(tokens)
    pairs = (toks[:, None] * wl.k + np.arange(wl.k)).reshape(-1)
    if check_h:
        h_gpu = run.h_csr[run.pair_pos[pairs]]
        assert_within(h_gpu, res.h[pairs], h_tolerance(res)[pairs], "h")
    worst = assert_within(run.y[toks], res.y[toks], oracle.tolerance(res.tsum)[toks], "y")
    return worst


def test_tiny_decode():
    wl = synth.tiny()
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


@pytest.mark.parametrize("T", [1, 2, 4, 8])
def test_decode_sweep(T):
    wl = synth.decode(T)
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


@pytest.mark.parametrize("U", [60, 30, 20, 10])
def test_union_sweep(U):
    wl = synth.union(U)
    run = run_layer(wl)
    assert run.err == 0
    assert run.n_active == U
    _check_layer(wl, run)


@pytest.mark.parametrize("T", [16, 32, 64, 80, 128])
def test_verify_batch(T):
    wl = synth.verify(T)
    run = run_layer(wl)
    assert run.err == 0
    # every row up to 64 tokens (640 pairs over ~235 experts); 24 spread rows beyond
    tokens = None if T <= 64 else np.linspace(0, T - 1, 24).astype(int)
    _check_layer(wl, run, tokens=tokens)


def test_verify_replays_bit_identical():
    """Ten CUDA-graph replays of the whole layer give one hash (deterministic combine)."""
    wl = synth.verify(128)
    gu, dn = device_banks(wl)
    layer = moe.MoeLayer(gu, dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    logits = torch.from_numpy(wl.logits).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, logits=logits, stream=s)      # allocate buffers, warm up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        y = layer.forward(x, logits=logits, stream=s)
    hashes = set()
    for _ in range(10):
        g.replay()
        torch.cuda.synchronize()
        hashes.add(hashlib.sha256(y.cpu().numpy().tobytes()).hexdigest())
    assert len(hashes) == 1
    # eager calls agree with the graph bit for bit
    y2 = layer.forward(x, logits=logits).cpu().numpy()
    assert hashlib.sha256(y2.tobytes()).hexdigest() in hashes


def test_split_batch_bit_identical():
    """Page 4's split check: a batch computed as two halves equals the whole, bit for bit."""
    wl = synth.decode(8)
    gu, dn = device_banks(wl)
    full = run_layer(wl, banks=(gu, dn), fetch=False).y
    for lo, hi in ((0, 4), (4, 8)):
        part = synth.Workload(wl.name, hi - lo, wl.H, wl.F, wl.E, wl.k, wl.x_bits[lo:hi],
                              wl.gate_up, wl.down, logits=wl.logits[lo:hi])
        y = run_layer(part, banks=(gu, dn), fetch=False).y
        assert np.array_equal(y, full[lo:hi])


def test_split_batch_bit_identical_sliced():
    """The same split check on the sliced tensor-core form (both halves at >= 256 pairs):
    a pair's slices depend only on its token and each output column is reduced on its own,
    so how pairs share tiles does not change a bit."""
    wl = synth.verify(128)
    gu, dn = device_banks(wl)
    full = run_layer(wl, banks=(gu, dn), fetch=False).y
    for lo, hi in ((0, 64), (64, 128)):
        part = synth.Workload(wl.name, hi - lo, wl.H, wl.F, wl.E, wl.k, wl.x_bits[lo:hi],
                              wl.gate_up, wl.down, logits=wl.logits[lo:hi])
        y = run_layer(part, banks=(gu, dn), fetch=False).y
        assert np.array_equal(y, full[lo:hi])


def test_interleaved_banks_import_bit_exact_and_run_the_same_layer():
    """Banks stored the pages' way (36-byte blocks: 4 scales then 32 code bytes per 64
    weights) convert on the GPU to exactly the oracle's planar bytes, and a layer on the
    converted banks is bit-identical to one on banks converted by the oracle."""
    from oracle import nvfp4
    wl = synth.decode(8)

    def interleave(bank):
        E, rows, half = bank.codes.shape
        in_f = half * 2
        c = bank.codes.reshape(E, rows, in_f // 64, 32)
        s = bank.scales.reshape(E, rows, in_f // 64, 4)
        return np.concatenate([s, c], axis=-1).reshape(E, rows, in_f // 64 * 36), in_f

    banks = []
    for bank in (wl.gate_up, wl.down):
        blob, in_f = interleave(bank)
        E, rows = blob.shape[:2]
        dev = moe.NvFp4Bank.from_interleaved(torch.from_numpy(np.ascontiguousarray(blob)).cuda(),
                                             E, rows, in_f)
        torch.cuda.synchronize()
        ref_c, ref_s = nvfp4.from_interleaved(blob, in_f)
        assert np.array_equal(dev.codes.cpu().numpy(), ref_c)
        assert np.array_equal(dev.scales.cpu().numpy(), ref_s)
        banks.append(dev)
    y_imp = run_layer(wl, banks=tuple(banks), fetch=False).y
    y_ref = run_layer(wl, fetch=False).y
    assert np.array_equal(y_imp, y_ref)


@pytest.mark.parametrize("shape", ["decode_T8", "sliced"])
def test_per_expert_alpha(shape):
    """Banks with a per-expert float32 second-level scale alpha (both decode forms)."""
    if shape == "decode_T8":
        wl = synth.decode(8)
    else:
        wl = synth.logits_workload("alpha_sliced", 32, 256, 128, 16, 8, seed=8)
        assert wl.P >= moe.decode_tensor_core_min_pairs()
    rng = np.random.default_rng(12)
    for bank in (wl.gate_up, wl.down):
        bank.alpha = rng.uniform(0.25, 1.75, size=bank.E).astype(np.float32)
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


def test_single_token_single_expert():
    """k = 1, T = 1: the smallest layer."""
    wl = synth.tiny(seed=3)
    one = synth.Workload("one", 1, wl.H, wl.F, wl.E, 1, wl.x_bits[:1], wl.gate_up, wl.down,
                         ids=np.array([[5]], np.int32), weights=np.array([[1.0]], np.float32))
    run = run_layer(one)
    _check_layer(one, run)


@pytest.mark.parametrize("F", [1024, 1408])
def test_wide_ff_decode(F):
    """ff widths up to the decode path's largest (wider h rows held in registers)."""
    wl = synth.logits_workload(f"wide_F{F}", 3, 256, F, 8, 2, seed=11)
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


@pytest.mark.parametrize("T", [4, 8])
def test_decode_largest_E_k_and_H(T):
    """The largest router width, top-k and hidden size a layer takes (E = 1024, k = 32,
    H = 4096): 128 pairs run the mma.sync kernels, 256 pairs the sliced tensor-core form."""
    wl = synth.logits_workload(f"limits_T{T}", T, 4096, 256, 1024, 32, seed=23)
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


@pytest.mark.parametrize("name,path", [("decode_T8", moe.PATH_DECODE), ("verify_T32", moe.PATH_DECODE),
                                       ("prefill_T64", moe.PATH_PREFILL)])
def test_expert_relabel_bit_identical(name, path):
    """Relabelling the experts (bank e' = bank pi^-1(e'), ids -> pi(ids)) reorders the CSR
    and the work but not any pair's arithmetic: y is bit-identical, on the mma.sync and
    sliced decode forms and on the prefill path."""
    wl = synth.by_name(name, seed=3)
    ids = wl.ids if wl.ids is not None else oracle.route_topk(wl.logits, wl.k)[0]
    w = wl.weights if wl.weights is not None else oracle.route_topk(wl.logits, wl.k)[1].astype(np.float32)
    base = synth.Workload(name, wl.T, wl.H, wl.F, wl.E, wl.k, wl.x_bits, wl.gate_up, wl.down,
                          ids=np.ascontiguousarray(ids, np.int32), weights=np.ascontiguousarray(w, np.float32))
    y0 = run_layer(base, path=path, fetch=False).y
    pi = np.random.default_rng(31).permutation(wl.E)
    inv = np.argsort(pi)

    def relabel(bank):
        return type(bank)(bank.codes[inv], bank.scales[inv], None if bank.alpha is None else bank.alpha[inv])
    moved = synth.Workload(name, wl.T, wl.H, wl.F, wl.E, wl.k, wl.x_bits, relabel(wl.gate_up),
                           relabel(wl.down), ids=pi[base.ids].astype(np.int32), weights=base.weights)
    y1 = run_layer(moved, path=path, fetch=False).y
    assert np.array_equal(y0, y1)


@pytest.mark.parametrize("name,path", [("decode_T8", moe.PATH_DECODE), ("verify_T32", moe.PATH_DECODE),
                                       ("prefill_T64", moe.PATH_PREFILL)])
def test_pinned_host_buffers_passed_to_the_calls(name, path):
    """The calls take pinned host memory for x, the router logits (or ids and weights) and
    y: the kernels read and write it over the host link, and y equals the device-buffer
    run bit for bit."""
    wl = synth.by_name(name, seed=7)
    gu, dn = device_banks(wl)
    layer = moe.MoeLayer(gu, dn, wl.k)
    b = layer.buffers(wl.T, path)
    x_d = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    x_h = x_d.cpu().pin_memory()
    y_h = torch.empty(wl.T, wl.H, dtype=torch.float32).pin_memory()
    if wl.logits is not None:
        l_d = torch.from_numpy(wl.logits).cuda()
        y_dev = layer.forward(x_d, logits=l_d, path=path).clone()
        moe.moe_route_topk(l_d.cpu().pin_memory(), wl.k, b["ids"], b["w"])
        ids_t, w_t = b["ids"], b["w"]
    else:
        i_d = torch.from_numpy(np.ascontiguousarray(wl.ids, np.int32)).cuda()
        w_d = torch.from_numpy(np.ascontiguousarray(wl.weights, np.float32)).cuda()
        y_dev = layer.forward(x_d, ids=i_d, w=w_d, path=path).clone()
        ids_t, w_t = i_d.cpu().pin_memory(), w_d.cpu().pin_memory()
    moe.moe_build_expert_csr(ids_t, wl.E, b["csr"], b["ws"])
    moe.moe_grouped_gate_up_silu_nvfp4(x_h, wl.k, wl.F, gu, b["csr"], b["ws"], path)
    moe.moe_grouped_down_combine_nvfp4(dn, b["csr"], w_t, wl.T, wl.H, wl.F, wl.k, y_h, b["ws"], path)
    torch.cuda.synchronize()
    assert torch.equal(y_h, y_dev.cpu())
    assert moe.get_device_error(b["ws"]) == 0


def test_csr_many_pairs_with_invalid_ids():
    """The grid-wide CSR (thousands of pairs) skips and flags out-of-range ids, keeps the
    rest in ascending pair order, and writes -1 as their CSR position."""
    T, k, E = 700, 8, 96
    rng = np.random.default_rng(5)
    ids = synth.skewed_ids(rng, T, k, E)
    bad = rng.choice(T * k, size=37, replace=False)
    ids.reshape(-1)[bad[:20]] = E + 3
    ids.reshape(-1)[bad[20:]] = -1
    csr = moe.ExpertCSR(E, T * k)
    ws = torch.zeros(moe.workspace_bytes(T, 256, 64, E, k, moe.PATH_DECODE), dtype=torch.uint8,
                     device="cuda")
    moe.moe_build_expert_csr(torch.from_numpy(ids).cuda(), E, csr, ws)
    torch.cuda.synchronize()
    ref = oracle.build_expert_csr(ids, E)
    assert np.array_equal(csr.expert_offsets.cpu().numpy(), ref.offsets)
    assert np.array_equal(csr.pair_ids.cpu().numpy()[:int(ref.offsets[-1])], ref.pair_ids)
    assert int(csr.n_active.item()) == ref.n_active
    assert np.array_equal(csr.active_experts.cpu().numpy()[:ref.n_active], ref.active)
    L = moe.workspace_layout(T, 256, 64, E, k, moe.PATH_DECODE)
    pos = ws[L["pair_pos"]:L["pair_pos"] + 4 * T * k].view(torch.int32).cpu().numpy()
    assert np.array_equal(pos, ref.pair_pos)
    assert moe.get_device_error(ws) & moe.DEVERR_EXPERT_ID


def test_invalid_expert_ids_are_flagged_and_skipped():
    wl = synth.tiny(seed=4)
    ids = np.array([[1, 3], [99, 3], [-2, 0], [7, 7]], np.int32)
    w = np.full((4, 2), 0.5, np.float32)
    bad = synth.Workload("bad", 4, wl.H, wl.F, wl.E, 2, wl.x_bits, wl.gate_up, wl.down,
                         ids=ids, weights=w)
    run = run_layer(bad)
    assert run.err & moe.DEVERR_EXPERT_ID
    res = oracle.ffn(bad.x_bits, ids, w.astype(np.float64), bad.gate_up, bad.down)
    ref = _check_csr(run, ids, bad.E)
    assert int(ref.offsets[-1]) == 6
    assert_within(run.y, res.y, oracle.tolerance(res.tsum), "y")
    # the error word is cleared by reading it
    assert moe.get_device_error(torch.zeros(256, dtype=torch.uint8, device="cuda")) == 0


def test_duplicate_expert_in_one_token():
    wl = synth.tiny(seed=9)
    ids = np.array([[2, 2], [2, 5], [5, 2], [2, 2]], np.int32)
    w = np.array([[0.3, 0.7], [0.5, 0.5], [0.9, 0.1], [0.25, 0.75]], np.float32)
    dup = synth.Workload("dup", 4, wl.H, wl.F, wl.E, 2, wl.x_bits, wl.gate_up, wl.down,
                         ids=ids, weights=w)
    run = run_layer(dup)
    _check_layer(dup, run)


def test_many_pairs_on_one_expert():
    """One expert with more pairs than one 8- or 16-token pass holds."""
    wl = synth.decode(T=40)
    ids = np.zeros((40, 10), np.int32)
    ids[:, 0] = 17                         # 40 pairs on expert 17
    ids[:, 1:] = synth.union_ids(40, 9, 400, 9) + 100
    w = np.full((40, 10), 0.1, np.float32)
    many = synth.Workload("many", 40, wl.H, wl.F, wl.E, 10, wl.x_bits, wl.gate_up, wl.down,
                          ids=ids, weights=w)
    run = run_layer(many)
    _check_layer(many, run, tokens=[0, 13, 39])


@pytest.mark.parametrize("T,H,F,E,k", [(64, 256, 64, 16, 8),      # one k-step for down
                                       (80, 256, 128, 7, 7),      # 80 pairs per expert: 10 tiles
                                       (40, 512, 384, 24, 8),     # K/2 = 192: 1.5 sub-tiles
                                       (52, 512, 1408, 32, 10)])  # widest decode F
def test_sliced_path_shapes(T, H, F, E, k):
    """From 256 pairs the decode path runs the sliced tensor-core GEMMs: ragged tiles, an
    expert spread over many 8-pair tiles, a down projection of one 64-wide k-step, a down
    row ending halfway into its second 128-byte sub-tile (F = 384; the zero-filled half's
    k-steps are skipped), and the widest F (its weight-scale rows staged whole)."""
    assert T * k >= moe.decode_tensor_core_min_pairs()
    wl = synth.logits_workload(f"sliced_{T}_{H}_{F}", T, H, F, E, k, seed=21)
    run = run_layer(wl)
    assert run.err == 0
    _check_layer(wl, run)


def test_sliced_path_invalid_ids_and_duplicates():
    """Invalid ids are skipped and flagged; a token may name one expert twice (sliced form)."""
    T, k, E = 64, 8, 40
    wl = synth.logits_workload("sliced_bad", T, 256, 128, E, k, seed=5)
    rng = np.random.default_rng(5)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    ids[3, 2] = E + 7
    ids[10, 0] = -1
    ids[20, 5] = ids[20, 6]
    w = rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)
    bad = synth.Workload("sliced_bad", T, wl.H, wl.F, E, k, wl.x_bits, wl.gate_up, wl.down,
                         ids=ids, weights=w)
    run = run_layer(bad)
    assert run.err & moe.DEVERR_EXPERT_ID
    res = oracle.ffn(bad.x_bits, ids, w.astype(np.float64), bad.gate_up, bad.down)
    _check_csr(run, ids, E)
    assert_within(run.y, res.y, oracle.tolerance(res.tsum), "y")


@pytest.mark.parametrize("T,E,k", [(64, 512, 10), (33, 7, 3), (40, 33, 32), (17, 64, 8),
                                   (50, 100, 6), (29, 300, 16), (12, 1024, 32), (5, 997, 1)])
def test_route_ties_to_lower_id(T, E, k):
    """Every router width (one warp up to 32 warps merged) against the oracle, on logits
    with many exact ties, signed zeros among them."""
    rng = np.random.default_rng(11 + E)
    logits = np.round(rng.standard_normal((T, E)) * 2).astype(np.float32)   # many exact ties
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, k, dtype=torch.float32, device="cuda")
    moe.moe_route_topk(torch.from_numpy(logits).cuda(), k, ids, w)
    ref_ids, ref_w = oracle.route_topk(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(w.cpu().numpy(), ref_w, rtol=2e-6)


@pytest.mark.parametrize("T,k,E", [(4096, 8, 288), (1, 1, 1), (3, 7, 1024), (2048, 1, 64),
                                   (1000, 5, 1024), (600, 7, 7)])
def test_csr_bit_exact_large(T, k, E):
    rng = np.random.default_rng(T + E)
    ids = synth.skewed_ids(rng, T, k, E)
    csr = moe.ExpertCSR(E, T * k)
    ws = torch.zeros(moe.workspace_bytes(T, 256, 64, E, k, moe.PATH_DECODE), dtype=torch.uint8,
                     device="cuda")
    moe.moe_build_expert_csr(torch.from_numpy(ids).cuda(), E, csr, ws)
    torch.cuda.synchronize()
    ref = oracle.build_expert_csr(ids, E)
    assert np.array_equal(csr.expert_offsets.cpu().numpy(), ref.offsets)
    assert np.array_equal(csr.pair_ids.cpu().numpy()[:T * k], ref.pair_ids)
    assert int(csr.n_active.item()) == ref.n_active
    assert np.array_equal(csr.active_experts.cpu().numpy()[:ref.n_active], ref.active)


@pytest.mark.parametrize("name", ["verify_T32", "sliced_F384"])
def test_sliced_h_slices_bit_exact_against_the_oracle(name):
    """The four residual slices of h the sliced form writes (codes, block scales, row
    exponents of every slice row) equal the oracle's q_i = Q(v - q_0 - ... - q_{i-1}) of the
    GPU's own h rows, bit for bit (the residuals are exact in float32 as in float64)."""
    from oracle import nvfp4
    if name == "verify_T32":
        wl = synth.verify(32)
    else:
        wl = synth.logits_workload("sliced_F384", 40, 512, 384, 24, 8, seed=21)
    assert wl.P >= moe.decode_tensor_core_min_pairs()
    run = run_layer(wl)
    assert run.err == 0
    L, F, NS = run.ws, wl.F, 4
    R = wl.P * NS
    pitch = (F // 16 + 15) // 16 * 16
    n_valid = int(run.offsets[-1])
    codes = run.ws_raw[L["qh_codes"]:L["qh_codes"] + R * F // 2].reshape(R, F // 2)
    scales = run.ws_raw[L["qh_scales"]:L["qh_scales"] + R * pitch].reshape(R, pitch)[:, :F // 16]
    exps = run.ws_raw[L["qh_exp"]:L["qh_exp"] + 4 * R].view(np.int32)
    v = run.h_csr[:n_valid].astype(np.float64)
    acc = np.zeros_like(v)
    for i in range(NS):
        c, sc, e = nvfp4.quantize(v - acc)
        rows = np.arange(n_valid) * NS + i
        assert np.array_equal(codes[rows], c), f"slice {i} codes"
        assert np.array_equal(scales[rows], sc), f"slice {i} scales"
        assert np.array_equal(exps[rows], e.astype(np.int32)), f"slice {i} exponents"
        acc = acc + nvfp4.dequant_q(c, sc, e)


@pytest.mark.parametrize("name", ["verify_T128", "verify_T32", "sliced_H4096"])
def test_sliced_x_slices_bit_exact_against_the_oracle(name):
    """The four residual slices of each pair's x row (its token's bf16 row) that the sliced
    form writes equal the oracle's quantiser applied to the running residual, bit for bit,
    in every CSR row: per-token CTAs (verify_T128), per-pair CTAs (verify_T32), H = 4096."""
    from oracle import nvfp4
    if name == "sliced_H4096":
        wl = synth.logits_workload("sliced_H4096", 32, 4096, 256, 64, 8, seed=22)
    else:
        wl = synth.by_name(name)
    assert wl.P >= moe.decode_tensor_core_min_pairs()
    run = run_layer(wl)
    assert run.err == 0
    L, H, NS = run.ws, wl.H, 4
    R = wl.P * NS
    n_valid = int(run.offsets[-1])
    codes = run.ws_raw[L["qx_codes"]:L["qx_codes"] + R * H // 2].reshape(R, H // 2)
    scales = run.ws_raw[L["qx_scales"]:L["qx_scales"] + R * H // 16].reshape(R, H // 16)
    exps = run.ws_raw[L["qx_exp"]:L["qx_exp"] + 4 * R].view(np.int32)
    tok = run.pair_ids[:n_valid] // wl.k
    v = synth.bf16_bits_to_f32(wl.x_bits)[tok].astype(np.float64)
    acc = np.zeros_like(v)
    for i in range(NS):
        c, sc, e = nvfp4.quantize(v - acc)
        rows = np.arange(n_valid) * NS + i
        assert np.array_equal(codes[rows], c), f"slice {i} codes"
        assert np.array_equal(scales[rows], sc), f"slice {i} scales"
        assert np.array_equal(exps[rows], e.astype(np.int32)), f"slice {i} exponents"
        acc = acc + nvfp4.dequant_q(c, sc, e)
