"""Prepacked scale planes (moe_nvfp4_prepack_sf) and the tensor-core GEMMs that read them.

(i) The atoms equal a plain restatement of the layout, bit for bit, in both row orders:
byte 16r + 4x + b of atom (e, t, j) is scale byte 4j + b of tile row 32x + r, where tile t's
row m is bank row 128t + m, or for a gate/up bank gate row 64t + m/2 (even m) and up row
64t + m/2 (odd m). (ii) A layer run with prepacked banks writes the same h, partials and y
as with the planar banks, bit for bit: the prefill GEMMs (down with its A tile resident, and
the general down GEMM at F > 768), the decode sliced form, and the decode path below it
(which reads the planar scales only); y also within the oracle's tolerance. (iii) Graph
replays with prepacked banks agree bit for bit.
"""
import hashlib

import numpy as np
import pytest
import torch

import synth
import oracle
import nvfp4_grouped_gemm_gb300 as moe
from gpu_util import run_layer, device_banks, assert_within
from prepack_layout import expected_atoms

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gate_up,E,rows,in_f", [(True, 3, 256, 512), (False, 3, 512, 192),
                                                 (True, 2, 1280, 2560), (False, 2, 2560, 640)])
def test_atoms_equal_the_layout(gate_up, E, rows, in_f):
    rng = np.random.default_rng(rows + in_f)
    scales = rng.integers(0, 127, size=(E, rows, in_f // 16), dtype=np.uint8)
    codes = np.zeros((E, rows, in_f // 2), np.uint8)
    bank = moe.NvFp4Bank(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda())
    packed = bank.prepack_sf(gate_up)
    torch.cuda.synchronize()
    assert packed.sf_atoms.numel() == scales.size
    assert np.array_equal(packed.sf_atoms.cpu().numpy(), expected_atoms(scales, gate_up))


def _prepacked(banks):
    gu, dn = banks
    return gu.prepack_sf(True), dn.prepack_sf(False)


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _same_with_prepacked(wl, path):
    banks = device_banks(wl)
    ref = run_layer(wl, path=path, banks=banks)
    got = run_layer(wl, path=path, banks=_prepacked(banks))
    assert ref.err == 0 and got.err == 0
    n = int(ref.offsets[-1])
    assert np.array_equal(_bits(got.h_csr[:n]), _bits(ref.h_csr[:n])), "h rows differ"
    assert np.array_equal(_bits(got.y), _bits(ref.y)), "y differs"
    return got


SHAPES = {
    "prefill_F1152": (256, 512, 1152, 4, 4),      # general down GEMM
    "prefill_F832": (256, 512, 832, 4, 4),        # its last k-stage holds one K-step of atoms
    "prefill_F4096": (32, 4096, 4096, 16, 4),     # largest F and H: 64 K-steps per row
    "sliced_F384": (40, 512, 384, 24, 8),         # sliced down: 6 of a stage's 12 K-steps
    "sliced_H4096": (32, 4096, 256, 64, 8),       # sliced gate/up over 64 K-steps per row
}


@pytest.mark.parametrize("name,path", [("prefill_T256", moe.PATH_PREFILL),
                                       ("prefill_F1152", moe.PATH_PREFILL),
                                       ("prefill_F832", moe.PATH_PREFILL),
                                       ("prefill_F4096", moe.PATH_PREFILL),
                                       ("verify_T32", moe.PATH_DECODE),
                                       ("verify_T128", moe.PATH_DECODE),
                                       ("sliced_F384", moe.PATH_DECODE),
                                       ("sliced_H4096", moe.PATH_DECODE),
                                       ("decode_T8", moe.PATH_DECODE)])
def test_layers_bit_identical_with_prepacked_banks(name, path):
    if name == "prefill_T256":
        wl = synth.prefill(seed=0, T=256)
    elif name in SHAPES:
        wl = synth.logits_workload(name, *SHAPES[name], seed=5)
    else:
        wl = synth.by_name(name)
    if path == moe.PATH_DECODE and name.startswith("sliced"):
        assert wl.P >= moe.decode_tensor_core_min_pairs()
    got = _same_with_prepacked(wl, path)
    if path == moe.PATH_DECODE:
        ids, w = oracle.route_topk(wl.logits, wl.k)
        res = oracle.ffn(wl.x_bits, ids, w, wl.gate_up, wl.down)
        assert_within(got.y, res.y, oracle.tolerance(res.tsum), "y")


def test_prepacked_alpha_banks_sliced_and_prefill():
    """Per-expert second-level scales with prepacked banks, on both tensor-core paths."""
    for wl, path in ((synth.verify(32), moe.PATH_DECODE),
                     (synth.prefill(seed=3, T=256), moe.PATH_PREFILL)):
        rng = np.random.default_rng(41)
        wl.gate_up.alpha = rng.uniform(0.25, 1.75, size=wl.E).astype(np.float32)
        wl.down.alpha = rng.uniform(0.5, 2.0, size=wl.E).astype(np.float32)
        _same_with_prepacked(wl, path)


def test_prepacked_graph_replays_bit_identical():
    wl = synth.verify(64)
    gu, dn = _prepacked(device_banks(wl))
    layer = moe.MoeLayer(gu, dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    logits = torch.from_numpy(wl.logits).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, logits=logits, stream=s)
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
    ref = run_layer(wl, banks=device_banks(wl), fetch=False).y
    assert hashlib.sha256(ref.tobytes()).hexdigest() in hashes


def test_plane_in_the_other_order_is_refused():
    wl = synth.verify(32)
    gu, dn = device_banks(wl)
    layer = moe.MoeLayer(gu.prepack_sf(False), dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    with pytest.raises(moe.MoeError):
        layer.forward(x, logits=torch.from_numpy(wl.logits).cuda())
