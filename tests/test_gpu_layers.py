"""Layers composed the way a model runs them: two layers back to back in one CUDA graph on
one stream and one workspace, and a decode and a prefill layer running at the same time on
two streams with workspaces of their own.  The library keeps no state between calls except
in the workspace the caller passes, so each layer's y equals its run on its own, bit for
bit."""
import numpy as np
import pytest
import torch

import synth
import nvfp4_grouped_gemm_gb300 as moe
from gpu_util import run_layer, device_banks

pytestmark = pytest.mark.gpu


def _inputs(wl):
    x = torch.from_numpy(wl.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    lg = torch.from_numpy(wl.logits).cuda() if wl.logits is not None else None
    return x, lg


def test_two_layers_in_one_graph_share_stream_and_workspace():
    """Two decode layers with different banks and inputs (the second sized like the first,
    its own routing), captured in one graph on one stream through one MoeLayer workspace:
    ten replays, each y equal to the layer alone."""
    a = synth.by_name("decode_T8", seed=1)
    b = synth.by_name("decode_T8", seed=2)
    ref_a = run_layer(a, fetch=False).y
    ref_b = run_layer(b, fetch=False).y
    ga, da = device_banks(a)
    gb, db = device_banks(b)
    la = moe.MoeLayer(ga, da, a.k)
    lb = moe.MoeLayer(gb, db, b.k)
    lb._bufs = la._bufs                               # one workspace for both layers
    xa, lga = _inputs(a)
    xb, lgb = _inputs(b)
    ya = torch.empty(a.T, a.H, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    la.forward(xa, logits=lga, stream=stream)         # allocations outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ya.copy_(la.forward(xa, logits=lga, stream=stream))
        yb = lb.forward(xb, logits=lgb, stream=stream)
    for _ in range(10):
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(ya.cpu().numpy(), ref_a)
        assert np.array_equal(yb.cpu().numpy(), ref_b)
    assert moe.get_device_error(la.buffers(a.T)["ws"]) == 0


def test_decode_and_prefill_layers_on_two_streams_at_once():
    """A decode layer and a prefill layer launched on two streams so that they overlap on the
    GPU, each with its own workspace: both results equal the layers run alone."""
    d = synth.by_name("decode_T8", seed=4)
    p = synth.by_name("prefill_T256", seed=4)
    ref_d = run_layer(d, fetch=False).y
    ref_p = run_layer(p, path=moe.PATH_PREFILL, fetch=False).y
    ld = moe.MoeLayer(*device_banks(d), d.k)
    lp = moe.MoeLayer(*device_banks(p), p.k)
    xd, lgd = _inputs(d)
    xp = torch.from_numpy(p.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ids_p = torch.from_numpy(np.ascontiguousarray(p.ids, np.int32)).cuda()
    w_p = torch.from_numpy(np.ascontiguousarray(p.weights, np.float32)).cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            yp = lp.forward(xp, ids=ids_p, w=w_p, path=moe.PATH_PREFILL, stream=s1)
        with torch.cuda.stream(s2):
            yd = ld.forward(xd, logits=lgd, stream=s2)
        torch.cuda.synchronize()
        assert np.array_equal(yd.cpu().numpy(), ref_d)
        assert np.array_equal(yp.cpu().numpy(), ref_p)
