"""The allocation-free CSR entry point (moe_build_expert_csr_static) against the regular
one, through the C ABI.

Some callers cannot allocate device memory (an engine that owns every allocation, work
issued inside a stream capture, latency-critical loops); this entry point keeps its
scratch in a fixed device array inside the library.  Its output must be bit-identical to
moe_build_expert_csr's, on two calls in a row (the shared array keeps the last call's
contents, which must not leak into the next result).  This file is collected last so that
a failure here stops a `-x` run only after every other test has run.
"""
import numpy as np
import pytest
import torch

import synth
import nvfp4_grouped_gemm_gb300 as moe

pytestmark = pytest.mark.gpu


def _csr_regular(ids, E):
    T, k = ids.shape
    csr = moe.ExpertCSR(E, T * k)
    ws = torch.zeros(moe.workspace_bytes(T, 256, 64, E, k, moe.PATH_DECODE), dtype=torch.uint8,
                     device="cuda")
    moe.moe_build_expert_csr(ids, E, csr, ws)
    return csr


def _csr_static(ids, E):
    T, k = ids.shape
    csr = moe.ExpertCSR(E, T * k)
    moe.moe_build_expert_csr_static(ids, E, csr)
    return csr


def _same(a, b, P):
    torch.cuda.synchronize()
    n = int(a.n_active.item())
    assert n == int(b.n_active.item())
    assert torch.equal(a.expert_offsets, b.expert_offsets)
    valid = int(a.expert_offsets[-1].item())
    assert torch.equal(a.pair_ids[:valid], b.pair_ids[:valid])
    assert torch.equal(a.active_experts[:n], b.active_experts[:n])


@pytest.mark.parametrize("T,k,E", [(8, 10, 512), (4096, 8, 288), (6553, 10, 1024)])
def test_static_csr_matches_regular_twice(T, k, E):
    rng = np.random.default_rng(T)
    for call in range(2):                          # two calls in a row, different routing
        ids = torch.from_numpy(synth.skewed_ids(rng, T, k, E)).cuda()
        _same(_csr_regular(ids, E), _csr_static(ids, E), T * k)


def test_static_csr_rejects_oversize():
    ids = torch.zeros(65537, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        _csr_static(ids, 4)
    assert e.value.status == 2
