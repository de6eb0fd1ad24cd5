"""The allocation-free CSR entry point (moe_build_expert_csr_static), through the C ABI,
against the regular entry point and the oracle.

Some callers cannot allocate device memory: a host engine or plugin that owns every
device allocation, or code where cudaMalloc (which may block and synchronise the device)
is not allowed.  This entry point keeps its scratch in a fixed device array inside the
library.  Its output must be bit-identical to moe_build_expert_csr's, and to the oracle's
CSR, on two calls in a row (the shared array keeps the last call's contents, which must
not leak into the next result).  This file is collected last so that a failure here stops
a `-x` run only after every other test has run.
"""
import numpy as np
import pytest
import torch

import synth
import oracle
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


def _same(a, b):
    torch.cuda.synchronize()
    n = int(a.n_active.item())
    assert n == int(b.n_active.item())
    assert torch.equal(a.expert_offsets, b.expert_offsets)
    valid = int(a.expert_offsets[-1].item())
    assert torch.equal(a.pair_ids[:valid], b.pair_ids[:valid])
    assert torch.equal(a.active_experts[:n], b.active_experts[:n])


def _same_as_oracle(csr, ids_np, E):
    ref = oracle.build_expert_csr(ids_np, E)
    n_valid = int(ref.offsets[-1])
    assert np.array_equal(csr.expert_offsets.cpu().numpy(), ref.offsets)
    assert np.array_equal(csr.pair_ids.cpu().numpy()[:n_valid], ref.pair_ids)
    assert int(csr.n_active.item()) == ref.n_active
    assert np.array_equal(csr.active_experts.cpu().numpy()[:ref.n_active], ref.active)
    return n_valid


@pytest.mark.parametrize("T,k,E", [(8, 10, 512), (4096, 8, 288), (6553, 10, 1024)])
def test_static_csr_matches_regular_and_oracle_twice(T, k, E):
    rng = np.random.default_rng(T)
    for call in range(2):                          # two calls in a row, different routing
        ids_np = synth.skewed_ids(rng, T, k, E)
        ids = torch.from_numpy(ids_np).cuda()
        st = _csr_static(ids, E)
        _same(_csr_regular(ids, E), st)
        _same_as_oracle(st, ids_np, E)


def test_static_csr_leaves_out_invalid_ids():
    """Out-of-range ids are dropped as by the regular entry point; with no error word, the
    caller sees it as expert_offsets[E] < T*k.  A clean call after it is unaffected."""
    T, k, E = 300, 8, 64
    rng = np.random.default_rng(9)
    ids_np = synth.skewed_ids(rng, T, k, E)
    bad = rng.choice(T * k, size=11, replace=False)
    ids_np.reshape(-1)[bad[:6]] = E + 5
    ids_np.reshape(-1)[bad[6:]] = -3
    st = _csr_static(torch.from_numpy(ids_np).cuda(), E)
    n_valid = _same_as_oracle(st, ids_np, E)
    assert n_valid == T * k - 11
    clean = synth.skewed_ids(rng, T, k, E)
    st2 = _csr_static(torch.from_numpy(clean).cuda(), E)
    assert _same_as_oracle(st2, clean, E) == T * k


def test_static_csr_rejects_oversize():
    ids = torch.zeros(65537, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        _csr_static(ids, 4)
    assert e.value.status == 2
