"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each test patches one oracle function with a wrong variant -- a swapped nibble
order, a sign error, a dropped term, a transposed operand, a wrong tie rule, an
unstable sort -- and asserts that one of the pins in test_oracle_formats /
test_oracle_moe then fails.
"""
import numpy as np
import pytest

import oracle
from oracle import moe, nvfp4

import test_oracle_formats as fmt
import test_oracle_moe as tm


def test_planted_nibble_swap_is_caught(monkeypatch):
    orig = nvfp4.dequant

    def bad(codes, scales):
        c = np.asarray(codes, np.uint8)
        return orig(((c & 0xF) << 4 | (c >> 4)).astype(np.uint8), scales)
    monkeypatch.setattr(nvfp4, "dequant", bad)
    with pytest.raises(AssertionError):
        tm.test_ffn_matches_brute_force_tiny()


def test_planted_sign_error_in_table_is_caught(monkeypatch, golden_dir):
    bad = nvfp4.E2M1_TABLE.copy()
    bad[9] = 0.5
    monkeypatch.setattr(nvfp4, "E2M1_TABLE", bad)
    with pytest.raises(AssertionError):
        fmt.test_e2m1_table_matches_ocp_mx_values(golden_dir)


def test_planted_gate_up_swap_is_caught(monkeypatch):
    orig = nvfp4.dequant

    def bad(codes, scales):
        d = orig(codes, scales)
        if d.shape[0] % 2 == 0 and d.shape[0] == 128:        # the tiny gate_up bank rows
            half = d.shape[0] // 2
            d = np.concatenate([d[half:], d[:half]])
        return d
    monkeypatch.setattr(nvfp4, "dequant", bad)
    with pytest.raises(AssertionError):
        tm.test_ffn_matches_brute_force_tiny()


def test_planted_dropped_term_is_caught(monkeypatch):
    orig = nvfp4.dequant

    def bad(codes, scales):
        d = orig(codes, scales)
        d[..., -1] = 0.0                                      # drop the last column's term
        return d
    monkeypatch.setattr(nvfp4, "dequant", bad)
    with pytest.raises(AssertionError):
        tm.test_ffn_single_expert_equals_dense_matmul()


def test_planted_transposed_scale_group_is_caught(monkeypatch):
    orig = nvfp4.dequant

    def bad(codes, scales):
        s = np.asarray(scales)
        return orig(codes, s[..., ::-1].copy())               # scale groups in reverse order
    monkeypatch.setattr(nvfp4, "dequant", bad)
    with pytest.raises(AssertionError):
        tm.test_ffn_matches_brute_force_tiny()


def test_planted_route_tie_rule_is_caught(monkeypatch):
    def bad(logits, k):
        logits = np.asarray(logits, np.float32)
        T, E = logits.shape
        ids = np.empty((T, k), np.int32)
        w = np.empty((T, k))
        for t in range(T):
            l = logits[t].astype(np.float64)
            order = np.lexsort((-np.arange(E), -l))          # ties to the HIGHER id
            ids[t] = order[:k]
            ex = np.exp(l[order[:k]] - l[order[0]])
            w[t] = ex / ex.sum()
        return ids, w
    monkeypatch.setattr(oracle, "route_topk", bad)
    with pytest.raises(AssertionError):
        tm.test_route_matches_python_sort_with_ties()


def test_planted_unstable_csr_is_caught(monkeypatch):
    orig = moe.build_expert_csr

    def bad(ids, E):
        c = orig(ids, E)
        for e in range(E):
            a, b = c.offsets[e], c.offsets[e + 1]
            c.pair_ids[a:b] = c.pair_ids[a:b][::-1]
        return c
    monkeypatch.setattr(oracle, "build_expert_csr", bad)
    with pytest.raises(AssertionError):
        tm.test_csr_matches_stable_argsort(300, 8, 288)


def test_planted_quantiser_tie_rule_is_caught(monkeypatch):
    def bad(keys, sb):
        keys = np.asarray(keys, np.float64)
        thr = nvfp4._E2M1_MIDS[None, :] * np.asarray(sb, np.float64).reshape(-1, 1)
        mag = np.zeros(keys.shape, np.uint8)
        for j in range(7):
            mag += (keys >= thr[:, j:j + 1]).astype(np.uint8)     # ties away from zero
        return mag
    monkeypatch.setattr(nvfp4, "e2m1_magnitude_codes", bad)
    with pytest.raises(AssertionError):
        fmt.test_quantize_matches_brute_force_random_rows()


def test_planted_silu_sign_is_caught(monkeypatch):
    monkeypatch.setattr(moe, "silu", lambda g: g / (1.0 + np.exp(g)))
    with pytest.raises(AssertionError):
        tm.test_ffn_matches_brute_force_tiny()


def test_planted_interleaved_order_swap_is_caught(monkeypatch, golden_dir):
    """Codes read before the scales in a 36-byte block."""
    def bad(blob, in_f):
        b = np.asarray(blob, np.uint8)
        nblk = in_f // 64
        r = b.reshape(b.shape[:-1] + (nblk, 36))
        return (r[..., :32].reshape(b.shape[:-1] + (in_f // 2,)).copy(),
                r[..., 32:].reshape(b.shape[:-1] + (in_f // 16,)).copy())
    monkeypatch.setattr(nvfp4, "from_interleaved", bad)
    with pytest.raises(AssertionError):
        fmt.test_interleaved_block_import_matches_hand_written_fixture(golden_dir)


def test_planted_ignored_alpha_is_caught(monkeypatch):
    """The per-expert second-level scale dropped from the weights."""
    monkeypatch.setattr(moe, "_expert_weights",
                        lambda bank, e: nvfp4.dequant(bank.codes[e], bank.scales[e]))
    with pytest.raises(AssertionError):
        tm.test_alpha_power_of_two_equals_scaled_block_scales()


def test_planted_alpha_applied_twice_is_caught(monkeypatch):
    """The per-expert scale applied to the weights twice."""
    orig = moe._expert_weights

    def bad(bank, e):
        alpha = getattr(bank, "alpha", None)
        w = orig(bank, e)
        return w if alpha is None else w * float(alpha[e])
    monkeypatch.setattr(moe, "_expert_weights", bad)
    with pytest.raises(AssertionError):
        tm.test_alpha_power_of_two_equals_scaled_block_scales()
