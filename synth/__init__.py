"""Seeded synthetic inputs for the routed-MoE NVFP4 FFN.

This module is shared by the CPU oracle and by the CUDA path's tests and
benchmark.  It only *draws* inputs; it holds none of the method's arithmetic
(no routing, grouping, decoding, GEMM or combine).  Every array is produced by
``numpy.random.default_rng(seed)`` in one fixed order:

1. router logits (or the given expert ids, then the routing weights)
2. activations x
3. gate/up codes, 4. gate/up scales, 5. down codes, 6. down scales

Shapes and distributions follow the five workloads the pages measure:

* tiny      -- T=4, hidden=256, ff=64, E=16, top-k=2 (oracle-sized case)
* decode    -- hidden=2560, ff=640, E=512, top-k=10, T in {1,2,4,8}
               ("moe_sel_census.rs" column curve; "moe_union_probe.rs" geometry)
* union     -- T=6, top-k=10 (60 slots), hidden=2560, ff=640, E=512, U distinct
               experts named round-robin ("moe_union_probe.rs", header comment)
* prefill   -- T=4096, hidden=4096, ff=640, E=288, top-k=8, expert of each pair
               floor(u^1.35 * E) ("moe_sk_repro.rs", fn route and fn main)
* verify    -- hidden=2560, ff=640, E=256, top-k=10, T in {16,32,64,80,128}
               ("Rank-local E256 MoE misses the Qwen K1 and K4 step budgets",
               rows table)

NVFP4 banks are planar: ``codes`` u8 [E, rows, in_f/2] (two E2M1 codes per
byte, low nibble = even element) and ``scales`` u8 [E, rows, in_f/16] (one
UE4M3 byte per 16 weights).  Codes are uniform random bytes (so each nibble is
uniform over all 16 codes, -0 included); scales are uniform over the UE4M3
encodings 0x08..0x30, exactly the encodings whose value lies in [2^-6, 0.5].
Activations are float32 N(0,1) rounded to nearest-even bfloat16 and returned
as their uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

SCALE_LO = 0x08  # UE4M3 encoding of 2^-6
SCALE_HI = 0x30  # UE4M3 encoding of 0.5


@dataclasses.dataclass
class Bank:
    """One NVFP4 weight bank, planar: codes [E, rows, in_f//2], scales [E, rows, in_f//16],
    and optionally alpha [E] float32 (a per-expert second-level scale)."""
    codes: np.ndarray
    scales: np.ndarray
    alpha: Optional[np.ndarray] = None

    @property
    def E(self) -> int:
        return self.codes.shape[0]

    @property
    def rows(self) -> int:
        return self.codes.shape[1]

    @property
    def in_f(self) -> int:
        return self.codes.shape[2] * 2


@dataclasses.dataclass
class Workload:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    x_bits: np.ndarray                 # uint16 [T, H] bfloat16 bit patterns
    gate_up: Bank                      # rows = 2F (gate rows first), in_f = H
    down: Bank                         # rows = H, in_f = F
    logits: Optional[np.ndarray] = None   # float32 [T, E] (router input), or None
    ids: Optional[np.ndarray] = None      # int32 [T, k] given routing, or None
    weights: Optional[np.ndarray] = None  # float32 [T, k] given routing weights, or None
    seed: int = 0
    meta: dict = dataclasses.field(default_factory=dict)

    @property
    def P(self) -> int:
        return self.T * self.k


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _draw_bank(rng: np.random.Generator, E: int, rows: int, in_f: int) -> Bank:
    if in_f % 16:
        raise ValueError("in_f must be a multiple of 16")
    codes = rng.integers(0, 256, size=(E, rows, in_f // 2), dtype=np.uint8)
    scales = rng.integers(SCALE_LO, SCALE_HI + 1, size=(E, rows, in_f // 16), dtype=np.uint8)
    return Bank(codes, scales)


def _draw_x(rng: np.random.Generator, T: int, H: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def _draw_weights(rng: np.random.Generator, T: int, k: int) -> np.ndarray:
    """Routing weights uniform(0,1), renormalised per token to sum to one."""
    w = rng.random((T, k))
    w = w / w.sum(axis=1, keepdims=True)
    return w.astype(np.float32)


def _draw_banks(rng, E, H, F):
    gu = _draw_bank(rng, E, 2 * F, H)
    dn = _draw_bank(rng, E, H, F)
    return gu, dn


def logits_workload(name: str, T: int, H: int, F: int, E: int, k: int, seed: int = 0,
                    E_bank: Optional[int] = None) -> Workload:
    """Workload whose routing comes from router logits N(0,1) [T, E]."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E), dtype=np.float32)
    x = _draw_x(rng, T, H)
    gu, dn = _draw_banks(rng, E if E_bank is None else E_bank, H, F)
    return Workload(name, T, H, F, E, k, x, gu, dn, logits=logits, seed=seed)


def tiny(seed: int = 0) -> Workload:
    """T=4 tokens, hidden=256, ff=64, E=16 experts, top-2."""
    return logits_workload("tiny", 4, 256, 64, 16, 2, seed)


def decode(T: int = 8, seed: int = 0) -> Workload:
    """Decode sweep point: hidden=2560, ff=640, E=512, top-10, T tokens."""
    return logits_workload(f"decode_T{T}", T, 2560, 640, 512, 10, seed)


def verify(T: int = 128, seed: int = 0) -> Workload:
    """Rank-local verify batch: hidden=2560, ff=640, E=256, top-10, T rows."""
    return logits_workload(f"verify_T{T}", T, 2560, 640, 256, 10, seed)


def union_ids(T: int, k: int, E: int, U: int) -> np.ndarray:
    """Slot s = t*k + j names expert list[s mod U], list[j] = j * (E // U)."""
    experts = np.arange(U, dtype=np.int64) * (E // U)
    slots = np.arange(T * k, dtype=np.int64)
    return experts[slots % U].reshape(T, k).astype(np.int32)


def union(U: int = 60, seed: int = 0, T: int = 6, k: int = 10, H: int = 2560, F: int = 640,
          E: int = 512) -> Workload:
    """Fixed 60 slots naming U distinct experts round-robin; weights uniform, renormalised."""
    rng = np.random.default_rng(seed)
    ids = union_ids(T, k, E, U)
    w = _draw_weights(rng, T, k)
    x = _draw_x(rng, T, H)
    gu, dn = _draw_banks(rng, E, H, F)
    return Workload(f"union_U{U}", T, H, F, E, k, x, gu, dn, ids=ids, weights=w, seed=seed,
                    meta={"U": U})


def skewed_ids(rng: np.random.Generator, T: int, k: int, E: int, power: float = 1.35) -> np.ndarray:
    """Expert of each pair = min(floor(u^power * E), E-1), u uniform(0,1)."""
    u = rng.random((T, k))
    e = np.floor(np.power(u, power) * E).astype(np.int64)
    return np.minimum(e, E - 1).astype(np.int32)


def prefill(seed: int = 0, T: int = 4096, H: int = 4096, F: int = 640, E: int = 288,
            k: int = 8) -> Workload:
    """Prefill grouped GEMM: 4096 tokens x top-8 over 288 experts, skewed routing."""
    rng = np.random.default_rng(seed)
    ids = skewed_ids(rng, T, k, E)
    w = _draw_weights(rng, T, k)
    x = _draw_x(rng, T, H)
    gu, dn = _draw_banks(rng, E, H, F)
    return Workload(f"prefill_T{T}", T, H, F, E, k, x, gu, dn, ids=ids, weights=w, seed=seed)


def by_name(name: str, seed: int = 0) -> Workload:
    """'tiny', 'decode_T8', 'union_U30', 'prefill', 'prefill_T256', 'verify_T64', ..."""
    if name == "tiny":
        return tiny(seed)
    if name.startswith("decode_T"):
        return decode(int(name[len("decode_T"):]), seed)
    if name.startswith("verify_T"):
        return verify(int(name[len("verify_T"):]), seed)
    if name.startswith("union_U"):
        return union(int(name[len("union_U"):]), seed)
    if name == "prefill":
        return prefill(seed)
    if name.startswith("prefill_T"):
        return prefill(seed, T=int(name[len("prefill_T"):]))
    raise KeyError(name)


def hash_route(p: int, n_expert: int) -> int:
    """The deterministic pair-index hash router of "moe_sk_repro.rs" (fn route), restated.

    A 64-bit multiply / xor-shift mix of the pair index gives u in [0,1); the
    expert is min(floor(u^1.35 * E), E-1).  It is an alternative, RNG-free
    generator of the same skewed distribution as :func:`skewed_ids`.
    """
    mask = (1 << 64) - 1
    h = (p * 0x9E3779B97F4A7C15) & mask
    h ^= h >> 29
    h = (h * 0xBF58476D1CE4E5B9) & mask
    h ^= h >> 32
    u = (h >> 11) / float(1 << 53)
    return min(int((u ** 1.35) * n_expert), n_expert - 1)
