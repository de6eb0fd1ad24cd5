"""CPU oracle for the routed-MoE NVFP4 FFN -- TEST INFRASTRUCTURE.

A plain, slow, float64 statement of what the hot path computes, written from
the pages' definitions (see ``oracle.moe`` and ``oracle.nvfp4``) and pinned by
the ``-m "not gpu"`` tests against facts outside itself: the E2M1/UE4M3 value
sets, the library's float8 decoder, brute force (``oracle.brute``), dense
matmul special cases and invariances.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's ``cpu_baseline``
and ``--impl reference`` legs may import it.  It shares no code with the CUDA
library or its Python binding; the only module both sides use is ``synth``,
which draws the seeded inputs and holds none of the method's arithmetic.

Parity status: every function here has at least one external pin.  The
numerical values of the device's float32 accumulations are checked to within
the stated tolerance ("parity unpinned" beyond it); the prefill quantisation
band (``moe.h_band``) models a float32 accumulation in 64-element K-steps and is
pinned against a float32 emulation of that accumulation.
"""
from . import nvfp4, moe  # noqa: F401
from .moe import (route_topk, build_expert_csr, ffn, tolerance, unique_expert_bytes,  # noqa: F401
                  useful_flops, qh_ambiguity, prefill_allowance, h_band, down_combine,
                  accumulation_scale, TOL_REL, TOL_ABS)
