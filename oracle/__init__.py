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

Parity status: every function here has at least one external pin except the
numerical values of the device's float32 accumulations, which are checked only
to within the stated tolerance ("parity unpinned" beyond it), and the prefill
quantisation band ``H_BAND``, which is derived from the float32 accumulation
bound rather than pinned.
"""
from . import nvfp4, moe  # noqa: F401
from .moe import (route_topk, build_expert_csr, ffn, tolerance, unique_expert_bytes,  # noqa: F401
                  useful_flops, qh_ambiguity, prefill_allowance, TOL_REL, TOL_ABS)
