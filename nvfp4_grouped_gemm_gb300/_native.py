"""ctypes bindings of libmoe_gb300.so (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_gb300.so")

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_size = ctypes.c_size_t

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT"}
PATH_AUTO, PATH_DECODE, PATH_PREFILL = 0, 1, 2
DEVERR_EXPERT_ID, DEVERR_TIMEOUT = 1, 2


SF_ATOMS_NONE, SF_ATOMS_GATE_UP, SF_ATOMS_ROWS = 0, 1, 2


class Bank(ctypes.Structure):
    _fields_ = [("codes", c_vp), ("scales", c_vp), ("E", c_i32), ("rows", c_i32), ("in_f", c_i32),
                ("alpha", c_vp), ("sf_atoms", c_vp), ("sf_atoms_order", c_i32)]


class CSR(ctypes.Structure):
    _fields_ = [("expert_offsets", c_vp), ("pair_ids", c_vp), ("active_experts", c_vp),
                ("n_active", c_vp)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, c_size) for n in (
        "total", "error_word", "pair_pos", "h", "xg", "xe", "hg", "he", "qx_codes", "qx_scales", "qx_exp",
        "qh_codes", "qh_scales", "qh_exp", "partial", "tiles", "slice_tiles", "sync", "row_tok")]


# (name, restype, argtypes) of every exported entry point declared in include/moe.h
SIGNATURES = [
    ("moe_workspace_bytes", c_size, [c_i32] * 6),
    ("moe_workspace_layout", c_i32, [c_i32] * 6 + [ctypes.POINTER(WsLayout)]),
    ("moe_prefill_min_pairs", c_i32, []),
    ("moe_decode_tensor_core_min_pairs", c_i32, []),
    ("moe_nvfp4_from_interleaved", c_i32, [c_vp, ctypes.c_int64, c_i32, c_vp, c_vp, c_vp]),
    ("moe_nvfp4_sf_atoms_bytes", c_size, [c_i32] * 3),
    ("moe_nvfp4_prepack_sf", c_i32, [c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_size, c_vp]),
    ("moe_resolve_path", c_i32, [c_i32] * 3),
    ("moe_kernel_launches", c_i32, [c_i32] * 6),
    ("moe_route_topk", c_i32, [c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp]),
    ("moe_build_expert_csr", c_i32, [c_vp, c_i32, c_i32, c_i32, CSR, c_vp, c_size, c_vp]),
    ("moe_grouped_gate_up_silu_nvfp4", c_i32,
     [c_vp, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(Bank), CSR, c_i32, c_vp, c_size, c_vp]),
    ("moe_grouped_down_combine_nvfp4", c_i32,
     [ctypes.POINTER(Bank), CSR, c_vp, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_size,
      c_vp]),
    ("moe_build_expert_csr_static", c_i32, [c_vp, c_i32, c_i32, c_i32, CSR, c_vp]),
    ("moe_decode_layer_nvfp4", c_i32,
     [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(Bank),
      ctypes.POINTER(Bank), c_vp, c_vp, c_size, c_vp]),
    ("moe_decode_layer_supported", c_i32, [c_i32] * 5),
    ("moe_status_string", ctypes.c_char_p, [c_i32]),
    ("moe_get_device_error", c_i32, [c_vp, c_vp, ctypes.POINTER(c_i32)]),
]

_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load the CUDA library; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -m nvfp4_grouped_gemm_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(_LIB_PATH)
    for name, res, args in SIGNATURES:
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
