"""Routed-MoE FFN with NVFP4 weights on GB300: thin Python binding of libmoe_gb300.so.

PyTorch is used only to own device memory and streams; every step of the layer runs
in the library's CUDA kernels.  Each function below marshals its arguments and calls
the C entry point of the same name (include/moe.h); a non-OK status raises MoeError.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np
import torch

from . import _native
from ._native import PATH_AUTO, PATH_DECODE, PATH_PREFILL, DEVERR_EXPERT_ID, DEVERR_TIMEOUT  # noqa
from ._native import SF_ATOMS_NONE, SF_ATOMS_GATE_UP, SF_ATOMS_ROWS  # noqa

__all__ = ["MoeError", "NvFp4Bank", "ExpertCSR", "workspace_bytes", "workspace_layout", "decode_tensor_core_min_pairs",
           "resolve_path", "prefill_min_pairs", "kernel_launches", "moe_route_topk", "moe_build_expert_csr",
           "moe_build_expert_csr_static",
           "moe_grouped_gate_up_silu_nvfp4", "moe_grouped_down_combine_nvfp4",
           "get_device_error", "MoeLayer", "PATH_AUTO", "PATH_DECODE", "PATH_PREFILL"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_native.STATUS.get(status, status)}")


def _check(status: int, where: str) -> None:
    if status != _native.MOE_OK:
        raise MoeError(status, where)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


class NvFp4Bank:
    """Planar NVFP4 bank on the device: codes u8 [E, rows, in_f/2], scales u8 [E, rows, in_f/16],
    and optionally alpha f32 [E], a per-expert second-level scale of the weights."""

    def __init__(self, codes: torch.Tensor, scales: torch.Tensor,
                 alpha: Optional[torch.Tensor] = None, sf_atoms: Optional[torch.Tensor] = None,
                 sf_atoms_order: int = 0):
        if codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
            raise TypeError("codes and scales must be uint8")
        if codes.dim() != 3 or scales.dim() != 3:
            raise ValueError("bank planes are [E, rows, bytes]")
        if not (codes.is_contiguous() and scales.is_contiguous()):
            raise ValueError("bank planes must be contiguous")
        if alpha is not None:
            if alpha.dtype != torch.float32 or alpha.numel() != codes.shape[0] or \
                    not alpha.is_contiguous() or alpha.device != codes.device:
                raise ValueError("alpha must be a contiguous float32 [E] tensor beside the codes")
        if sf_atoms is not None and (sf_atoms.dtype != torch.uint8 or not sf_atoms.is_contiguous()
                                     or sf_atoms.device != codes.device):
            raise ValueError("sf_atoms must be a contiguous uint8 tensor beside the codes")
        self.codes, self.scales, self.alpha = codes, scales, alpha
        self.sf_atoms = sf_atoms
        self.sf_atoms_order = sf_atoms_order if sf_atoms is not None else _native.SF_ATOMS_NONE
        self.E, self.rows, self.in_f = codes.shape[0], codes.shape[1], codes.shape[2] * 2
        self._c = _native.Bank(codes.data_ptr(), scales.data_ptr(), self.E, self.rows, self.in_f,
                               alpha.data_ptr() if alpha is not None else None,
                               sf_atoms.data_ptr() if sf_atoms is not None else None,
                               self.sf_atoms_order)

    def prepack_sf(self, gate_up: bool, stream=None) -> "NvFp4Bank":
        """The same bank with its scale plane also written as tensor-memory atoms
        (moe_nvfp4_prepack_sf) in the row order of the gate/up call (gate_up=True) or of the
        down call. The tensor-core GEMMs then copy each stage's weight scale factors straight
        into tensor memory; results are bit-identical to the bank without them."""
        order = _native.SF_ATOMS_GATE_UP if gate_up else _native.SF_ATOMS_ROWS
        lib = _native.load()
        n = lib.moe_nvfp4_sf_atoms_bytes(self.E, self.rows, self.in_f)
        if n == 0:
            raise ValueError("prepacking needs rows % 128 == 0 and in_f % 64 == 0")
        atoms = torch.empty(n, dtype=torch.uint8, device=self.codes.device)
        _check(lib.moe_nvfp4_prepack_sf(_ptr(self.scales), self.E, self.rows, self.in_f, order,
                                        _ptr(atoms), n, _stream(stream)), "moe_nvfp4_prepack_sf")
        return NvFp4Bank(self.codes, self.scales, self.alpha, sf_atoms=atoms, sf_atoms_order=order)

    @classmethod
    def from_interleaved(cls, blob: torch.Tensor, E: int, rows: int, in_f: int,
                         alpha: Optional[torch.Tensor] = None, stream=None) -> "NvFp4Bank":
        """A bank from the pages' interleaved storage: blob u8 [E, rows, in_f/64*36] on the
        device (36-byte blocks of 4 UE4M3 scales then 32 code bytes), converted on the GPU."""
        if blob.dtype != torch.uint8 or not blob.is_contiguous() or not blob.is_cuda:
            raise TypeError("blob must be a contiguous uint8 CUDA tensor")
        if blob.numel() != E * rows * (in_f // 64) * 36 or in_f % 64:
            raise ValueError("blob size does not match E * rows * in_f/64 * 36")
        codes = torch.empty(E, rows, in_f // 2, dtype=torch.uint8, device=blob.device)
        scales = torch.empty(E, rows, in_f // 16, dtype=torch.uint8, device=blob.device)
        _check(_native.load().moe_nvfp4_from_interleaved(_ptr(blob), E * rows, in_f, _ptr(codes),
                                                         _ptr(scales), _stream(stream)),
               "moe_nvfp4_from_interleaved")
        return cls(codes, scales, alpha)

    @classmethod
    def from_numpy(cls, bank, device="cuda") -> "NvFp4Bank":
        alpha = getattr(bank, "alpha", None)
        return cls(torch.from_numpy(bank.codes).to(device), torch.from_numpy(bank.scales).to(device),
                   None if alpha is None else torch.from_numpy(
                       np.ascontiguousarray(alpha, dtype=np.float32)).to(device))

    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel()


class ExpertCSR:
    """Device buffers of the expert-first CSR for up to P pairs over E experts."""

    def __init__(self, E: int, P: int, device="cuda"):
        self.E, self.P = E, P
        self.expert_offsets = torch.zeros(E + 1, dtype=torch.int32, device=device)
        self.pair_ids = torch.zeros(max(P, 1), dtype=torch.int32, device=device)
        self.active_experts = torch.zeros(E, dtype=torch.int32, device=device)
        self.n_active = torch.zeros(1, dtype=torch.int32, device=device)
        self._c = _native.CSR(self.expert_offsets.data_ptr(), self.pair_ids.data_ptr(),
                              self.active_experts.data_ptr(), self.n_active.data_ptr())


def workspace_bytes(T: int, H: int, F: int, E: int, k: int, path: int = PATH_AUTO) -> int:
    return int(_native.load().moe_workspace_bytes(T, H, F, E, k, path))


def workspace_layout(T: int, H: int, F: int, E: int, k: int, path: int = PATH_AUTO) -> dict:
    L = _native.WsLayout()
    _check(_native.load().moe_workspace_layout(T, H, F, E, k, path, ctypes.byref(L)),
           "moe_workspace_layout")
    return {n: int(getattr(L, n)) for n, _ in _native.WsLayout._fields_}


def resolve_path(T: int, k: int, path: int = PATH_AUTO) -> int:
    return int(_native.load().moe_resolve_path(T, k, path))


def kernel_launches(T: int, H: int, F: int, E: int, k: int, path: int = PATH_AUTO) -> int:
    """Kernels launched per layer by the CSR, gate/up and down calls (add 1 for routing)."""
    return int(_native.load().moe_kernel_launches(T, H, F, E, k, path))


def prefill_min_pairs() -> int:
    return int(_native.load().moe_prefill_min_pairs())


def decode_tensor_core_min_pairs() -> int:
    """Pairs (T*k) from which the decode path runs its tensor-core (sliced) form."""
    return int(_native.load().moe_decode_tensor_core_min_pairs())


def moe_route_topk(logits: torch.Tensor, k: int, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                   stream=None) -> None:
    T, E = logits.shape
    _check(_native.load().moe_route_topk(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w),
                                         _stream(stream)), "moe_route_topk")


def moe_build_expert_csr(topk_ids: torch.Tensor, E: int, csr: ExpertCSR, ws: torch.Tensor,
                         stream=None) -> None:
    T, k = topk_ids.shape
    _check(_native.load().moe_build_expert_csr(_ptr(topk_ids), T, k, E, csr._c, _ptr(ws),
                                               ws.numel() * ws.element_size(), _stream(stream)),
           "moe_build_expert_csr")


def moe_build_expert_csr_static(topk_ids: torch.Tensor, E: int, csr: ExpertCSR,
                                stream=None) -> None:
    """The CSR without a workspace (scratch in a fixed device array inside the library);
    for callers that cannot allocate device memory. T*k <= 65536."""
    if topk_ids.dtype != torch.int32 or not topk_ids.is_contiguous() or topk_ids.dim() != 2:
        raise TypeError("topk_ids must be a contiguous int32 [T, k] tensor")
    if not topk_ids.is_cuda or topk_ids.device.index != torch.cuda.current_device():
        raise ValueError("topk_ids must be on the current CUDA device")
    T, k = topk_ids.shape
    if csr.E != E or csr.pair_ids.numel() < T * k or csr.expert_offsets.device != topk_ids.device:
        raise ValueError("csr must be sized for E experts and T*k pairs on the same device")
    _check(_native.load().moe_build_expert_csr_static(_ptr(topk_ids), T, k, E, csr._c,
                                                      _stream(stream)),
           "moe_build_expert_csr_static")


def moe_grouped_gate_up_silu_nvfp4(x_bf16: torch.Tensor, k: int, F: int, w_gate_up: NvFp4Bank,
                                   csr: ExpertCSR, ws: torch.Tensor, path: int = PATH_AUTO,
                                   stream=None) -> None:
    T, H = x_bf16.shape
    _check(_native.load().moe_grouped_gate_up_silu_nvfp4(
        _ptr(x_bf16), T, H, F, k, ctypes.byref(w_gate_up._c), csr._c, path, _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_grouped_gate_up_silu_nvfp4")


def moe_grouped_down_combine_nvfp4(w_down: NvFp4Bank, csr: ExpertCSR, topk_w: torch.Tensor,
                                   T: int, H: int, F: int, k: int, y: torch.Tensor,
                                   ws: torch.Tensor, path: int = PATH_AUTO, stream=None) -> None:
    _check(_native.load().moe_grouped_down_combine_nvfp4(
        ctypes.byref(w_down._c), csr._c, _ptr(topk_w), T, H, F, k, path, _ptr(y), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)), "moe_grouped_down_combine_nvfp4")


def decode_layer_supported(T: int, H: int, F: int, E: int, k: int) -> bool:
    """Whether moe_decode_layer_nvfp4 (the one-kernel decode layer) takes these sizes."""
    return bool(_native.load().moe_decode_layer_supported(T, H, F, E, k))


def moe_decode_layer_nvfp4(x_bf16: torch.Tensor, k: int, w_gate_up: NvFp4Bank,
                           w_down: NvFp4Bank, y: torch.Tensor, ws: torch.Tensor,
                           topk_ids: torch.Tensor, topk_w: torch.Tensor,
                           logits: Optional[torch.Tensor] = None, stream=None) -> None:
    """The whole decode layer in one kernel.  With ``logits`` the picks and weights are
    written to ``topk_ids`` / ``topk_w``; without, they are read from them."""
    T, H = x_bf16.shape
    _check(_native.load().moe_decode_layer_nvfp4(
        _ptr(logits) if logits is not None else None, _ptr(topk_ids), _ptr(topk_w),
        _ptr(x_bf16), T, H, w_down.in_f, k, ctypes.byref(w_gate_up._c), ctypes.byref(w_down._c),
        _ptr(y), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
        "moe_decode_layer_nvfp4")


def get_device_error(ws: torch.Tensor, stream=None) -> int:
    code = ctypes.c_int32(0)
    st = _native.load().moe_get_device_error(_ptr(ws), _stream(stream), ctypes.byref(code))
    if st not in (_native.MOE_OK, 5):
        _check(st, "moe_get_device_error")
    return int(code.value)


class MoeLayer:
    """One routed-MoE FFN layer: the two NVFP4 banks plus the per-shape scratch.

    ``forward`` issues the four C-ABI calls on the current stream.  Buffers are
    allocated once per (T, path) and reused, so repeated calls allocate nothing and can
    be captured in a CUDA graph.
    """

    def __init__(self, gate_up: NvFp4Bank, down: NvFp4Bank, k: int):
        if gate_up.E != down.E or gate_up.rows != 2 * down.in_f or down.rows != gate_up.in_f:
            raise ValueError("bank shapes do not form a layer")
        self.gate_up, self.down, self.k = gate_up, down, k
        self.E, self.H, self.F = gate_up.E, gate_up.in_f, down.in_f
        self._bufs = {}

    def buffers(self, T: int, path: int = PATH_AUTO) -> dict:
        key = (T, path)
        if key not in self._bufs:
            dev = self.gate_up.codes.device
            nb = workspace_bytes(T, self.H, self.F, self.E, self.k, path)
            if nb == 0:
                raise MoeError(2, "workspace_bytes")
            self._bufs[key] = {
                "ws": torch.zeros(nb, dtype=torch.uint8, device=dev),
                "csr": ExpertCSR(self.E, T * self.k, dev),
                "ids": torch.zeros(T, self.k, dtype=torch.int32, device=dev),
                "w": torch.zeros(T, self.k, dtype=torch.float32, device=dev),
                "y": torch.zeros(T, self.H, dtype=torch.float32, device=dev),
            }
        return self._bufs[key]

    def forward(self, x_bf16: torch.Tensor, logits: Optional[torch.Tensor] = None,
                ids: Optional[torch.Tensor] = None, w: Optional[torch.Tensor] = None,
                path: int = PATH_AUTO, stream=None) -> torch.Tensor:
        T = x_bf16.shape[0]
        b = self.buffers(T, path)
        if logits is not None:
            moe_route_topk(logits, self.k, b["ids"], b["w"], stream)
            ids, w = b["ids"], b["w"]
        elif ids is None or w is None:
            raise ValueError("pass logits, or ids and w")
        moe_build_expert_csr(ids, self.E, b["csr"], b["ws"], stream)
        moe_grouped_gate_up_silu_nvfp4(x_bf16, self.k, self.F, self.gate_up, b["csr"], b["ws"],
                                       path, stream)
        moe_grouped_down_combine_nvfp4(self.down, b["csr"], w, T, self.H, self.F, self.k, b["y"],
                                       b["ws"], path, stream)
        return b["y"]

    def forward_fused(self, x_bf16: torch.Tensor, logits: Optional[torch.Tensor] = None,
                      ids: Optional[torch.Tensor] = None, w: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
        """The same layer through moe_decode_layer_nvfp4 (one kernel; decode sizes within
        decode_layer_supported).  Uses the DECODE buffers; with logits the picks and
        weights land in buffers()["ids"] / ["w"]."""
        T = x_bf16.shape[0]
        b = self.buffers(T, PATH_DECODE)
        if logits is None and (ids is None or w is None):
            raise ValueError("pass logits, or ids and w")
        if logits is not None:
            ids, w = b["ids"], b["w"]
        moe_decode_layer_nvfp4(x_bf16, self.k, self.gate_up, self.down, b["y"], b["ws"], ids, w,
                               logits=logits, stream=stream)
        return b["y"]
