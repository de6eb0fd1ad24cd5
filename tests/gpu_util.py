"""Helpers for the GPU parity tests: run one layer through the C ABI and read back
every intermediate the oracle can be compared with."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import nvfp4_grouped_gemm_gb300 as moe


@dataclasses.dataclass
class DeviceRun:
    ids: np.ndarray
    w: np.ndarray
    offsets: np.ndarray
    pair_ids: np.ndarray
    active: np.ndarray
    n_active: int
    pair_pos: np.ndarray
    h_csr: np.ndarray           # [P, F] rows in CSR order
    partial_csr: np.ndarray     # [P, H]
    y: np.ndarray
    err: int
    ws: dict
    ws_raw: Optional[np.ndarray] = None     # host copy of the whole workspace
    layer: Optional[object] = None

    def region(self, name, nbytes, dtype, shape):
        off = self.ws[name]
        return self.ws_raw[off:off + nbytes].view(dtype).reshape(shape)


def qh_scale_pitch(F: int) -> int:
    """Row pitch of the Q(h) block scales in the prefill workspace (F/16 rounded up to 16)."""
    return (F // 16 + 15) // 16 * 16


def device_banks(wl, device="cuda"):
    return (moe.NvFp4Bank.from_numpy(wl.gate_up, device), moe.NvFp4Bank.from_numpy(wl.down, device))


def ws_view(ws: torch.Tensor, off: int, nbytes: int, dtype) -> torch.Tensor:
    return ws[off:off + nbytes].view(dtype)


def run_layer(wl, path=moe.PATH_DECODE, banks=None, ids=None, w=None, fetch=True,
              layer: Optional[moe.MoeLayer] = None) -> DeviceRun:
    dev = "cuda"
    if layer is None:
        gu, dn = banks if banks is not None else device_banks(wl, dev)
        layer = moe.MoeLayer(gu, dn, wl.k)
    x = torch.from_numpy(wl.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    if wl.logits is not None and ids is None:
        logits = torch.from_numpy(wl.logits).to(dev)
        y = layer.forward(x, logits=logits, path=path)
    else:
        ids_np = wl.ids if ids is None else ids
        w_np = wl.weights if w is None else w
        ids_t = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(dev)
        w_t = torch.from_numpy(np.ascontiguousarray(w_np, dtype=np.float32)).to(dev)
        y = layer.forward(x, ids=ids_t, w=w_t, path=path)
    torch.cuda.synchronize()
    b = layer.buffers(wl.T, path)
    L = moe.workspace_layout(wl.T, wl.H, wl.F, wl.E, wl.k, path)
    P = wl.P
    ws = b["ws"]
    err = moe.get_device_error(ws)
    csr = b["csr"]
    if not fetch:
        return DeviceRun(None, None, None, None, None, 0, None, None, None, y.cpu().numpy(), err, L)
    out = DeviceRun(
        ids=b["ids"].cpu().numpy() if wl.logits is not None and ids is None else None,
        w=b["w"].cpu().numpy() if wl.logits is not None and ids is None else None,
        offsets=csr.expert_offsets.cpu().numpy(),
        pair_ids=csr.pair_ids.cpu().numpy(),
        active=csr.active_experts.cpu().numpy(),
        n_active=int(csr.n_active.item()),
        pair_pos=ws_view(ws, L["pair_pos"], 4 * P, torch.int32).cpu().numpy(),
        h_csr=ws_view(ws, L["h"], 4 * P * wl.F, torch.float32).view(P, wl.F).cpu().numpy(),
        partial_csr=ws_view(ws, L["partial"], 4 * P * wl.H, torch.float32).view(P, wl.H).cpu().numpy(),
        y=y.cpu().numpy().copy(),
        err=err,
        ws=L,
        ws_raw=ws.cpu().numpy(),
        layer=layer,
    )
    return out


def h_tolerance(res, rel=2e-3, abs_=1e-5):
    """|h_gpu - h| bound from the gate and up accumulation scales (first-order)."""
    g, u = res.g, res.u
    sg = 1.0 / (1.0 + np.exp(-g))
    dsilu = sg * (1.0 + g * (1.0 - sg))
    scale = np.abs(dsilu) * np.abs(u) * res.g_abs + np.abs(g * sg) * res.u_abs
    return rel * scale + abs_


def assert_within(got, ref, tol, what=""):
    err = np.abs(got - ref)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err / tol), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")
    return float((err / tol).max()) if err.size else 0.0
