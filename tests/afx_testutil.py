"""Helpers shared by the GPU tests: move containers to the device, run the
library through its C ABI, bring results back."""
from __future__ import annotations

import numpy as np


def cuda_ready():
    import torch
    return torch.cuda.is_available()


def to_dev(arr: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.cuda()


def gpu_decode(afx, container: np.ndarray, desc, out_pad: int = 0, out_offset: int = 0):
    """Decode on the GPU; returns (uint16 numpy of n weights, status int, guard bytes intact)."""
    import torch
    dev = to_dev(container)
    total = desc.n + out_offset + out_pad
    out = torch.full((max(total, 1),), 0x5A5A, dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    view = out[out_offset:out_offset + desc.n]
    afx.afx_decode(desc, dev, view if desc.n else out, status_dev=status)
    torch.cuda.synchronize()
    host = out.cpu().numpy().view(np.uint16)
    guards = np.concatenate([host[:out_offset], host[out_offset + desc.n:total]])
    intact = bool((guards == 0x5A5A).all())
    return host[out_offset:out_offset + desc.n].copy(), int(status.item()), intact


def gpu_gemv(afx, container: np.ndarray, desc, rows: int, cols: int, x: np.ndarray):
    """Fused decode + GEMV on the GPU; returns (y float32 [B][rows], status)."""
    import torch
    dev = to_dev(container)
    xd = to_dev(x.reshape(x.shape[0] if x.ndim == 2 else 1, cols).view(np.int16))
    B = xd.shape[0]
    y = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, afx.afx_decode_gemv_workspace(desc, B) // 4), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    afx.afx_decode_gemv(desc, dev, rows, cols, xd, y, ws, status_dev=status)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(status.item())


def within_gemv_tolerance(y: np.ndarray, y_ref: np.ndarray, A: np.ndarray, rel: float = 2e-3) -> bool:
    """|y - y_ref| <= rel * sum|w x| per output (plus float32 rounding of y_ref itself)."""
    err = np.abs(y.astype(np.float64) - y_ref.astype(np.float64))
    bound = rel * A + np.abs(y_ref.astype(np.float64)) * 2.0 ** -23
    return bool(np.all(err <= bound))


def gpu_decode_any(afx, container: np.ndarray, desc, out_pad: int = 0, out_offset: int = 0, host: bool = False):
    """gpu_decode for any element format (uint16 out for BF16 / FP16, uint8 for
    E4M3); host=True keeps the container in pinned host memory (zero copy)."""
    import torch
    e4m3 = desc.format == afx.AFX_FMT_E4M3
    src = torch.from_numpy(np.ascontiguousarray(container))
    src = src.pin_memory() if host else src.cuda()
    total = desc.n + out_offset + out_pad
    guard = 0x5A if e4m3 else 0x5A5A
    out = torch.full((max(total, 1),), guard, dtype=torch.uint8 if e4m3 else torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    view = out[out_offset:out_offset + desc.n]
    afx.afx_decode(desc, src, view if desc.n else out, status_dev=status)
    torch.cuda.synchronize()
    host_out = out.cpu().numpy()
    if not e4m3:
        host_out = host_out.view(np.uint16)
    guards = np.concatenate([host_out[:out_offset], host_out[out_offset + desc.n:total]])
    intact = bool((guards == guard).all())
    return host_out[out_offset:out_offset + desc.n].copy(), int(status.item()), intact
