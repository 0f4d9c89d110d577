"""Moves a seeded :class:`~paged_mla_decode_09_gb300.workloads.Workload` onto a GPU.

Pure data movement (numpy -> torch CUDA tensors of the storage types the
C ABI expects); no arithmetic of the method.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class DeviceBatch:
    q_nope: object  # bf16 [B, Q, H, 512]
    q_pe: object  # bf16 [B, Q, H, 64]
    kv_cache: object  # bf16 or uint8 (e4m3 codes) [num_pages, 64, 576]
    page_table: object  # int32 [B, max_pages]
    seq_lens: object  # int32 [B]
    scale: float
    kv_scale: float
    q_len: int


def to_device(wl, device="cuda") -> DeviceBatch:
    import torch

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

    if wl.kv_dtype == "bf16":
        kv = bf16(wl.kv_cache)
    else:
        kv = torch.from_numpy(np.ascontiguousarray(wl.kv_cache)).to(device)
    return DeviceBatch(
        q_nope=bf16(wl.q_nope),
        q_pe=bf16(wl.q_pe),
        kv_cache=kv,
        page_table=torch.from_numpy(np.ascontiguousarray(wl.page_table)).to(device),
        seq_lens=torch.from_numpy(np.ascontiguousarray(wl.seq_lens)).to(device),
        scale=wl.scale,
        kv_scale=wl.kv_scale,
        q_len=wl.q_len,
    )


def out_to_f64(out) -> np.ndarray:
    """bf16 device tensor -> float64 numpy (exact)."""
    return out.float().cpu().numpy().astype(np.float64)
