"""Helpers for the GPU tests: move synth arrays to the device and call the library's C ABI."""
from __future__ import annotations

import numpy as np
import torch

import row_wise_online_gb300 as rwo
import synth


def to_device(x_host: np.ndarray, dtype: int | None = None) -> torch.Tensor:
    """uint16 host arrays are bf16 bit patterns unless dtype is synth.F16."""
    if x_host.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x_host).view(np.int16)).cuda()
        return t.view(torch.float16 if dtype == synth.F16 else torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x_host)).cuda()


def to_host(y: torch.Tensor) -> np.ndarray:
    if y.dtype in (torch.bfloat16, torch.float16):
        return y.view(torch.int16).cpu().numpy().view(np.uint16)
    return y.cpu().numpy()


def run_softmax(x: torch.Tensor, variant: int = rwo.VARIANT_AUTO, state: bool = True):
    """y and (m, d, lse) device tensors from softmax_rows_ex; checks the status word."""
    M = x.numel() // x.shape[-1]
    m = d = lse = None
    if state:
        m = torch.full((M,), float("nan"), dtype=torch.float32, device=x.device)
        d = torch.full_like(m, float("nan"))
        lse = torch.full_like(m, float("nan"))
    y = rwo.softmax_rows_ex(x, m_out=m, d_out=d, lse_out=lse, variant=variant)
    assert rwo.get_status() == rwo.OK
    return y, m, d, lse


def rows_of(w: synth.Workload, rows) -> np.ndarray:
    return synth.generate_rows(w, rows)
