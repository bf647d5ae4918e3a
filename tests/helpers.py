"""Shared test helpers: tensor <-> oracle representation and the parity metric."""
from __future__ import annotations

import numpy as np
import torch

# Parity tolerances for decode attention, row-normwise relative error
# max_(b,hq,i) max_d |gpu - oracle| / max_d |oracle|: fp32 inputs 1e-5, bf16
# inputs (fp32 accumulation, bf16-rounded output: 2^-9 relative per element)
# 1e-2, fp16 inputs (fp16-rounded output: 2^-12 relative, plus the fp32
# arithmetic's 1e-6) 2e-3.
TOL = {"f32": 1e-5, "bf16": 1e-2, "f16": 2e-3}


def to_np(t: torch.Tensor) -> np.ndarray:
    """Oracle representation of a CPU/GPU tensor: float32, or raw uint16 bits for bf16."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def row_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-300)
    return float((num / den).max())


def elem_rel_err(got: np.ndarray, ref: np.ndarray, floor: float = 1e-6) -> float:
    return float((np.abs(got - ref) / np.maximum(np.abs(ref), floor)).max())
