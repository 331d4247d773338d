"""Helpers for the GPU parity tests: device inputs and oracle comparisons."""
from __future__ import annotations

import numpy as np
import torch

DEV = torch.device("cuda:0")


def xbits(x_bf16: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 numpy bits for the oracle."""
    return x_bf16.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check_bound(y_gpu: np.ndarray, y_ref: np.ndarray, s: np.ndarray, rel: float, what: str):
    """|y - y_ref| <= rel * S element by element; returns the worst ratio."""
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    bound = rel * s
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements outside {rel}*S, e.g. {idx.tolist()} "
                             f"err={err[bad][:5]} bound={bound[bad][:5]}")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / bound, 0.0)
    return float(r.max()) if r.size else 0.0
