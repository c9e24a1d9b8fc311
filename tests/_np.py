"""Conversion of torch tensors to the float64 numpy arrays the oracle reads.

bf16 and fp32 values widen exactly to float64, so the oracle sees the very
values the CUDA path reads.
"""
import numpy as np
import torch


def to_np(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    t = t.detach()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    if t.dtype in (torch.int32, torch.int64):
        return t.cpu().numpy()
    return t.cpu().double().numpy()


def max_rel_err(got, ref):
    """Normwise max relative error: max|got - ref| / max|ref| over the compared entries."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / denom) if denom > 0 else float(np.max(np.abs(got)))
