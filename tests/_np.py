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


def max_rel_err_per_head(got, ref, head_axis=-2):
    """Largest normwise relative error of any single head: for each index h of
    ``head_axis``, max|got - ref| / max|ref| over that head's entries.  An error
    confined to a head whose outputs are small next to the others' shows here
    although the whole-tensor figure hides it."""
    got = np.moveaxis(np.asarray(got, dtype=np.float64), head_axis, 0)
    ref = np.moveaxis(np.asarray(ref, dtype=np.float64), head_axis, 0)
    worst = 0.0
    for g, r in zip(got, ref):
        worst = max(worst, max_rel_err(g, r))
    return worst


def check_close(got, ref, tol, what=None, head_axis=-2):
    """Whole-tensor and per-head normwise relative error both below ``tol``;
    returns the two figures."""
    whole = max_rel_err(got, ref)
    per_head = max_rel_err_per_head(got, ref, head_axis)
    assert whole < tol and per_head < tol, \
        f"{what}: normwise {whole:.3e}, worst head {per_head:.3e}, tolerance {tol}"
    return whole, per_head
