"""Helpers shared by the GPU parity tests (marshalling and error measures only)."""
import numpy as np


def to_dev(x, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_fro(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return np.linalg.norm(x - ref) / (den if den > 0 else 1.0)


def max_rel_elem(x, ref, floor_frac=1e-3):
    """max |x - ref| / max(|ref|, floor_frac * max|ref|): elementwise relative error with
    a floor for entries that cancel to near zero."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = max(floor_frac * np.abs(ref).max(), 1e-30)
    return float(np.max(np.abs(x - ref) / np.maximum(np.abs(ref), floor)))


def bf16_tensor(x32):
    """float32 array holding bf16 values -> torch bfloat16 tensor on the GPU (exact)."""
    import torch
    return to_dev(x32).to(torch.bfloat16)
