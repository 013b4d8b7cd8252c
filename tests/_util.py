"""Comparison helpers shared by the parity tests (no method arithmetic)."""

import numpy as np


def cmp(a, b):
    """(cosine similarity, max|a-b| / max|b|) of two arrays, in fp64."""
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0, 0.0
    cos = float(a @ b / (na * nb)) if na > 0 and nb > 0 else 0.0
    scale = np.max(np.abs(b))
    rel = float(np.max(np.abs(a - b)) / scale) if scale > 0 else float(np.max(np.abs(a)))
    return cos, rel


def assert_close(a, b, cos_min, rel_max, what=""):
    cos, rel = cmp(a, b)
    assert cos >= cos_min and rel <= rel_max, f"{what}: cos {cos:.7f} (min {cos_min}), maxrel {rel:.3e} (max {rel_max})"


def bf16_round(x):
    """Round fp32/fp64 values to the nearest bfloat16 (ties to even), returned as fp32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float32).numpy()
