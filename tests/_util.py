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


def ns_bf16_model(g, steps=5, coefs=(3.4445, -4.7750, 2.0315), store_bf16=True):
    """Newton-Schulz with bf16 storage: a model of where the bf16 kernels round.

    Not the oracle (that is oracle.newton_schulz, fp64): this rounds to bf16
    exactly where the tensor-core path stores bf16 -- the normalised input X0
    and, every iteration, A = X X^T, B = c2 A A + c1 A and X = B X + c0 X --
    and accumulates in fp32, so cos(model, oracle) is the accuracy that bf16
    storage itself allows on this input's spectrum.  Five iterations amplify
    the rounding in the directions of the smallest singular values by up to
    3.4445^5 ~ 490, so a gradient with a long tail of tiny singular values
    (a low-rank-ish gradient) loses more than a N(0, 1) matrix does.
    """
    import torch
    a, b, c = (np.float32(x) for x in coefs)
    x = np.asarray(g, dtype=np.float32)
    x = x / np.float32(np.linalg.norm(x.astype(np.float64)) + 1e-7)
    tall = x.shape[0] > x.shape[1]
    t = torch.from_numpy(np.ascontiguousarray(x.T if tall else x))

    def r(v):
        return v.to(torch.bfloat16).to(torch.float32) if store_bf16 else v

    t = r(t)
    for _ in range(steps):
        A = r(t @ t.T)
        Bm = r(c * (A @ A) + b * A)
        t = r(Bm @ t + a * t)
    out = t.numpy().astype(np.float64)
    return out.T if tall else out


def muon_update_cos_min(geff, x_ref, cap=0.999, cos=None):
    """Smallest cosine accepted between a bf16 Muon update and the fp64 one.

    cap (0.999) wherever bf16 storage allows it; where the input's spectrum
    makes bf16 storage itself lose more (ns_bf16_model's cosine c_model below
    ~0.9995), the bound is 1 - 2 (1 - c_model): the kernel's rounding has the
    model's size, and the factor 2 leaves room for its other summation order.
    """
    if cos is not None and cos >= cap:   # the cap holds: no need for the model
        return cap, None
    cm, _ = cmp(ns_bf16_model(geff), x_ref)
    return min(cap, 1.0 - 2.0 * (1.0 - cm)), cm
