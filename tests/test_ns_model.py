"""The bf16-storage model of Newton-Schulz that sets the Muon update bound.

tests/_util.py's ns_bf16_model runs the iteration with bf16 storage where the
kernels store bf16; the GPU Muon tests accept cos(GPU, fp64) >= min(0.999,
1 - 2 (1 - c)) with c its cosine to the fp64 oracle.  Pinned here: without
the rounding it is the oracle's map (fp32 against fp64); with it, a N(0, 1)
matrix keeps cosine >= 0.9999 while a gradient-like spectrum with a long tail
of tiny singular values loses more, as the 3.4445-per-step gain on small
singular directions predicts.
"""

import numpy as np

import oracle
from tests._util import cmp, muon_update_cos_min, ns_bf16_model


def test_without_rounding_it_is_the_oracle_map():
    g = np.random.default_rng(0).normal(size=(96, 160))
    x = ns_bf16_model(g, store_bf16=False)
    cos, rel = cmp(x, oracle.newton_schulz(g))
    assert cos > 1 - 1e-9 and rel < 1e-4, (cos, rel)
    xt = ns_bf16_model(g.T, store_bf16=False)   # tall input: through the transpose
    assert cmp(xt, oracle.newton_schulz(g.T))[1] < 1e-4


def test_normal_matrix_keeps_the_cap():
    g = np.random.default_rng(1).normal(size=(128, 256))
    cmin, cm = muon_update_cos_min(g, oracle.newton_schulz(g))
    assert cm > 0.9999 and cmin == 0.999


def test_long_spectral_tail_loses_more():
    rng = np.random.default_rng(2)
    u, _ = np.linalg.qr(rng.normal(size=(128, 128)))
    v, _ = np.linalg.qr(rng.normal(size=(256, 128)))
    sv = np.geomspace(1.0, 1e-6, 128)           # singular values over six decades
    g = (u * sv) @ v.T
    c_tail = cmp(ns_bf16_model(g), oracle.newton_schulz(g))[0]
    gn = rng.normal(size=(128, 256))
    c_norm = cmp(ns_bf16_model(gn), oracle.newton_schulz(gn))[0]
    assert c_tail < c_norm, (c_tail, c_norm)
    cmin, cm = muon_update_cos_min(g, oracle.newton_schulz(g))
    assert cmin == min(0.999, 1 - 2 * (1 - cm))
