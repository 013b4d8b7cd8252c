"""Pins of the oracle's Muon and AdamW against closed forms and the SVD."""

import numpy as np
import pytest

import oracle
from oracle.optim import NS_COEFS


def _scalar_map(x, steps=5, coefs=NS_COEFS):
    a, b, c = coefs
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("shape", [(24, 24), (16, 48), (48, 16)])
def test_newton_schulz_is_the_spectral_map(shape):
    # each iteration is an odd matrix polynomial of X, so the output is
    # U p5(S / ||G||) V^T with the singular vectors of G unchanged
    rng = np.random.default_rng(0)
    g = rng.normal(size=shape)
    u, s, vt = np.linalg.svd(g, full_matrices=False)
    expect = (u * _scalar_map(s / (np.linalg.norm(g) + 1e-7))) @ vt
    np.testing.assert_allclose(oracle.newton_schulz(g), expect, atol=1e-10)


def test_newton_schulz_singular_value_band():
    # scalar map: normalised singular values >= 1e-2 land in [0.68, 1.21]
    xs = np.geomspace(1e-2, 1.0, 20001)
    ys = _scalar_map(xs)
    assert ys.min() > 0.68 and ys.max() < 1.21
    # a wide N(0,1) matrix with the d20 aspect ratio (1:4)
    rng = np.random.default_rng(1)
    g = rng.normal(size=(160, 640))
    sv = np.linalg.svd(oracle.newton_schulz(g), compute_uv=False)
    assert sv.min() > 0.6 and sv.max() < 1.3


def test_muon_first_step_closed_form():
    rng = np.random.default_rng(2)
    for shape in [(20, 20), (40, 10), (10, 40)]:
        w, g = rng.normal(size=shape), rng.normal(size=shape)
        lr = 0.02
        w1, buf, x = oracle.muon_step(w, g, np.zeros(shape), lr, momentum=0.95)
        # zero buffer: g' = (1 + mu) g, and the normalisation removes the scale
        u, s, vt = np.linalg.svd(g, full_matrices=False)
        o = (u * _scalar_map(s / np.linalg.norm(g))) @ vt
        scale = np.sqrt(max(1.0, shape[0] / shape[1]))
        np.testing.assert_allclose(w1, w - lr * scale * o, atol=1e-8)
        np.testing.assert_allclose(buf, g, rtol=0, atol=0)


def test_muon_momentum_geometric_series():
    rng = np.random.default_rng(3)
    g = rng.normal(size=(8, 8))
    w, buf, mu = np.zeros((8, 8)), np.zeros((8, 8)), 0.9
    for k in range(1, 6):
        w, buf, _ = oracle.muon_step(w, g, buf, 0.0, momentum=mu)
        np.testing.assert_allclose(buf, g * (1 - mu ** k) / (1 - mu), rtol=1e-13)


def test_muon_nesterov_direction():
    # g2 = -0.5 g1: Nesterov's g' = (mu^2 - 0.5 mu - 0.5) g1 < 0 at mu = 0.95,
    # plain momentum's buf = (mu - 0.5) g1 > 0: the update direction flips
    rng = np.random.default_rng(4)
    g1 = rng.normal(size=(12, 12))
    _, buf, x1 = oracle.muon_step(np.zeros_like(g1), g1, np.zeros_like(g1), 0.0)
    _, _, xn = oracle.muon_step(np.zeros_like(g1), -0.5 * g1, buf, 0.0, nesterov=True)
    _, _, xp = oracle.muon_step(np.zeros_like(g1), -0.5 * g1, buf, 0.0, nesterov=False)
    # equal up to the 1e-7 in the normaliser (the |g'| differ)
    np.testing.assert_allclose(xn, -x1, atol=1e-5)
    np.testing.assert_allclose(xp, x1, atol=1e-5)


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(5)
    w, g = rng.normal(size=100), rng.normal(size=100)
    lr, wd, eps = 1e-2, 0.1, 1e-8
    w1, m, v = oracle.adamw_step(w, g, np.zeros(100), np.zeros(100), lr,
                                 eps=eps, weight_decay=wd, step=1)
    np.testing.assert_allclose(w1, w * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-12)


def test_adamw_constant_gradient_is_sign_step():
    # constant g: bias correction makes m_hat = g and v_hat = g^2 at every step
    rng = np.random.default_rng(6)
    g = rng.normal(size=50)
    w, m, v = np.zeros(50), np.zeros(50), np.zeros(50)
    lr = 1e-3
    for t in range(1, 7):
        w_prev = w
        w, m, v = oracle.adamw_step(w, g, m, v, lr, step=t)
        np.testing.assert_allclose(w - w_prev, -lr * g / (np.abs(g) + 1e-8), rtol=1e-9)


def test_adamw_second_step_after_zero_gradient():
    # step 1 with g, step 2 with 0: m_hat = b1 g/(1+b1), v_hat = b2 g^2/(1+b2)
    b1, b2, lr, eps = 0.9, 0.95, 1e-2, 1e-8
    g = np.array([0.3, -2.0, 5.0])
    w, m, v = oracle.adamw_step(np.zeros(3), g, np.zeros(3), np.zeros(3), lr, b1, b2, eps, 0.0, 1)
    w2, _, _ = oracle.adamw_step(w, np.zeros(3), m, v, lr, b1, b2, eps, 0.0, 2)
    step = -lr * (b1 / (1 + b1)) * g / (np.abs(g) * np.sqrt(b2 / (1 + b2)) + eps)
    np.testing.assert_allclose(w2 - w, step, rtol=1e-12)
