"""Pins of the oracle's hand-derived backward: central finite differences in fp64.

The oracle's forward is the plain definition of the step; its backward is
derived by hand, so it is checked against the forward itself by central
differences on the tiny configuration (a transposed operand, a dropped term
or a wrong sign anywhere in the backward changes a directional derivative).
"""

import numpy as np
import pytest

import oracle
from oracle.model import Config

CFG = Config(depth=2, d_model=128, n_head=2, vocab=512)


@pytest.fixture(scope="module")
def setup():
    rng = np.random.default_rng(0)
    # std 0.1 so that attention scores and the MLP are far from linear
    params = [rng.normal(0, 0.1, size=s) for s in oracle.param_shapes(CFG)]
    tok = rng.integers(0, 512, (2, 16))
    tgt = rng.integers(0, 512, (2, 16))
    tb = rng.integers(1, 9, 512)
    loss, bpb, grads = oracle.loss_and_grads(params, CFG, tok, tgt, tb)
    return params, tok, tgt, tb, grads


def _loss(params, tok, tgt, tb):
    return oracle.forward(params, CFG, tok, tgt, tb)[0]


def test_directional_derivative_every_tensor(setup):
    params, tok, tgt, tb, grads = setup
    rng = np.random.default_rng(1)
    h = 1e-4
    for i, p in enumerate(params):
        u = rng.normal(size=p.shape)
        u /= np.linalg.norm(u)
        pp = list(params)
        pp[i] = p + h * u
        lp = _loss(pp, tok, tgt, tb)
        pp[i] = p - h * u
        lm = _loss(pp, tok, tgt, tb)
        fd = (lp - lm) / (2 * h)
        an = float(np.sum(grads[i] * u))
        assert abs(fd - an) <= 1e-6 * abs(an) + 1e-11, (i, fd, an)


def test_sampled_coordinates(setup):
    params, tok, tgt, tb, grads = setup
    rng = np.random.default_rng(2)
    h = 1e-5
    for i, p in enumerate(params):
        g = grads[i]
        gmax = np.max(np.abs(g))
        if i == 0:
            # embedding: half the samples on rows that were looked up
            rows = np.concatenate([rng.choice(np.unique(tok), 8), rng.integers(0, p.shape[0], 8)])
        else:
            rows = rng.integers(0, p.shape[0], 16)
        cols = rng.integers(0, p.shape[1], rows.size)
        for r, c in zip(rows, cols):
            pp = list(params)
            q = p.copy()
            q[r, c] += h
            pp[i] = q
            lp = _loss(pp, tok, tgt, tb)
            q[r, c] -= 2 * h
            lm = _loss(pp, tok, tgt, tb)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[r, c]) <= 1e-6 * gmax + 1e-10, (i, r, c, fd, g[r, c])


def test_unused_embedding_rows_have_zero_grad(setup):
    params, tok, tgt, tb, grads = setup
    unused = np.setdiff1d(np.arange(CFG.vocab), tok)
    assert np.all(grads[0][unused] == 0.0)


def test_grad_scale_is_linear(setup):
    params, tok, tgt, tb, grads = setup
    _, _, g2 = oracle.loss_and_grads(params, CFG, tok, tgt, tb, grad_scale=0.5)
    for a, b in zip(grads, g2):
        np.testing.assert_allclose(0.5 * a, b, rtol=1e-12, atol=1e-300)
