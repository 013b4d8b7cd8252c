"""Pins of the oracle's greedy generation (no KV cache: the plain definition).

nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the base model
is sampled as an autocomplete; the Engine's KV cache only saves recomputation.
"""

import numpy as np

import oracle
from oracle import generate as og
from oracle.model import Config

TINY = Config(depth=2, d_model=128, n_head=1, vocab=96)


def _params(cfg, seed=0, std=0.05):
    rng = np.random.default_rng(seed)
    return [rng.normal(0, std, size=s) for s in oracle.param_shapes(cfg)]


def test_zero_head_ties_go_to_the_lowest_id():
    params = _params(TINY)
    params[-1] = np.zeros_like(params[-1])
    prompt = np.random.default_rng(1).integers(0, TINY.vocab, (2, 5))
    assert np.array_equal(og.greedy(params, TINY, prompt, 4), np.zeros((2, 4), dtype=np.int64))


def test_identity_model_repeats_the_last_token():
    # all block weights zero: the residual stream is the embedding; with orthonormal
    # embedding rows and lm_head = wte the logits of row t are |e_t| * delta(t, v) / rms,
    # so the greedy continuation repeats the prompt's last token
    cfg = Config(depth=1, d_model=128, n_head=1, vocab=64)
    rng = np.random.default_rng(2)
    q, _ = np.linalg.qr(rng.normal(size=(cfg.d_model, cfg.d_model)))
    wte = q[:cfg.vocab] * 3.0
    params = [wte] + [np.zeros(s) for s in oracle.param_shapes(cfg)[1:-1]] + [wte.copy()]
    prompt = rng.integers(0, cfg.vocab, (3, 6))
    out = og.greedy(params, cfg, prompt, 5)
    assert np.array_equal(out, np.repeat(prompt[:, -1:], 5, axis=1))


def test_prefix_logits_equal_full_forward_rows():
    # the logits after a prefix are the full forward's row at the prefix's end (causality)
    params = _params(TINY)
    seq = np.random.default_rng(3).integers(0, TINY.vocab, (2, 9))
    z = og.logits_of(params, TINY, seq)
    for t in (0, 3, 8):
        np.testing.assert_allclose(og.next_logits(params, TINY, seq[:, :t + 1]), z[:, t], rtol=0, atol=1e-12)


def test_teacher_forcing_reproduces_greedy():
    params = _params(TINY, std=0.2)
    prompt = np.random.default_rng(4).integers(0, TINY.vocab, (2, 7))
    cont = og.greedy(params, TINY, prompt, 6)
    z = og.teacher_forced_logits(params, TINY, prompt, cont)
    assert z.shape == (2, 6, TINY.vocab)
    assert np.array_equal(np.argmax(z, axis=-1), cont)
