"""Pins of the oracle's evaluation pass and learning-rate schedule.

Sources: nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the
optimizer step takes 524,288 tokens; 560M parameters x 20 tokens each is
~11.2B tokens, i.e. ~21,400 steps; the learning rate scales as 1/sqrt(dim);
lrm falls linearly to 0 near the end of training; validation loss is
reported as bits per byte.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import schedule as osched
from oracle.model import Config
from pretraining_step_03_b300 import shapes

TINY = Config(depth=2, d_model=128, n_head=2, vocab=512)


def _params(cfg, seed=0, std=0.05):
    rng = np.random.default_rng(seed)
    return [rng.normal(0, std, size=s) for s in oracle.param_shapes(cfg)]


def _batch(cfg, B, T, seed=3):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, cfg.vocab, (B, T)), rng.integers(0, cfg.vocab, (B, T)),
            rng.integers(1, 9, cfg.vocab))


# ------------------------------------------------------------ evaluation pass
def test_eval_sums_zero_unembedding_closed_form():
    # zero lm_head: every nll is ln V, so sum nll = N ln V and bpb = log2(V) / mean bytes
    params = _params(TINY)
    params[-1] = np.zeros_like(params[-1])
    tok, tgt, _ = _batch(TINY, 2, 8)
    tb = np.full(TINY.vocab, 4)
    s = oracle.eval_sums(params, TINY, tok, tgt, tb)
    N = tok.size
    assert abs(s[0] - N * math.log(TINY.vocab)) < 1e-9
    assert s[1] == s[0] and s[2] == 4 * N
    assert abs(oracle.bpb_of_sums(s) - math.log2(TINY.vocab) / 4) < 1e-12


def test_eval_sums_rows_are_independent():
    # each row is its own causal sequence: the sums of two halves of a batch add up
    # to the sums of the whole batch, and the ratio of sums is the corpus bpb
    params = _params(TINY)
    tok, tgt, tb = _batch(TINY, 4, 16)
    whole = oracle.eval_sums(params, TINY, tok, tgt, tb)
    a = oracle.eval_sums(params, TINY, tok[:1], tgt[:1], tb)
    b = oracle.eval_sums(params, TINY, tok[1:], tgt[1:], tb)
    for k in range(3):
        assert abs(a[k] + b[k] - whole[k]) <= 1e-9 * abs(whole[k])
    loss, bpb, _ = oracle.forward(params, TINY, tok, tgt, tb)
    assert abs(whole[0] / tok.size - loss) < 1e-12
    assert abs(oracle.bpb_of_sums(whole) - bpb) < 1e-12


def test_eval_sums_skip_zero_byte_targets():
    params = _params(TINY)
    tok, tgt, tb = _batch(TINY, 2, 16)
    tb = tb.copy()
    tb[tgt[0, 0]] = 0
    s = oracle.eval_sums(params, TINY, tok, tgt, tb)
    _, _, cache = oracle.forward(params, TINY, tok, tgt, tb)
    keep = tb[tgt.reshape(-1)] > 0
    assert s[1] < s[0]
    assert abs(s[1] - cache["nll"][keep].sum()) < 1e-12
    assert s[2] == tb[tgt.reshape(-1)].sum()


# ------------------------------------------------------------ schedule
def test_run_length_matches_pages():
    n = shapes.n_params(20, 1280, 10, 65536)
    assert 20 * n / 1e9 == pytest.approx(11.2, abs=0.05)       # "560M x 20 ~ 11.2B tokens"
    assert osched.chinchilla_steps(n, 32 * 2048 * 8) == 21400  # "11.2B / 0.5M ~ 21400"
    assert shapes.chinchilla_steps(20, 1280, 10, 65536, 524288) == 21400


def test_lrm_closed_forms():
    n, f = 100, 0.2                      # warm-down over the last 20 steps
    assert all(osched.lrm(s, n, f) == 1.0 for s in range(80))
    assert osched.lrm(80, n, f) == 1.0   # continuous where the warm-down starts
    assert osched.lrm(90, n, f) == 0.5
    assert osched.lrm(99, n, f) == pytest.approx(1 / 20)
    d = [osched.lrm(s, n, f) - osched.lrm(s + 1, n, f) for s in range(80, 99)]
    assert max(d) == pytest.approx(1 / 20) and min(d) == pytest.approx(1 / 20)   # linear
    assert all(osched.lrm(s, n, 0.0) == 1.0 for s in range(n))
    assert [osched.lrm(s, 4, 1.0) for s in range(4)] == [1.0, 0.75, 0.5, 0.25]


def test_width_scaling_is_inverse_sqrt():
    base = (0.02, 0.2, 0.004)
    for d in (512, 1280, 1664, 1920):
        mu, e, u = osched.learning_rates(0, 10, 0.2, d, 1280, base)
        assert mu == base[0]
        assert e * math.sqrt(d) == pytest.approx(base[1] * math.sqrt(1280), rel=1e-12)
        assert u * math.sqrt(d) == pytest.approx(base[2] * math.sqrt(1280), rel=1e-12)
