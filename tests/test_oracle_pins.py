"""Pins of the oracle forward against the pages and closed-form mathematics."""

import json
import math
import os

import numpy as np

import oracle
from oracle.model import Config
from pretraining_step_03_b300 import shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TINY = Config(depth=2, d_model=128, n_head=2, vocab=512)


def _params(cfg, seed=0, std=0.05):
    rng = np.random.default_rng(seed)
    return [rng.normal(0, std, size=s) for s in oracle.param_shapes(cfg)]


def _batch(cfg, B, T, seed=3):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, cfg.vocab, (B, T)), rng.integers(0, cfg.vocab, (B, T)),
            rng.integers(1, 9, cfg.vocab))


# ------------------------------------------------------------ loss and bpb
def test_zero_unembedding_gives_ln_vocab():
    for cfg in (TINY, Config(depth=1, d_model=64, n_head=1, vocab=65536)):
        params = _params(cfg)
        params[-1] = np.zeros_like(params[-1])
        tok, tgt, tb = _batch(cfg, 2, 8)
        loss, bpb, cache = oracle.forward(params, cfg, tok, tgt, tb)
        assert abs(loss - math.log(cfg.vocab)) < 1e-12
        grads = oracle.backward(cache, cfg)
        # logits all zero: softmax is uniform, so dWu[v] = mean_i (1/V - [t_i = v]) yf_i
        N = tok.size
        onehot = np.zeros((N, cfg.vocab))
        onehot[np.arange(N), tgt.reshape(-1)] = 1.0
        expect = ((1.0 / cfg.vocab) - onehot).T @ cache["yf"] / N
        np.testing.assert_allclose(grads[-1], expect, rtol=1e-10, atol=1e-15)


def test_unembedding_grad_rows_sum_to_zero():
    # softmax - onehot sums to zero over the vocabulary for every token
    params = _params(TINY)
    tok, tgt, tb = _batch(TINY, 2, 16)
    _, _, grads = oracle.loss_and_grads(params, TINY, tok, tgt, tb)
    assert np.max(np.abs(grads[-1].sum(axis=0))) < 1e-14


def test_bpb_with_constant_bytes():
    params = _params(TINY)
    tok, tgt, _ = _batch(TINY, 2, 16)
    for c in (1, 3):
        loss, bpb, _ = oracle.forward(params, TINY, tok, tgt, np.full(TINY.vocab, c))
        assert abs(bpb * c * math.log(2) - loss) < 1e-12


def test_bpb_ignores_zero_byte_targets():
    # a target whose byte count is 0 adds to neither sum: if every target
    # but one has zero bytes, bpb is that one token's nll / (ln2 * bytes)
    params = _params(TINY)
    tok, tgt, _ = _batch(TINY, 1, 8)
    tgt = tgt.copy()
    tgt[0, :] = 7
    tgt[0, 5] = 9
    tb = np.zeros(TINY.vocab, dtype=np.int64)
    tb[9] = 3
    loss, bpb, cache = oracle.forward(params, TINY, tok, tgt, tb)
    nll5 = cache["nll"][5]
    assert abs(bpb - nll5 / (3 * math.log(2))) < 1e-12


# ------------------------------------------------------------ causality
def test_causality_future_token_leaves_past_logits_unchanged():
    params = _params(TINY, std=0.1)
    tok, tgt, tb = _batch(TINY, 2, 16)
    z0 = oracle.forward(params, TINY, tok, tgt, tb)[2]["z"].reshape(2, 16, -1)
    t = 6
    tok2 = tok.copy()
    tok2[0, t + 1] = (tok2[0, t + 1] + 1) % TINY.vocab
    z1 = oracle.forward(params, TINY, tok2, tgt, tb)[2]["z"].reshape(2, 16, -1)
    assert np.array_equal(z0[0, : t + 1], z1[0, : t + 1])
    assert np.array_equal(z0[1], z1[1])
    assert not np.allclose(z0[0, t + 1:], z1[0, t + 1:])


# ------------------------------------------------------------ attention
def test_attention_single_position_is_v():
    rng = np.random.default_rng(0)
    q, k, v = (rng.normal(size=(3, 1, 4, 16)) for _ in range(3))
    o, p, lse = oracle.causal_attention(q, k, v)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(lse, np.einsum("bthd,bthd->bht", q, k) / 4.0, rtol=1e-14)


def test_attention_brute_force_loops():
    rng = np.random.default_rng(1)
    B, T, H, D = 2, 5, 2, 4
    q, k, v = (rng.normal(size=(B, T, H, D)) for _ in range(3))
    o, _, lse = oracle.causal_attention(q, k, v)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                sc = [sum(q[b, t, h, j] * k[b, s, h, j] for j in range(D)) / math.sqrt(D)
                      for s in range(t + 1)]
                mx = max(sc)
                w = [math.exp(x - mx) for x in sc]
                tot = sum(w)
                assert abs(lse[b, h, t] - (mx + math.log(tot))) < 1e-12
                for j in range(D):
                    ref = sum(w[s] * v[b, s, h, j] for s in range(t + 1)) / tot
                    assert abs(o[b, t, h, j] - ref) < 1e-12


# ------------------------------------------------------------ RMSNorm
def test_rmsnorm_mean_square_and_backward_identity():
    rng = np.random.default_rng(2)
    x = rng.normal(size=(7, 33)) * rng.uniform(1e-3, 10, size=(7, 1))
    y, r = oracle.rmsnorm(x)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + 1e-6), rtol=1e-12)
    dy = rng.normal(size=x.shape)
    dx = oracle.rmsnorm_backward(dy, y, r)
    # scale invariance up to eps: <dx, x> = <dy, y> * eps / (ms + eps)
    lhs = np.sum(dx * x, axis=-1)
    rhs = np.sum(dy * y, axis=-1) * 1e-6 / (ms + 1e-6)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-6, atol=1e-12)


# ------------------------------------------------------------ RoPE
def test_rope_is_relative_and_orthogonal():
    rng = np.random.default_rng(3)
    T, D = 12, 16
    cos, sin = oracle.rope_tables(T, D)
    qv, kv = rng.normal(size=D), rng.normal(size=D)
    q = np.broadcast_to(qv, (1, T, 1, D)).copy()
    k = np.broadcast_to(kv, (1, T, 1, D)).copy()
    rq, rk = oracle.rope(q, cos, sin)[0, :, 0], oracle.rope(k, cos, sin)[0, :, 0]
    np.testing.assert_allclose(rq[0], qv, rtol=0, atol=0)           # position 0 is identity
    dots = rq @ rk.T
    for s in range(1, 5):                                             # depends on t1 - t2 only
        np.testing.assert_allclose(np.diagonal(dots, s)[1:], np.diagonal(dots, s)[:-1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(rq, axis=-1), np.linalg.norm(qv), rtol=1e-13)
    x = rng.normal(size=(2, T, 3, D))
    np.testing.assert_allclose(oracle.rope_backward(oracle.rope(x, cos, sin), cos, sin), x, atol=1e-13)
    # pair (j, j + D/2) rotates by t * 10000^(-2j/D): check one angle by hand
    t, j = 5, 3
    ang = t * 10000.0 ** (-2 * j / D)
    e = np.zeros((1, T, 1, D))
    e[0, t, 0, j] = 1.0
    out = oracle.rope(e, cos, sin)[0, t, 0]
    assert abs(out[j] - math.cos(ang)) < 1e-15 and abs(out[j + D // 2] - math.sin(ang)) < 1e-15


# ------------------------------------------------------------ geometry (pages)
def test_d20_parameter_count_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "d20_pages.json")))
    cfg = Config(g["depth"], g["d_model"], g["n_head"], 65536)
    assert cfg.head_dim == g["head_dim"]
    n = sum(r * c for r, c in oracle.param_shapes(cfg))
    assert n == 560_988_160
    assert abs(n / g["params_approx"] - 1) < 0.005
    assert 12 * 1280 ** 2 * 20 + 2 * 65536 * 1280 == n
    # the library's own geometry agrees with the oracle's
    assert shapes.param_shapes(20, 1280, 10, 65536) == oracle.param_shapes(cfg)


def test_d20_flop_convention_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "d20_pages.json")))
    assert g["rows_per_gpu"] * g["seq_len"] * 8 == g["tokens_per_step"]
    fpt = shapes.flops_per_token(20, 1280, 65536, 2048)
    assert abs(fpt - 3.492e9) / 3.492e9 < 1e-3
    total = fpt * g["iterations_approx"] * g["tokens_per_step"]
    assert abs(total / g["total_flops_approx"] - 1) < 0.05
    assert abs(g["chinchilla_tokens"] / g["tokens_per_step"] / g["iterations_approx"] - 1) < 0.01
