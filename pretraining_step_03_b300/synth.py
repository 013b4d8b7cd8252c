"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This module holds no arithmetic of the training step itself: only random
draws with the shapes and distributions of the pretraining workload
(nanochat speedrun walkthrough, lyylswood.com, section 预搜检: rows of 2048
tokens, 32 rows per GPU, a ~560M-parameter 20-layer model; tokenizer section:
about 4.8 characters per token).  FineWeb-EDU is not available, so a Zipf
token stream over the vocabulary stands in for it.
"""

import numpy as np

from .shapes import param_shapes


def init_params(depth, d_model, n_head, vocab, seed=0, std=0.02):
    """fp32 weights ~ N(0, std) in the library's parameter order."""
    rng = np.random.default_rng(seed)
    return [rng.normal(0.0, std, size=s).astype(np.float32)
            for s in param_shapes(depth, d_model, n_head, vocab)]


def zipf_rows(B, T, vocab, s=1.1, seed=1):
    """B rows of T+1 tokens, P(rank k) ~ k^-s over ranks 1..vocab.

    Ranks are mapped to token ids by a seeded permutation, so frequent ids
    are scattered over the vocabulary.  Returns (tokens, targets) int32
    [B, T] with targets = tokens shifted left by one.
    """
    rng = np.random.default_rng(seed)
    ranks = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(ranks ** (-s))
    cdf /= cdf[-1]
    u = rng.random((B, T + 1))
    idx = np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1)
    perm = rng.permutation(vocab)
    rows = perm[idx].astype(np.int32)
    return np.ascontiguousarray(rows[:, :T]), np.ascontiguousarray(rows[:, 1:])


def uniform_rows(B, T, vocab, seed=1):
    """B rows of T+1 tokens uniform in [0, vocab); (tokens, targets) as above."""
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, vocab, size=(B, T + 1), dtype=np.int64).astype(np.int32)
    return np.ascontiguousarray(rows[:, :T]), np.ascontiguousarray(rows[:, 1:])


def token_bytes_binomial(vocab, seed=2):
    """UTF-8 byte length per token id: 1 + Binomial(15, 3.8/15), range [1, 16], mean 4.8."""
    rng = np.random.default_rng(seed)
    return (1 + rng.binomial(15, 3.8 / 15, size=vocab)).astype(np.int32)


def token_bytes_uniform(vocab, lo=1, hi=8, seed=2):
    """Byte length per token id uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=vocab).astype(np.int32)


def normal(shape, seed, std=1.0, dtype=np.float32):
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, std, size=shape).astype(dtype)
