"""Greedy generation from the model, by its plain definition: no KV cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the
base model is run as an autocomplete on prompts; inference goes through an
Engine with a KV cache that implements prefill and decode.  A KV cache only
saves recomputation, so the oracle computes what it must equal: the logits
of the next token are the last row of the full forward over the sequence so
far, and greedy decoding appends their argmax (the lowest id among equal
maxima, as numpy's argmax).
"""

import numpy as np

from .model import forward


def logits_of(params, cfg, tokens):
    """Logits of every position of tokens [B, T]: the forward's z, [B, T, V]."""
    B, T = tokens.shape
    dummy_tgt = np.zeros_like(tokens)
    ones = np.ones(cfg.vocab, dtype=np.int64)
    _, _, cache = forward(params, cfg, tokens, dummy_tgt, ones)
    return cache["z"].reshape(B, T, cfg.vocab)


def next_logits(params, cfg, tokens):
    """Logits of the token after tokens [B, T]: [B, V]."""
    return logits_of(params, cfg, tokens)[:, -1, :]


def greedy(params, cfg, prompt, n_new):
    """Greedy continuation of prompt [B, T0] by n_new tokens: [B, n_new]."""
    seq = np.asarray(prompt)
    out = []
    for _ in range(n_new):
        nxt = np.argmax(next_logits(params, cfg, seq), axis=-1)
        out.append(nxt)
        seq = np.concatenate([seq, nxt[:, None]], axis=1)
    return np.stack(out, axis=1)


def teacher_forced_logits(params, cfg, prompt, continuation):
    """Logits that predict each token of continuation [B, n] given the prompt and the
    continuation's earlier tokens: [B, n, V] (row i predicts continuation[:, i])."""
    prompt = np.asarray(prompt)
    cont = np.asarray(continuation)
    seq = np.concatenate([prompt, cont[:, :-1]], axis=1)
    z = logits_of(params, cfg, seq)
    return z[:, prompt.shape[1] - 1:, :]
