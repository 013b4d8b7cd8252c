"""Batches built from a few distinct sequences, and the oracle's exact
expectation for them (test infrastructure, no method arithmetic of its own).

A full-size batch (32 x 2048 tokens at d20) is too large for the fp64 oracle,
but every row is an independent causal sequence and the loss is a mean over
rows.  So a batch whose row b holds sequence order[b] of k distinct Zipf
sequences has

    loss      = sum_j (c_j / B) loss_j
    gradients = sum_j (c_j / B) grad_j          (times grad_scale)
    bpb       = sum_j c_j S1_j / (ln 2 * sum_j c_j S2_j)

where c_j counts the rows holding sequence j and (S1_j, S2_j) are the
oracle's sums of nll over byte-counted targets and of bytes for sequence j
(bits per byte is a ratio of sums).  The oracle runs the k sequences once.
The row order is a seeded permutation, so neighbouring rows, tiles of rows
and the two halves of the batch all hold different sequences: a kernel that
reads or writes the wrong row gives a different answer.
"""

import functools
import math
from dataclasses import dataclass

import numpy as np

import oracle
from oracle.model import Config
from pretraining_step_03_b300 import synth
from tests._util import bf16_round


@dataclass
class Mixed:
    seq_tok: np.ndarray      # [k, T] int32
    seq_tgt: np.ndarray      # [k, T] int32
    order: np.ndarray        # [B] sequence index of each row

    @property
    def tokens(self):
        return np.ascontiguousarray(self.seq_tok[self.order])

    @property
    def targets(self):
        return np.ascontiguousarray(self.seq_tgt[self.order])

    def counts(self):
        return np.bincount(self.order, minlength=self.seq_tok.shape[0])


def mixed(counts, T, vocab, seq_seed=1, order_seed=0):
    """len(counts) distinct Zipf(1.1) sequences of T tokens, sequence j on counts[j]
    rows, the rows in a seeded, non-periodic order."""
    counts = np.asarray(counts)
    assert np.all(counts >= 1)
    tok, tgt = synth.zipf_rows(len(counts), T, vocab, seed=seq_seed)
    order = np.repeat(np.arange(len(counts)), counts)
    return Mixed(tok, tgt, np.random.default_rng(1000 + order_seed).permutation(order))


@dataclass
class SeqResult:
    loss: float
    sums: tuple              # (sum nll, sum nll over byte-counted targets, sum bytes)
    grads: dict              # param index -> fp64 gradient of the sequence's mean loss


def _sums(cache, token_bytes):
    nll = cache["nll"]
    nb = np.asarray(token_bytes, dtype=np.int64)[cache["tgt"]]
    return float(np.sum(nll)), float(np.sum(nll[nb > 0])), float(np.sum(nb))


@functools.lru_cache(maxsize=4)
def _oracle_sequences(cfg, param_seed, bf16, seq_key, keep, backward):
    """Oracle results for each sequence of a Mixed batch (cached per process, so the
    tests of one configuration share one oracle run)."""
    (k, T, vocab, seq_seed) = seq_key
    params = synth.init_params(cfg.depth, cfg.d_model, cfg.n_head, cfg.vocab, seed=param_seed)
    if bf16:
        params = [bf16_round(p) for p in params]
    tok, tgt = synth.zipf_rows(k, T, vocab, seed=seq_seed)
    tb = synth.token_bytes_binomial(vocab, seed=2)
    out = []
    for j in range(k):
        loss, _, cache = oracle.forward(params, cfg, tok[j:j + 1], tgt[j:j + 1], tb)
        grads = {}
        if backward:
            g = oracle.backward(cache, cfg)
            grads = {i: g[i] for i in keep}
            del g
        out.append(SeqResult(loss, _sums(cache, tb), grads))
        del cache
    return tuple(out)


def oracle_expectation(cfg, mix, param_seed=0, bf16=True, keep=(), backward=True, grad_scale=1.0,
                       seq_seed=1):
    """(loss, bpb, sums, grads) the oracle gives for the batch mix: exact combinations
    of its per-sequence results, grads restricted to the indices in keep."""
    k, T = mix.seq_tok.shape
    res = _oracle_sequences(cfg, param_seed, bf16, (k, T, cfg.vocab, seq_seed), tuple(sorted(keep)),
                            backward)
    c = mix.counts().astype(np.float64)
    B = float(c.sum())
    loss = float(sum(c[j] / B * r.loss for j, r in enumerate(res)))
    sums = tuple(float(sum(c[j] * r.sums[s] for j, r in enumerate(res))) for s in range(3))
    bpb = sums[1] / (math.log(2.0) * sums[2])
    grads = {i: sum(grad_scale * c[j] / B * r.grads[i] for j, r in enumerate(res)) for i in keep} if backward else {}
    return loss, bpb, sums, grads


def d20_config():
    return Config(20, 1280, 10, 65536)


# The d20 full-size batch of the step, evaluation and decode tests, and the
# gradients they compare: wte | L0 wq, wv | L0 w1 | L0 w2 | L10 wo | L19 w2 | lm_head.
D20_KEEP = (0, 1, 3, 5, 6, 1 + 6 * 10 + 3, 1 + 6 * 19 + 5, 6 * 20 + 1)


def d20_mix(T=2048):
    """32 rows: three sequences on 14, 11 and 7 rows."""
    return mixed((14, 11, 7), T, 65536, seq_seed=1, order_seed=0)


# ---------------------------------------------------------------- deeper models
# d26 and d30 (section 该你了: the device batch falls to 16 rows and two
# accumulation micro-steps keep the optimizer batch): the expectations are
# stored by tests/golden/make_depth_expectations.py, which runs only the
# oracle, because three d30 sequences take the fp64 oracle minutes.
DEPTH_CONFIGS = {
    "d26": Config(26, 1664, 13, 65536),
    "d30": Config(30, 1920, 15, 65536),
}
DEPTH_B, DEPTH_T, DEPTH_MICRO = 16, 2048, 2


def depth_keep(depth):
    """Tensors compared: wte | L0 wq, wv, wo, w1, w2 | middle wq | last w1, w2 | lm_head."""
    mid, last = depth // 2, depth - 1
    return (0, 1, 3, 4, 5, 6, 1 + 6 * mid, 1 + 6 * last + 4, 1 + 6 * last + 5, 6 * depth + 1)


DEPTH_COUNTS = ((8, 5, 3), (3, 6, 7))   # rows per sequence in micro-batch 0 and 1 (16 each)


def depth_mixes(cfg):
    """The micro-batches: the same three sequences, in other proportions and row orders."""
    return [mixed(DEPTH_COUNTS[m], DEPTH_T, cfg.vocab, seq_seed=1, order_seed=10 + m) for m in range(DEPTH_MICRO)]


def sample_index(shape, i, rows=None, n=2048):
    """Flat indices compared for tensor i: n seeded entries (restricted to the given rows,
    e.g. the token ids present, when rows is not None) and the whole last row, where
    ragged tiles end."""
    r, c = shape
    rng = np.random.default_rng(500 + i)
    rr = rng.integers(0, r, n) if rows is None else np.asarray(rows)[rng.integers(0, len(rows), n)]
    cc = rng.integers(0, c, n)
    last = rows[-1] if rows is not None else r - 1
    flat = np.concatenate([rr.astype(np.int64) * c + cc, int(last) * c + np.arange(c, dtype=np.int64)])
    return flat


def depth_sample_rows(cfg, i, mixes):
    """Rows worth sampling for tensor i: the token ids present for wte, all rows otherwise."""
    if i != 0:
        return None
    return np.unique(np.concatenate([m.seq_tok.ravel() for m in mixes]))
