"""Writes the oracle's expectations for the d26 and d30 step tests.

    python -m tests.golden.make_depth_expectations d30 d26

Runs only the fp64 oracle (oracle/) on the seeded synthetic inputs of
tests/_mix.py: the model of the nanochat walkthrough's depth section
(lyylswood.com, section 该你了: depth 26 and 30, device batch 16 x 2048, two
gradient-accumulation micro-steps), three distinct Zipf sequences spread over
the 16 rows of each micro-batch.  For each configuration it stores, in
tests/golden/<name>_mix.npz:

  loss[m], bpb[m], sums[m]   the oracle's mean loss, bits per byte and the sums
                             {nll, nll over byte-counted targets, bytes} of
                             micro-batch m (count-weighted over the sequences)
  g<i>                       the accumulated gradient of tensor i,
                             sum_m (1/2) grad(mean loss of micro-batch m),
                             at the flat indices tests/_mix.sample_index gives

Each sequence takes the oracle about three minutes at d30 and ~45 GB of host
memory, so the sequences run one after another.
"""

import os
import sys
import time

import numpy as np

import oracle
from pretraining_step_03_b300 import synth
from tests import _mix
from tests._util import bf16_round

HERE = os.path.dirname(os.path.abspath(__file__))


def path(name):
    return os.path.join(HERE, f"{name}_mix.npz")


def make(name):
    cfg = _mix.DEPTH_CONFIGS[name]
    mixes = _mix.depth_mixes(cfg)
    keep = _mix.depth_keep(cfg.depth)
    params = synth.init_params(cfg.depth, cfg.d_model, cfg.n_head, cfg.vocab, seed=0)
    for i in range(len(params)):
        params[i] = bf16_round(params[i])
    tb = synth.token_bytes_binomial(cfg.vocab, seed=2)
    shapes = {i: params[i].shape for i in keep}
    idx = {i: _mix.sample_index(shapes[i], i, _mix.depth_sample_rows(cfg, i, mixes)) for i in keep}
    seq_tok, seq_tgt = mixes[0].seq_tok, mixes[0].seq_tgt
    k = seq_tok.shape[0]
    per = []
    for j in range(k):
        t0 = time.time()
        loss, _, cache = oracle.forward(params, cfg, seq_tok[j:j + 1], seq_tgt[j:j + 1], tb)
        sums = _mix._sums(cache, tb)
        g = oracle.backward(cache, cfg)
        del cache
        per.append((loss, sums, {i: g[i].ravel()[idx[i]] for i in keep}))
        del g
        print(f"{name}: sequence {j} in {time.time() - t0:.0f} s", flush=True)
    out = {}
    loss_m, bpb_m, sums_m = [], [], []
    acc = {i: 0.0 for i in keep}
    for mix in mixes:
        c = mix.counts().astype(np.float64)
        B = c.sum()
        loss_m.append(sum(c[j] / B * per[j][0] for j in range(k)))
        s = [sum(c[j] * per[j][1][q] for j in range(k)) for q in range(3)]
        sums_m.append(s)
        bpb_m.append(s[1] / (np.log(2.0) * s[2]))
        for i in keep:
            acc[i] = acc[i] + sum(c[j] / B / len(mixes) * per[j][2][i] for j in range(k))
    out["loss"] = np.array(loss_m)
    out["bpb"] = np.array(bpb_m)
    out["sums"] = np.array(sums_m)
    for i in keep:
        out[f"g{i}"] = acc[i].astype(np.float32)
    np.savez_compressed(path(name), **out)
    print(f"wrote {path(name)}", flush=True)


if __name__ == "__main__":
    for name in sys.argv[1:] or ["d30", "d26"]:
        make(name)
