"""Parity of the evaluation pass (forward, loss and bits per byte, no backward).

nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the run
reports validation bits per byte from time to time.  nc_eval_loss keeps the
running sums {sum nll, sum nll over byte-counted targets, sum bytes}, so bpb
over several batches is the corpus ratio of sums.

Checks: the sums over two batches against the oracle's (relative error
<= 1e-5 in fp32 mode, 1e-3 in bf16 mode, as the loss); the batch's
{loss, bpb} bit-identical to what the training pass reports for the same
batch and weights; gradients and weights untouched (bit for bit).  At the
benchmark's d20 size (32 x 2048) the batch holds three distinct Zipf
sequences in a non-periodic row order, and the expected sums are the
count-weighted sums of the oracle's per-sequence sums.
"""

import math

import numpy as np
import pytest

import oracle
from oracle.model import Config
from pretraining_step_03_b300 import synth
from tests import _mix
from tests._util import bf16_round

pytestmark = pytest.mark.gpu

DEPTH, D, H, V, B, T = 2, 128, 2, 512, 4, 64
CFG = Config(DEPTH, D, H, V)
REL = {"fp32": 1e-5, "bf16": 1e-3}


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_tiny_eval_sums_and_no_side_effects(mode):
    import torch
    from pretraining_step_03_b300.model import Model
    params = synth.init_params(DEPTH, D, H, V, seed=0)
    tok_a, tgt_a = synth.uniform_rows(B, T, V, seed=1)
    tok_b, tgt_b = synth.uniform_rows(B, T, V, seed=11)
    tb = synth.token_bytes_uniform(V, 1, 8, seed=2)
    tb[tgt_b[0, 3]] = 0                        # one target that counts for no bytes
    m = Model(DEPTH, D, H, V, B, T, dtype=mode)
    m.set_params(params)
    dt = m.device_i32
    rng = np.random.default_rng(4)
    pattern = [rng.normal(0, 1, s).astype(np.float32) for s in m.shapes]
    for i, g in enumerate(pattern):
        m.set_grad(i, g)
    w_before = [m.get_param(i) for i in range(m.n_params)]
    out = torch.zeros(2, dtype=torch.float32, device=m.device)
    sums = m.eval_loss(dt(tok_a), dt(tgt_a), dt(tb), B, T, accumulate=0)
    m.eval_loss(dt(tok_b), dt(tgt_b), dt(tb), B, T, accumulate=1, sums=sums, out=out)
    torch.cuda.synchronize()
    got = sums.cpu().numpy()
    batch = out.cpu().numpy().copy()
    assert m.check_flag() == 0
    for i in range(m.n_params):
        assert np.array_equal(m.get_grad(i), pattern[i]), f"eval touched gradient {i}"
        assert np.array_equal(m.get_param(i), w_before[i]), f"eval touched weight {i}"
    op = [bf16_round(p) for p in params] if mode == "bf16" else params
    ra = oracle.eval_sums(op, CFG, tok_a, tgt_a, tb)
    rb = oracle.eval_sums(op, CFG, tok_b, tgt_b, tb)
    ref = [ra[k] + rb[k] for k in range(3)]
    assert got[2] == ref[2]                    # integer byte count: exact
    for k in range(2):
        assert abs(got[k] - ref[k]) / abs(ref[k]) <= REL[mode], (k, got[k], ref[k])
    bpb = got[1] / (math.log(2.0) * got[2])
    assert abs(bpb - oracle.bpb_of_sums(ref)) / oracle.bpb_of_sums(ref) <= REL[mode]
    # the same batch through the training pass reports the same bits
    fb = m.forward_backward(dt(tok_b), dt(tgt_b), dt(tb), B, T)
    torch.cuda.synchronize()
    assert np.array_equal(fb.cpu().numpy(), batch), (fb.cpu().numpy(), batch)


def test_d20_eval_full_size_distinct_rows():
    """The d20 evaluation pass at 32 x 2048: three distinct Zipf sequences over the
    32 rows (tests/_mix.py), so the sums are exact count-weighted sums of the
    oracle's per-sequence sums."""
    import torch
    from pretraining_step_03_b300.model import Model
    depth, d, h, v, Bf, Tf = 20, 1280, 10, 65536, 32, 2048
    mix = _mix.d20_mix(Tf)
    params = synth.init_params(depth, d, h, v, seed=0)
    tb = synth.token_bytes_binomial(v, seed=2)
    m = Model(depth, d, h, v, Bf, Tf, dtype="bf16")
    m.set_params(params)
    dt = m.device_i32
    tok, tgt = dt(mix.tokens), dt(mix.targets)
    out = torch.zeros(2, dtype=torch.float32, device=m.device)
    sums = m.eval_loss(tok, tgt, dt(tb), Bf, Tf, out=out)
    torch.cuda.synchronize()
    got = sums.cpu().numpy()
    batch = out.cpu().numpy().copy()
    fb = m.forward_backward(tok, tgt, dt(tb), Bf, Tf)
    torch.cuda.synchronize()
    assert np.array_equal(fb.cpu().numpy(), batch)
    assert m.check_flag() == 0
    m.close()
    del m
    torch.cuda.empty_cache()
    _, ref_bpb, ref, _ = _mix.oracle_expectation(_mix.d20_config(), mix, keep=_mix.D20_KEEP)
    assert got[2] == ref[2]                    # integer byte count: exact
    for k in range(2):
        assert abs(got[k] - ref[k]) / abs(ref[k]) <= 1e-3, (k, got[k], ref[k])
    assert abs(batch[1] - ref_bpb) / ref_bpb <= 1e-3, (batch[1], ref_bpb)
