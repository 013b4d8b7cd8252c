"""The deeper models of the depth sweep at their benchmark launch configuration.

nanochat speedrun walkthrough (lyylswood.com), section 该你了: depth is the
one size knob; at depth 26 and 30 the device batch falls to 16 rows of 2048
tokens and two gradient-accumulation micro-steps keep the optimizer batch.
d26: d_model 1664, 13 heads; d30: d_model 1920, 15 heads (head dim 128,
vocab 65536, bf16).  Neither width is a multiple of the 256-wide CTA-pair
tile, and 13 and 15 heads give attention grids of odd height, so these
configurations run ragged tiles everywhere the d20 step does not.

Each micro-batch holds three distinct Zipf sequences on 16 rows in a seeded,
non-periodic order, in different proportions in the two micro-batches
(tests/_mix.py).  The fp64 oracle's per-sequence results combine exactly
into each micro-batch's loss and bits per byte and into the accumulated
gradient; three d30 sequences take the oracle minutes, so those values were
written by tests/golden/make_depth_expectations.py (oracle only) and are
read here.  Tolerances as for the d20 step: loss and bpb relative error
<= 1e-3; gradients cosine >= 0.999, max-rel <= 2e-2, on each tensor's
stored sample (2048 seeded entries and the whole last row).  The step then
runs Muon and AdamW on those gradients (their parity at these widths given
identical gradients is tests/test_gpu_optim_full.py).
"""

import os

import numpy as np
import pytest

from pretraining_step_03_b300 import synth
from tests import _mix
from tests._util import assert_close

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", ["d26", "d30"])
def test_depth_step_two_micro_steps(name):
    import torch
    from pretraining_step_03_b300.model import Model
    cfg = _mix.DEPTH_CONFIGS[name]
    ref = np.load(os.path.join(GOLDEN, f"{name}_mix.npz"))
    mixes = _mix.depth_mixes(cfg)
    keep = _mix.depth_keep(cfg.depth)
    B, T = _mix.DEPTH_B, _mix.DEPTH_T
    tb = synth.token_bytes_binomial(cfg.vocab, seed=2)
    m = Model(cfg.depth, cfg.d_model, cfg.n_head, cfg.vocab, B, T, dtype="bf16")
    params = synth.init_params(cfg.depth, cfg.d_model, cfg.n_head, cfg.vocab, seed=0)
    for i, p in enumerate(params):
        m.set_param(i, p)
    shapes = {i: params[i].shape for i in keep}
    del params
    dt = m.device_i32
    outs = [torch.zeros(2, dtype=torch.float32, device=m.device) for _ in mixes]
    tbd = dt(tb)
    for k, mix in enumerate(mixes):
        m.forward_backward(dt(mix.tokens), dt(mix.targets), tbd, B, T, accumulate=int(k > 0),
                           grad_scale=1.0 / len(mixes), out=outs[k])
    torch.cuda.synchronize()
    assert m.check_flag() == 0
    for k, out in enumerate(outs):
        loss, bpb = out.cpu().numpy().astype(np.float64)
        assert abs(loss - ref["loss"][k]) / ref["loss"][k] <= 1e-3, (name, k, loss, ref["loss"][k])
        assert abs(bpb - ref["bpb"][k]) / ref["bpb"][k] <= 1e-3, (name, k, bpb, ref["bpb"][k])
    for i in keep:
        idx = _mix.sample_index(shapes[i], i, _mix.depth_sample_rows(cfg, i, mixes))
        assert_close(m.get_grad(i).ravel()[idx], ref[f"g{i}"], 0.999, 2e-2, f"{name} grad {i}")
    # the optimizer step on the accumulated gradients
    m.muon_step(0.02)
    m.adamw_step(0.2, 0.004, step=1)
    torch.cuda.synchronize()
    assert m.check_flag() == 0
    for i in (1, 1 + 6 * (cfg.depth - 1) + 5, 6 * cfg.depth + 1):
        assert np.all(np.isfinite(m.get_param(i)))
    m.close()
