"""The pages' whole optimizer step: accumulated micro-batches and the run's
learning-rate schedule, through nc_train_step from host buffers.

nanochat speedrun walkthrough (lyylswood.com), section 预搜检: one optimizer
step takes 32 x 2048 x 8 = 524,288 tokens (eight accumulated micro-batches on
one GPU), the learning rate scales as 1/sqrt(dim) and lrm falls linearly to 0
near the end of the run.  Tiny configuration (depth 2, d_model 128, vocab
512, 8 micro-batches of 4 x 64), learning rates from the library's schedule on
the device side and from the oracle's on the other.

Tolerances: accumulated gradients cosine >= 0.99999 / max-rel <= 1e-4 (fp32)
and 0.999 / 2e-2 (bf16); the reported mean loss and bpb relative error
<= 1e-5 / 1e-3; the loss after the step (weights moved by Muon and AdamW)
<= 1e-4 (fp32: the gradient differences pass through Newton-Schulz) / 2e-3
(bf16).
"""

import numpy as np
import pytest

import oracle
from oracle import schedule as osched
from oracle.model import Config
from pretraining_step_03_b300 import synth
from tests._util import assert_close, bf16_round

pytestmark = pytest.mark.gpu

DEPTH, D, H, V, B, T, NM = 2, 128, 2, 512, 4, 64, 8
CFG = Config(DEPTH, D, H, V)
BASE = (0.02, 0.2, 0.004)       # Muon, embedding, unembedding at the reference width
D_REF = 256                     # so the AdamW rates are scaled by sqrt(2)
RUN, WARMDOWN, STEP = 10, 0.5, 7   # step 7 of 10 lies in the warm-down: lrm = 0.6
HPX = dict(momentum=0.95, beta1=0.8, beta2=0.95, eps=1e-10, wd=0.0)
TOL = {"fp32": dict(gcos=0.99999, grel=1e-4, loss=1e-5, after=1e-4),
       "bf16": dict(gcos=0.999, grel=2e-2, loss=1e-3, after=2e-3)}


@pytest.fixture(scope="module")
def data():
    params = synth.init_params(DEPTH, D, H, V, seed=0)
    tok, tgt = synth.uniform_rows(NM * B, T, V, seed=21)
    tb = synth.token_bytes_uniform(V, 1, 8, seed=2)
    return params, tok.reshape(NM, B, T), tgt.reshape(NM, B, T), tb


def _oracle_micro(op, tok, tgt, tb):
    losses, bpbs, grads = [], [], None
    for j in range(NM):
        l, b, g = oracle.loss_and_grads(op, CFG, tok[j], tgt[j], tb, grad_scale=1.0 / NM)
        losses.append(l)
        bpbs.append(b)
        grads = g if grads is None else [a + c for a, c in zip(grads, g)]
    return float(np.mean(losses)), float(np.mean(bpbs)), grads


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_eight_micro_batch_accumulation(mode, data):
    from pretraining_step_03_b300.model import Model
    params, tok, tgt, tb = data
    m = Model(DEPTH, D, H, V, B, T, dtype=mode)
    m.set_params(params)
    dt = m.device_i32
    for j in range(NM):
        m.forward_backward(dt(tok[j]), dt(tgt[j]), dt(tb), B, T, accumulate=int(j > 0), grad_scale=1.0 / NM)
    op = [bf16_round(p) for p in params] if mode == "bf16" else params
    _, _, ref = _oracle_micro(op, tok, tgt, tb)
    for i in range(m.n_params):
        assert_close(m.get_grad(i), ref[i], TOL[mode]["gcos"], TOL[mode]["grel"], f"{mode} 8-micro grad {i}")


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_scheduled_train_step_from_host_buffers(mode, data):
    import torch
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model
    params, tok, tgt, tb = data
    m = Model(DEPTH, D, H, V, B, T, dtype=mode)
    m.set_params(params)
    lr_m, lr_e, lr_u = L.nc_lr_schedule(STEP, RUN, WARMDOWN, D, D_REF, BASE)
    tb_d = m.device_i32(tb)
    loss, bpb = m.train_step(np.ascontiguousarray(tok.reshape(-1), dtype=np.int32),
                             np.ascontiguousarray(tgt.reshape(-1), dtype=np.int32), tb_d, B, T, NM,
                             lr_m, lr_e, lr_u, 1, HPX["momentum"], 5, beta1=HPX["beta1"],
                             beta2=HPX["beta2"], eps=HPX["eps"], weight_decay=HPX["wd"])
    out = torch.zeros(2, dtype=torch.float32, device=m.device)
    m.eval_loss(m.device_i32(tok[0]), m.device_i32(tgt[0]), tb_d, B, T, out=out)
    torch.cuda.synchronize()
    after = float(out.cpu().numpy()[0])
    assert m.check_flag() == 0
    op = [bf16_round(p) for p in params] if mode == "bf16" else params
    ref_loss, ref_bpb, g = _oracle_micro(op, tok, tgt, tb)
    tol = TOL[mode]
    assert abs(loss - ref_loss) / ref_loss <= tol["loss"], (loss, ref_loss)
    assert abs(bpb - ref_bpb) / ref_bpb <= tol["loss"], (bpb, ref_bpb)
    o_m, o_e, o_u = osched.learning_rates(STEP, RUN, WARMDOWN, D, D_REF, BASE)
    w = []
    for i, p in enumerate(params):
        p = np.asarray(p, dtype=np.float64)
        if i in (0, len(params) - 1):
            lr = o_e if i == 0 else o_u
            w.append(oracle.adamw_step(p, g[i], 0 * p, 0 * p, lr, HPX["beta1"], HPX["beta2"], HPX["eps"],
                                       HPX["wd"], 1)[0])
        else:
            w.append(oracle.muon_step(p, g[i], 0 * p, o_m, HPX["momentum"], True, 5)[0])
    if mode == "bf16":
        w = [bf16_round(x) for x in w]
    ref_after = oracle.forward(w, CFG, tok[0], tgt[0], tb)[0]
    assert abs(after - ref_after) / ref_after <= tol["after"], (after, ref_after)
