"""The full d20 step at the benchmark's launch configuration (32 x 2048
tokens, 20 layers, d_model 1280, 10 heads of 128, vocab 65536, bf16).

The oracle cannot run 65,536 tokens through fp64 in a test, so the batch is
32 identical copies of one Zipf row: the mean loss, bits per byte and every
gradient of the batch then equal those of the single row, which the oracle
computes (T = 2048, about 30 s on the host).  Tolerances as for bf16 parity:
loss relative error <= 1e-3; gradients cosine >= 0.999, max-rel <= 2e-2.
"""

import numpy as np
import pytest

import oracle
from oracle.model import Config
from pretraining_step_03_b300 import synth
from tests._util import assert_close, bf16_round

pytestmark = pytest.mark.gpu


def test_d20_full_size_identical_rows():
    import torch
    from pretraining_step_03_b300.model import Model
    depth, d, h, v, B, T = 20, 1280, 10, 65536, 32, 2048
    params = synth.init_params(depth, d, h, v, seed=0)
    tok1, tgt1 = synth.zipf_rows(1, T, v, seed=1)
    tb = synth.token_bytes_binomial(v, seed=2)
    tok = np.repeat(tok1, B, axis=0)
    tgt = np.repeat(tgt1, B, axis=0)
    m = Model(depth, d, h, v, B, T, dtype="bf16")
    m.set_params(params)
    out = m.forward_backward(m.device_i32(tok), m.device_i32(tgt), m.device_i32(tb), B, T)
    torch.cuda.synchronize()
    loss, bpb = out.cpu().numpy().astype(np.float64)
    assert m.check_flag() == 0
    check = [0, 1, 4, 6, 1 + 6 * 10 + 3, 1 + 6 * 19 + 5, 6 * depth + 1]
    got = {i: m.get_grad(i) for i in check}
    m.close()
    del m
    torch.cuda.empty_cache()
    ref_loss, ref_bpb, ref_g = oracle.loss_and_grads([bf16_round(p) for p in params], Config(depth, d, h, v),
                                                     tok1, tgt1, tb)
    assert abs(loss - ref_loss) / ref_loss <= 1e-3, (loss, ref_loss)
    assert abs(bpb - ref_bpb) / ref_bpb <= 1e-3, (bpb, ref_bpb)
    for i in check:
        assert_close(got[i], ref_g[i], 0.999, 2e-2, f"d20 grad {i}")
