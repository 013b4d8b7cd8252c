"""The full d20 step at the benchmark's launch configuration (32 x 2048
tokens, 20 layers, d_model 1280, 10 heads of 128, vocab 65536, bf16).

The fp64 oracle cannot run 65,536 tokens in a test, so the batch holds three
distinct Zipf sequences spread over the 32 rows in a seeded, non-periodic
order (tests/_mix.py): the batch's mean loss, bits per byte and every
gradient are then exact count-weighted combinations of the three sequences'
oracle results, while a kernel that reads or writes the wrong batch row
(the GEMM M-tiles past row 2048, the attention grid's batch index, the
cross-entropy row, the embedding-backward segments) changes the answer.
Tolerances as for bf16 parity: loss and bpb relative error <= 1e-3;
gradients cosine >= 0.999, max-rel <= 2e-2.
"""

import numpy as np
import pytest

from tests import _mix
from tests._util import assert_close
from pretraining_step_03_b300 import synth

pytestmark = pytest.mark.gpu

DEPTH, D, H, V, B, T = 20, 1280, 10, 65536, 32, 2048
KEEP = _mix.D20_KEEP


def test_d20_full_size_distinct_rows():
    import torch
    from pretraining_step_03_b300.model import Model
    mix = _mix.d20_mix(T)
    assert len(set(mix.order[:8].tolist())) > 1 and not np.array_equal(mix.order[:16], mix.order[16:])
    params = synth.init_params(DEPTH, D, H, V, seed=0)
    tb = synth.token_bytes_binomial(V, seed=2)
    m = Model(DEPTH, D, H, V, B, T, dtype="bf16")
    m.set_params(params)
    out = m.forward_backward(m.device_i32(mix.tokens), m.device_i32(mix.targets), m.device_i32(tb), B, T)
    torch.cuda.synchronize()
    loss, bpb = out.cpu().numpy().astype(np.float64)
    assert m.check_flag() == 0
    got = {i: m.get_grad(i) for i in KEEP}
    m.close()
    del m
    torch.cuda.empty_cache()
    ref_loss, ref_bpb, _, ref_g = _mix.oracle_expectation(_mix.d20_config(), mix, keep=KEEP)
    assert abs(loss - ref_loss) / ref_loss <= 1e-3, (loss, ref_loss)
    assert abs(bpb - ref_bpb) / ref_bpb <= 1e-3, (bpb, ref_bpb)
    for i in KEEP:
        assert_close(got[i], ref_g[i], 0.999, 2e-2, f"d20 grad {i}")
