"""Muon and AdamW at the full d20 sizes against the fp64 oracle.

The optimizer step of the d20 model (bf16 mode): Muon over all 120 block
matrices (five bf16 Newton-Schulz iterations, the tall W1 matrices taken
through their transpose), AdamW on the 65536 x 1280 embedding and LM head.
Gradients are set on a sample of matrices (a square attention matrix, the
output projection, a tall W1, a wide W2, wte and lm_head); every other
matrix has a zero gradient and must stay unchanged.  Two steps, so the
momentum and Adam moments are exercised.  Tolerances are those of the tiny
optimizer test: weights cosine >= 0.999 and max-rel <= 2e-2; Muon's
orthogonalised update cos >= 0.999 against the oracle (these N(0, sigma)
gradients leave bf16 storage at ~0.99996, see tests/_util.py ns_bf16_model)
and, in the oracle's singular basis, within 0.1 of its singular values and
inside [0.6, 1.3] where those are >= 0.68; AdamW's update cos >= 0.999,
max-rel <= 2e-2.
"""

import numpy as np
import pytest

import oracle
from tests._util import assert_close, cmp, muon_update_cos_min

pytestmark = pytest.mark.gpu

DEPTH, D, H, V = 20, 1280, 10, 65536
HP = dict(muon_lr=0.02, momentum=0.95, lr_emb=0.2, lr_unemb=0.004, beta1=0.8, beta2=0.95, eps=1e-10,
          wd=0.0)
# wte | L0 wq | L0 wo | L7 w1 (5120 x 1280, tall) | L19 w2 (1280 x 5120, wide) | lm_head
SEL = [0, 1, 4, 1 + 6 * 7 + 4, 1 + 6 * 19 + 5, 6 * DEPTH + 1]
UNTOUCHED = [2, 1 + 6 * 10 + 0, 1 + 6 * 12 + 4]


def _muon_update_checks(prev, got, xref, geff, what):
    r, c = got.shape
    x = (prev - got) / (HP["muon_lr"] * np.sqrt(max(1.0, r / c)))
    cos, _ = cmp(x, xref)
    cmin, cmodel = muon_update_cos_min(geff, xref, cos=cos)
    assert cos >= cmin, f"{what}: Muon update cos {cos} (min {cmin}, bf16 storage model {cmodel})"
    u, sv, vt = np.linalg.svd(xref, full_matrices=False)
    proj = np.einsum("ki,kl,il->i", u, x, vt)
    sel = sv >= 0.68
    assert sel.any(), what
    assert np.all(np.abs(proj[sel] - sv[sel]) <= 0.1), (what, np.max(np.abs(proj[sel] - sv[sel])))
    assert np.all((proj[sel] >= 0.6) & (proj[sel] <= 1.3)), (what, proj[sel].min(), proj[sel].max())


def _optimizer_parity(depth, d, h, v, sel, untouched, seed):
    from pretraining_step_03_b300.model import Model
    m = Model(depth, d, h, v, 1, 128, dtype="bf16", seed=seed)
    rng = np.random.default_rng(7)
    last = 6 * depth + 1
    w = {i: m.get_param(i).astype(np.float64) for i in sel}
    still = {i: m.get_param(i) for i in untouched}
    buf = {i: np.zeros_like(w[i]) for i in sel}
    am = {i: np.zeros_like(w[i]) for i in sel}
    av = {i: np.zeros_like(w[i]) for i in sel}
    prev_g = {}
    for step in (1, 2):
        grads = {}
        for i in sel:
            g = rng.normal(0.0, 1e-3, w[i].shape).astype(np.float32)
            if step == 2:   # correlated with step 1 so the momentum matters
                g = (0.5 * prev_g[i] + g).astype(np.float32)
            grads[i] = g
            m.set_grad(i, g)
        prev_g = grads
        m.muon_step(HP["muon_lr"], HP["momentum"], True, 5)
        m.adamw_step(HP["lr_emb"], HP["lr_unemb"], HP["beta1"], HP["beta2"], HP["eps"], HP["wd"], step)
        for i in sel:
            g = grads[i].astype(np.float64)
            prev = w[i]
            if i in (0, last):
                lr = HP["lr_emb"] if i == 0 else HP["lr_unemb"]
                ref, am[i], av[i] = oracle.adamw_step(prev, g, am[i], av[i], lr, HP["beta1"], HP["beta2"],
                                                      HP["eps"], HP["wd"], step)
                got = m.get_param(i).astype(np.float64)
                assert_close(got, ref, 0.999, 2e-2, f"step {step} AdamW weight {i}")
                assert_close(got - prev, ref - prev, 0.999, 2e-2, f"step {step} AdamW update {i}")
            else:
                ref, buf[i], xref = oracle.muon_step(prev, g, buf[i], HP["muon_lr"], HP["momentum"], True, 5)
                got = m.get_param(i).astype(np.float64)
                assert_close(got, ref, 0.999, 2e-2, f"step {step} Muon weight {i}")
                _muon_update_checks(prev, got, xref, g + HP["momentum"] * buf[i],
                                    f"step {step} matrix {i} {got.shape}")
            w[i] = got   # both sides continue from the same weights
        for i in untouched:   # zero gradient: no update
            np.testing.assert_array_equal(m.get_param(i), still[i])
    assert m.check_flag() == 0


def test_d20_optimizer_step_matches_oracle():
    _optimizer_parity(DEPTH, D, H, V, SEL, UNTOUCHED, seed=3)


def test_ragged_width_optimizer_step_matches_oracle():
    """d_model 384 = 256 + 128: Newton-Schulz products with a ragged 256-tile edge
    (the symmetric products mirror full and partial 32 x 32 chunks)."""
    depth = 2
    sel = [0, 1, 1 + 4, 1 + 5, 6 + 1 + 3, 6 * depth + 1]
    _optimizer_parity(depth, 384, 3, 512, sel, [2, 6 + 1 + 1], seed=4)


def test_d30_optimizer_step_matches_oracle():
    """d30 widths (d_model 1920 = 7.5 x 256): square, tall and wide Newton-Schulz
    products with ragged 256-tile edges; AdamW on 65536 x 1920."""
    depth = 30
    sel = [0, 1, 1 + 3, 1 + 6 * 7 + 4, 1 + 6 * 29 + 5, 6 * depth + 1]
    _optimizer_parity(depth, 1920, 15, 65536, sel, [2, 1 + 6 * 15 + 4], seed=5)


def test_d20_muon_all_matrices_nesterov_normal_gradients():
    """The optimizer microbenchmark's Muon workload: N(0, 1) fp32 gradients on all 80
    square and 40 rectangular d20 matrices, zero momentum buffers (one momentum
    update, Nesterov), five bf16 Newton-Schulz iterations.  Every matrix's
    orthogonalised update against the fp64 oracle: cosine >= 0.999."""
    from pretraining_step_03_b300.model import Model
    m = Model(DEPTH, D, H, V, 1, 128, dtype="bf16", seed=6)
    rng = np.random.default_rng(11)
    mats = list(range(1, 6 * DEPTH + 1))
    w0, grads = {}, {}
    for i in mats:
        w0[i] = m.get_param(i).astype(np.float64)
        grads[i] = rng.normal(0.0, 1.0, w0[i].shape).astype(np.float32)
        m.set_grad(i, grads[i])
    lr = HP["muon_lr"]
    m.muon_step(lr, HP["momentum"], True, 5)
    cos = []
    for i in mats:
        got = m.get_param(i).astype(np.float64)
        r, c = got.shape
        x = (w0[i] - got) / (lr * np.sqrt(max(1.0, r / c)))
        _, _, xref = oracle.muon_step(w0[i], grads[i], np.zeros_like(w0[i]), lr, HP["momentum"], True, 5)
        cs, _ = cmp(x, xref)
        cos.append(cs)
        assert cs >= 0.999, f"matrix {i} {got.shape}: Muon update cos {cs}"
    assert m.check_flag() == 0
    sq = [c for i, c in zip(mats, cos) if (i - 1) % 6 < 4]
    rect = [c for i, c in zip(mats, cos) if (i - 1) % 6 >= 4]
    for name, v in (("square 1280x1280", sq), ("rectangular 1280x5120", rect)):
        print(f"Muon update cosine vs fp64, {name} ({len(v)} matrices): min {min(v):.6f} "
              f"median {float(np.median(v)):.6f} max {max(v):.6f}")
