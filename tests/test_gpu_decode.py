"""Parity of inference with a KV cache (prefill + greedy decode) against the
oracle's cache-free definition.

nanochat speedrun walkthrough (lyylswood.com), section 预搜检: the base model
is sampled through an Engine with a KV cache that implements prefill and
decode.  The oracle computes what the cache must reproduce: the logits of the
next token are the last row of the full forward over the sequence so far.

Checks, with the GPU's own greedy tokens fed to the oracle (teacher forcing):
  * the logits of every step: cosine >= 0.99999 / max|a-b|/max|b| <= 1e-4
    (fp32 mode), 0.999 / 2e-2 (bf16 mode);
  * each greedy token is the argmax of the GPU's own logits (ties to the
    lowest id), an argmax of the oracle's logits within delta = 2 * rel * max|z|,
    and equal to the oracle's argmax wherever the oracle's top-2 margin exceeds
    delta (several tokens are correct only inside that band);
  * the cached k (after RoPE) and v against the oracle's;
  * an identity model (zero blocks, orthonormal tied embeddings) repeats the
    prompt's last token exactly;
  * the d20 model at full size, 32 prompts of 512 tokens made of three
    distinct prompts in a non-periodic row order: rows with the same prompt
    generate the same tokens, and each prompt's logits match the oracle's.
"""

import numpy as np
import pytest

import oracle
from oracle import generate as og
from oracle.model import Config
from pretraining_step_03_b300 import synth
from tests import _mix
from tests._util import assert_close, bf16_round

pytestmark = pytest.mark.gpu

TOL = {"fp32": (0.99999, 1e-4), "bf16": (0.999, 2e-2)}


def _run(m, params_cfg, prompt, n_new, cache_B, cache_T):
    import torch
    B, T0 = prompt.shape
    cache = m.kv_cache(cache_B, cache_T)
    logits = torch.zeros(n_new, B, m.vocab, dtype=torch.float32, device=m.device)
    nxt = torch.zeros(n_new, B, dtype=torch.int32, device=m.device)
    m.prefill(cache, m.device_i32(prompt), B, T0, logits=logits[0], next_tok=nxt[0])
    for i in range(1, n_new):
        m.decode_step(cache, nxt[i - 1], B, T0 + i - 1, logits=logits[i], next_tok=nxt[i])
    torch.cuda.synchronize()
    assert m.check_flag() == 0
    return cache, logits.cpu().numpy().transpose(1, 0, 2), nxt.cpu().numpy().T.astype(np.int64)


def _check_tokens(tok, z_gpu, z_ref, rel):
    for b in range(tok.shape[0]):
        for i in range(tok.shape[1]):
            t = tok[b, i]
            assert t == int(np.argmax(z_gpu[b, i])), (b, i)        # the GPU's own argmax, lowest id on ties
            ref = z_ref[b, i]
            delta = 2 * rel * np.max(np.abs(ref))
            assert ref[t] >= ref.max() - delta, (b, i, ref[t], ref.max())
            top2 = np.sort(ref)[-2:]
            if top2[1] - top2[0] > delta:
                assert t == int(np.argmax(ref)), (b, i)


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T0,n_new", [(3, 37, 20), (4, 1, 6)])
def test_prefill_decode_against_oracle(mode, B, T0, n_new):
    from pretraining_step_03_b300.model import Model
    depth, d, H, V = 2, 256, 2, 512
    cfg = Config(depth, d, H, V)
    params = synth.init_params(depth, d, H, V, seed=0)
    params = [p * 4.0 for p in params]            # sharper softmaxes than the 0.02 init
    prompt = np.random.default_rng(5 + T0).integers(0, V, (B, T0))
    m = Model(depth, d, H, V, 4, 64, dtype=mode)
    m.set_params(params)
    cache, z_gpu, tok = _run(m, cfg, prompt, n_new, 4, 64)
    op = [bf16_round(p) for p in params] if mode == "bf16" else params
    z_ref = og.teacher_forced_logits(op, cfg, prompt, tok)
    cos, rel = TOL[mode]
    for i in range(n_new):
        assert_close(z_gpu[:, i], z_ref[:, i], cos, rel, f"{mode} step {i} logits")
    _check_tokens(tok, z_gpu, z_ref, rel)
    # the cache holds k (after RoPE) and v of every position written so far
    import torch
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    kv = cache.buf.view(dt).float().cpu().numpy().reshape(depth, 2, 4, 64, d)
    seq = np.concatenate([prompt, tok[:, :-1]], axis=1)
    _, _, oc = oracle.forward(op, cfg, seq, np.zeros_like(seq), np.ones(V, dtype=np.int64))
    n = seq.shape[1]
    for l in range(depth):
        assert_close(kv[l, 0, :B, :n], oc["layers"][l]["k"].reshape(B, n, d), cos, rel, f"{mode} cached k {l}")
        assert_close(kv[l, 1, :B, :n], oc["layers"][l]["v"].reshape(B, n, d), cos, rel, f"{mode} cached v {l}")


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_identity_model_repeats_last_token(mode):
    from pretraining_step_03_b300.model import Model
    depth, d, H, V = 1, 128, 1, 64
    rng = np.random.default_rng(2)
    q, _ = np.linalg.qr(rng.normal(size=(d, d)))
    wte = q[:V] * 3.0
    shapes = oracle.param_shapes(Config(depth, d, H, V))
    params = [wte] + [np.zeros(s) for s in shapes[1:-1]] + [wte.copy()]
    prompt = rng.integers(0, V, (3, 6))
    m = Model(depth, d, H, V, 4, 32, dtype=mode)
    m.set_params(params)
    out = m.generate(m.kv_cache(4, 32), m.device_i32(prompt).reshape(3, 6), 7)
    got = out.cpu().numpy().T
    assert np.array_equal(got, np.repeat(prompt[:, -1:], 7, axis=1)), got


def test_argument_checks():
    from pretraining_step_03_b300 import _lib as L
    from pretraining_step_03_b300.model import Model
    import torch
    m = Model(1, 128, 1, 64, 4, 32, dtype="bf16")
    cache = m.kv_cache(4, 32)
    tok = torch.zeros(4, dtype=torch.int32, device=m.device)
    with pytest.raises(L.NcError):
        m.decode_step(cache, tok, 4, 32)                 # pos == cache_T
    with pytest.raises(L.NcError):
        m.decode_step(cache, tok, 5, 0)                  # B > cache_B
    big = m.kv_cache(4, 64)                              # cache_T > the model's max_T
    with pytest.raises(L.NcError):
        m.prefill(big, tok, 1, 4)
    with pytest.raises(L.NcError):
        m.prefill(cache, tok, 1, 33)                     # T0 > cache_T
    assert m.check_flag() == 0


def test_d20_full_size_distinct_prompts():
    """d20 at full size: 32 prompts of 512 tokens, three distinct Zipf prompts in a
    non-periodic row order (tests/_mix.py).  Rows that hold the same prompt must
    generate the same tokens, and each of the three against the oracle."""
    import torch
    from pretraining_step_03_b300.model import Model
    depth, d, H, V, B, T0, n_new = 20, 1280, 10, 65536, 32, 512, 8
    params = synth.init_params(depth, d, H, V, seed=0)
    mix = _mix.mixed((9, 13, 10), T0, V, seq_seed=1, order_seed=2)
    m = Model(depth, d, H, V, B, 2048, dtype="bf16")
    m.set_params(params)
    cache, z_gpu, tok = _run(m, None, mix.tokens, n_new, B, 1024)
    m.close()
    del m, cache
    torch.cuda.empty_cache()
    first = [int(np.flatnonzero(mix.order == j)[0]) for j in range(3)]
    for b in range(B):
        assert np.array_equal(tok[b], tok[first[mix.order[b]]]), f"row {b} differs from its prompt's first row"
    z_ref = og.teacher_forced_logits([bf16_round(p) for p in params], Config(depth, d, H, V), mix.seq_tok,
                                     tok[first])
    for j, b in enumerate(first):
        for i in range(n_new):
            assert_close(z_gpu[b, i], z_ref[j, i], 0.999, 2e-2, f"d20 prompt {j} (row {b}) step {i} logits")
    _check_tokens(tok[first], z_gpu[first], z_ref, 2e-2)


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_replayed_steps_equal_direct_launches(mode):
    """Decode steps replayed from a recorded CUDA graph give the same bits as direct
    launches (two fixed token buffers in turn; 10 steps, so 8 are replays)."""
    import torch
    from pretraining_step_03_b300.model import Model
    depth, d, H, V, B, T0, steps = 2, 256, 2, 512, 3, 9, 10
    params = [p * 4.0 for p in synth.init_params(depth, d, H, V, seed=0)]
    prompt = np.random.default_rng(8).integers(0, V, (B, T0))
    results = []
    for graphs in (True, False):
        m = Model(depth, d, H, V, 4, 64, dtype=mode)
        m.set_params(params)
        m.decode_graphs(graphs)
        cache = m.kv_cache(4, 64)
        buf = [torch.zeros(B, dtype=torch.int32, device=m.device) for _ in range(2)]
        logits = torch.zeros(B, V, dtype=torch.float32, device=m.device)
        m.prefill(cache, m.device_i32(prompt), B, T0, next_tok=buf[0])
        seen = []
        for i in range(steps):
            m.decode_step(cache, buf[i % 2], B, T0 + i, logits=logits, next_tok=buf[(i + 1) % 2])
            seen.append((logits.cpu().numpy().copy(), buf[(i + 1) % 2].cpu().numpy().copy()))
        assert m.check_flag() == 0
        results.append(seen)
        m.close()
    for i, ((za, ta), (zb, tb)) in enumerate(zip(*results)):
        assert np.array_equal(za, zb), f"{mode} step {i}: logits differ"
        assert np.array_equal(ta, tb), f"{mode} step {i}: tokens differ"
