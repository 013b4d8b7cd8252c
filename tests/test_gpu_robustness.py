"""Robustness on the GPU without faulting it: nothing is written outside the
caller's buffers (canary guard bands around the model arena and around the
outputs of the kernel-level entry points), and a bounded wait that runs out
is reported through the flag word while the context stays usable."""

import numpy as np
import pytest

from pretraining_step_03_b300 import synth
from tests._util import bf16_round

pytestmark = pytest.mark.gpu

GUARD = 1 << 20      # bytes of canary on each side
CANARY = 0xA5


def _guarded(torch, nbytes, dev):
    """A uint8 buffer with GUARD canary bytes on each side of an nbytes interior (256-aligned)."""
    buf = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=dev)
    return buf, buf.data_ptr() + GUARD


def _guards_intact(buf, nbytes):
    g = buf.cpu().numpy()
    return bool(np.all(g[:GUARD] == CANARY)) and bool(np.all(g[GUARD + nbytes:] == CANARY))


def test_model_step_stays_inside_its_arena():
    """A whole step (forward, backward with the norm backward in the GEMM epilogues, Muon,
    AdamW) at CTA-pair widths with a ragged last row tile writes nothing outside the arena."""
    import torch
    from pretraining_step_03_b300 import _lib as L
    depth, d, h, v, b, t = 2, 256, 2, 4096, 2, 200
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    nbytes = L.nc_arena_bytes(depth, d, h, v, b, t, L.NC_BF16)
    buf, arena = _guarded(torch, nbytes, dev)
    m = L.nc_init_model(depth, d, h, v, 7, arena, nbytes, L.NC_BF16, b, t, s)
    tok, tgt = synth.zipf_rows(b, t, v, seed=3)
    tb = synth.token_bytes_binomial(v, seed=2)
    tk, tg, tbd = (torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(dev) for x in (tok, tgt, tb))
    out = torch.zeros(2, dtype=torch.float32, device=dev)
    for step in (1, 2):
        L.nc_forward_backward(m, tk.data_ptr(), tg.data_ptr(), tbd.data_ptr(), b, t, 0, 1.0, out.data_ptr())
        L.nc_muon_step(m, 0.02, 0.95, 1, 5, (3.4445, -4.7750, 2.0315))
        L.nc_adamw_step(m, 0.2, 0.004, 0.9, 0.95, 1e-8, 0.0, step)
    torch.cuda.synchronize()
    assert L.nc_check_device_flag(m) == 0
    assert np.all(np.isfinite(out.cpu().numpy()))
    L.nc_free(m)
    assert _guards_intact(buf, nbytes)


def test_kernel_entry_points_stay_inside_their_outputs():
    """The GEMM (ragged CTA-pair tiles, fp32 and bf16 C) and the attention forward and
    backward write only their output matrices."""
    import torch
    from pretraining_step_03_b300 import _lib as L
    dev = torch.device("cuda")
    s = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(0)
    # GEMM: C[M, N] = A[M, K] B[N, K]^T, C in a guarded buffer
    M, N, K = 520, 776, 200
    a = torch.from_numpy(bf16_round(rng.normal(size=(M, K)))).to(dev, torch.bfloat16)
    bm = torch.from_numpy(bf16_round(rng.normal(size=(N, K)))).to(dev, torch.bfloat16)
    for cdt, es in ((L.NC_FP32, 4), (L.NC_BF16, 2)):
        nbytes = M * N * es
        buf, c = _guarded(torch, nbytes, dev)
        L.nc_gemm_bf16(M, N, K, 1, a.data_ptr(), K, 0, 0, bm.data_ptr(), K, 0, 0, c, N, 0, cdt, 1.0, 0.0, 0,
                       0, s)
        torch.cuda.synchronize()
        assert _guards_intact(buf, nbytes), cdt
    # attention (head dim 128, ragged T) with O, lse, dq, dk, dv in guarded buffers
    B, T, H, D = 2, 200, 3, 128
    q, k, vv, do = (torch.from_numpy(bf16_round(rng.normal(size=(B, T, H, D)).astype(np.float32))).to(
        dev, torch.bfloat16) for _ in range(4))
    nb = B * T * H * D * 2
    bo, o = _guarded(torch, nb, dev)
    bl, lse = _guarded(torch, B * H * T * 4, dev)
    L.nc_attention_forward(q.data_ptr(), k.data_ptr(), vv.data_ptr(), H * D, o, H * D, lse, B, T, H, D, L.NC_BF16, s)
    ws = torch.empty(L.nc_attention_workspace_bytes(B, T, H), dtype=torch.uint8, device=dev)
    outs = [_guarded(torch, nb, dev) for _ in range(3)]
    L.nc_attention_backward(q.data_ptr(), k.data_ptr(), vv.data_ptr(), H * D, o, do.data_ptr(), H * D, lse,
                            outs[0][1], outs[1][1], outs[2][1], H * D, ws.data_ptr(), B, T, H, D, L.NC_BF16, s)
    torch.cuda.synchronize()
    assert L.nc_check_kernel_flag(s) == 0
    assert _guards_intact(bo, nb) and _guards_intact(bl, B * H * T * 4)
    for buf, _ in outs:
        assert _guards_intact(buf, nb)


def test_wait_that_runs_out_is_flagged_and_context_survives():
    """A kernel whose mbarrier wait can never complete gives up after the library's wait
    limit, sets NC_FLAG_TIMEOUT and returns; the next launches on the context still run."""
    import torch
    from pretraining_step_03_b300 import _lib as L
    s = torch.cuda.current_stream().cuda_stream
    assert L.nc_check_kernel_flag(s) == 0
    L.nc_selftest_wait_timeout(s)
    assert L.nc_check_kernel_flag(s) == L.NC_FLAG_TIMEOUT
    assert L.nc_check_kernel_flag(s) == 0   # reading clears it
    # the context is intact: a GEMM after the aborted kernel gives the right product
    dev = torch.device("cuda")
    rng = np.random.default_rng(1)
    a = bf16_round(rng.normal(size=(300, 64)))
    bm = bf16_round(rng.normal(size=(280, 64)))
    A = torch.from_numpy(a).to(dev, torch.bfloat16)
    Bm = torch.from_numpy(bm).to(dev, torch.bfloat16)
    C = torch.zeros(300, 280, dtype=torch.float32, device=dev)
    L.nc_gemm_bf16(300, 280, 64, 1, A.data_ptr(), 64, 0, 0, Bm.data_ptr(), 64, 0, 0, C.data_ptr(), 280, 0,
                   L.NC_FP32, 1.0, 0.0, 0, 0, s)
    torch.cuda.synchronize()
    ref = a.astype(np.float64) @ bm.astype(np.float64).T
    assert np.max(np.abs(C.cpu().numpy() - ref)) / np.max(np.abs(ref)) <= 1e-4
    assert L.nc_check_kernel_flag(s) == 0
