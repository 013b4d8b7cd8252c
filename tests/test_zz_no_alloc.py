"""The allocation-free attention backward against the workspace version.

nc_attention_backward_noalloc serves callers that cannot allocate device
memory (their device memory is reserved by another runtime, or they cannot
afford cudaMalloc's device-wide synchronisation): its row-statistics scratch
is a fixed array inside the library.  Two calls in a row, on different
inputs, must each match nc_attention_backward (caller workspace) within the
bf16 attention tolerance (cosine >= 0.999, max-rel <= 2e-2).  This file is
named to be collected last.
"""

import numpy as np
import pytest

from tests._util import assert_close

pytestmark = pytest.mark.gpu


def _inputs(seed, B, T, H, D):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    qkv = torch.randn(B * T, 3 * H * D, device="cuda", generator=g).to(torch.bfloat16)
    dout = torch.randn(B * T, H * D, device="cuda", generator=g).to(torch.bfloat16)
    return qkv, dout


def _forward(L, qkv, B, T, H, D, s):
    import torch
    o = torch.empty(B * T, H * D, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B, H, T, device="cuda", dtype=torch.float32)
    q, k, v = (qkv.data_ptr() + i * H * D * 2 for i in range(3))
    L.nc_attention_forward(q, k, v, 3 * H * D, o.data_ptr(), H * D, lse.data_ptr(), B, T, H, D, L.NC_BF16, s)
    return o, lse


def test_noalloc_backward_matches_workspace_version_twice():
    import torch
    from pretraining_step_03_b300 import _lib as L
    B, T, H, D = 2, 384, 4, 128
    s = torch.cuda.current_stream().cuda_stream
    for seed in (11, 12):   # two calls in a row, different inputs
        qkv, dout = _inputs(seed, B, T, H, D)
        o, lse = _forward(L, qkv, B, T, H, D, s)
        q, k, v = (qkv.data_ptr() + i * H * D * 2 for i in range(3))
        ref = torch.empty_like(qkv)
        got = torch.full_like(qkv, float("nan"))
        ws = torch.empty(L.nc_attention_workspace_bytes(B, T, H), device="cuda", dtype=torch.uint8)
        r = [ref.data_ptr() + i * H * D * 2 for i in range(3)]
        gp = [got.data_ptr() + i * H * D * 2 for i in range(3)]
        L.nc_attention_backward(q, k, v, 3 * H * D, o.data_ptr(), dout.data_ptr(), H * D, lse.data_ptr(),
                                r[0], r[1], r[2], 3 * H * D, ws.data_ptr(), B, T, H, D, L.NC_BF16, s)
        L.nc_attention_backward_noalloc(q, k, v, 3 * H * D, o.data_ptr(), dout.data_ptr(), H * D,
                                        lse.data_ptr(), gp[0], gp[1], gp[2], 3 * H * D, B, T, H, D,
                                        L.NC_BF16, s)
        torch.cuda.synchronize()
        a = got.float().cpu().numpy()
        b = ref.float().cpu().numpy()
        assert np.all(np.isfinite(a))
        for i, name in enumerate(("dq", "dk", "dv")):
            sl = slice(i * H * D, (i + 1) * H * D)
            assert_close(a[:, sl], b[:, sl], 0.999, 2e-2, f"seed {seed} {name}")


def test_noalloc_backward_rejects_oversized_problem():
    from pretraining_step_03_b300 import _lib as L
    big_B = (1 << 20) // (8 * 128) + 1   # B*H*T just above the built-in scratch
    with pytest.raises(L.NcError) as e:
        L.nc_attention_backward_noalloc(16, 16, 16, 1024, 16, 16, 1024, 16, 16, 16, 16, 1024, big_B, 128, 8,
                                        128, L.NC_BF16, 0)
    assert e.value.code == L.NC_ERR_ARG
    assert "exceeds" in L.nc_last_error()
