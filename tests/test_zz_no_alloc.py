"""The allocation-free attention backward, through the C ABI.

nc_attention_backward_noalloc serves callers that cannot allocate device
memory (their device memory is reserved by another runtime, or they cannot
afford cudaMalloc's device-wide synchronisation): its row-statistics scratch
is a fixed array inside the library.  Checked here:

* two calls in a row, on different inputs, each against the fp64 oracle
  (bf16 attention tolerance: cosine >= 0.999, max-rel <= 2e-2) and against
  nc_attention_backward with a caller workspace;
* the fp32 / head-dim-64 path (CUDA-core kernels, another statistics
  kernel) against the oracle at the fp32 tolerance (max-rel <= 1e-4);
* that a call allocates nothing: neither torch's allocator nor the device's
  free memory changes across it (after a first call has looked the scratch
  address up);
* that no kernel set the kernel-level flag word.

This file is named to be collected last.
"""

import numpy as np
import pytest

import oracle
from tests._util import assert_close, bf16_round

pytestmark = pytest.mark.gpu


def _case(seed, B, T, H, D, mode):
    """Seeded N(0, 1) inputs (rounded to bf16 in bf16 mode), the kernel's forward, and
    the oracle's gradients computed from the same inputs."""
    import torch
    from pretraining_step_03_b300 import _lib as L
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.normal(size=(B, T, H, D)).astype(np.float32) for _ in range(4))
    if mode == "bf16":
        q, k, v, do = (bf16_round(x) for x in (q, k, v, do))
    tdt = torch.bfloat16 if mode == "bf16" else torch.float32
    dtc = L.NC_BF16 if mode == "bf16" else L.NC_FP32
    Q, K, Vv, DO = (torch.from_numpy(x).to("cuda", tdt) for x in (q, k, v, do))
    O = torch.empty_like(Q)
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    L.nc_attention_forward(Q.data_ptr(), K.data_ptr(), Vv.data_ptr(), H * D, O.data_ptr(), H * D,
                           lse.data_ptr(), B, T, H, D, dtc, s)
    ref = []
    for b in range(B):
        sl = slice(b, b + 1)
        _, p, _ = oracle.causal_attention(q[sl], k[sl], v[sl])
        ref.append(oracle.causal_attention_backward(do[sl], q[sl], k[sl], v[sl], p))
    return dict(Q=Q, K=K, V=Vv, O=O, DO=DO, lse=lse, dtc=dtc, s=s, ref=ref)


def _noalloc(c, B, T, H, D):
    import torch
    from pretraining_step_03_b300 import _lib as L
    grads = [torch.full_like(c["Q"], float("nan")) for _ in range(3)]
    L.nc_attention_backward_noalloc(c["Q"].data_ptr(), c["K"].data_ptr(), c["V"].data_ptr(), H * D,
                                    c["O"].data_ptr(), c["DO"].data_ptr(), H * D, c["lse"].data_ptr(),
                                    grads[0].data_ptr(), grads[1].data_ptr(), grads[2].data_ptr(), H * D,
                                    B, T, H, D, c["dtc"], c["s"])
    return grads


def _with_workspace(c, B, T, H, D):
    import torch
    from pretraining_step_03_b300 import _lib as L
    grads = [torch.empty_like(c["Q"]) for _ in range(3)]
    ws = torch.empty(L.nc_attention_workspace_bytes(B, T, H), device="cuda", dtype=torch.uint8)
    L.nc_attention_backward(c["Q"].data_ptr(), c["K"].data_ptr(), c["V"].data_ptr(), H * D,
                            c["O"].data_ptr(), c["DO"].data_ptr(), H * D, c["lse"].data_ptr(),
                            grads[0].data_ptr(), grads[1].data_ptr(), grads[2].data_ptr(), H * D,
                            ws.data_ptr(), B, T, H, D, c["dtc"], c["s"])
    return grads


def _host(grads):
    return [g.float().cpu().numpy() for g in grads]


def test_noalloc_backward_matches_oracle_twice():
    import torch
    from pretraining_step_03_b300 import _lib as L
    B, T, H, D = 2, 384, 4, 128
    for seed in (11, 12):   # two calls in a row, different inputs
        c = _case(seed, B, T, H, D, "bf16")
        got = _host(_noalloc(c, B, T, H, D))
        ws = _host(_with_workspace(c, B, T, H, D))
        torch.cuda.synchronize()
        assert L.nc_check_kernel_flag(c["s"]) == 0
        for i, name in enumerate(("dq", "dk", "dv")):
            assert np.all(np.isfinite(got[i])), name
            for b in range(B):
                assert_close(got[i][b], c["ref"][b][i][0], 0.999, 2e-2, f"seed {seed} {name} b={b} vs oracle")
            assert_close(got[i], ws[i], 0.999, 2e-2, f"seed {seed} {name} vs workspace version")


def test_noalloc_backward_fp32_head_dim_64():
    import torch
    from pretraining_step_03_b300 import _lib as L
    B, T, H, D = 2, 77, 3, 64
    for seed in (21, 22):
        c = _case(seed, B, T, H, D, "fp32")
        got = _host(_noalloc(c, B, T, H, D))
        torch.cuda.synchronize()
        assert L.nc_check_kernel_flag(c["s"]) == 0
        for i, name in enumerate(("dq", "dk", "dv")):
            for b in range(B):
                assert_close(got[i][b], c["ref"][b][i][0], 0.99999, 1e-4, f"fp32 seed {seed} {name} b={b}")


def test_noalloc_backward_allocates_nothing():
    import torch
    B, T, H, D = 2, 256, 2, 128
    c = _case(31, B, T, H, D, "bf16")
    out = [torch.empty_like(c["Q"]) for _ in range(3)]
    from pretraining_step_03_b300 import _lib as L

    def call():
        L.nc_attention_backward_noalloc(c["Q"].data_ptr(), c["K"].data_ptr(), c["V"].data_ptr(), H * D,
                                        c["O"].data_ptr(), c["DO"].data_ptr(), H * D, c["lse"].data_ptr(),
                                        out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), H * D,
                                        B, T, H, D, c["dtc"], c["s"])

    call()                      # the first call on the device looks the scratch address up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before, (free_before, free_after)


def test_noalloc_backward_rejects_oversized_problem():
    from pretraining_step_03_b300 import _lib as L
    big_B = (1 << 20) // (8 * 128) + 1   # B*H*T just above the built-in scratch
    with pytest.raises(L.NcError) as e:
        L.nc_attention_backward_noalloc(16, 16, 16, 1024, 16, 16, 1024, 16, 16, 16, 16, 1024, big_B, 128, 8,
                                        128, L.NC_BF16, 0)
    assert e.value.code == L.NC_ERR_ARG
    assert "exceeds" in L.nc_last_error()
