"""The tensor-core GEMM through the C ABI against fp64 products of the same bf16 inputs.

Covers every operand layout (K-major / MN-major for A and B), ragged M/N/K
tails, fp32 and bf16 outputs, beta accumulation, batching and split-K.
Tolerance: max|C - ref| / max|ref| <= 1e-4 for fp32 outputs (fp32
accumulation of exactly-representable bf16 products) and 8e-3 for bf16
outputs (one bf16 rounding, 2^-8 relative).
"""

import numpy as np
import pytest

from tests._util import bf16_round

pytestmark = pytest.mark.gpu


def _run(M, N, K, ta, tb, batch=1, c_dtype="f32", beta=0.0, ws_bytes=0, seed=0):
    import torch
    from pretraining_step_03_b300 import _lib as L
    rng = np.random.default_rng(seed)
    a = bf16_round(rng.normal(size=(batch, K, M) if ta else (batch, M, K)))
    b = bf16_round(rng.normal(size=(batch, K, N) if tb else (batch, N, K)))
    c0 = bf16_round(rng.normal(size=(batch, M, N)))
    dev = torch.device("cuda")
    A = torch.from_numpy(a).to(dev, torch.bfloat16)
    Bt = torch.from_numpy(b).to(dev, torch.bfloat16)
    cdt = torch.float32 if c_dtype == "f32" else torch.bfloat16
    C = torch.from_numpy(c0).to(dev, cdt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    lda = M if ta else K
    ldb = N if tb else K
    L.nc_gemm_bf16(M, N, K, batch, A.data_ptr(), lda, a[0].size, int(ta), Bt.data_ptr(), ldb, b[0].size,
                   int(tb), C.data_ptr(), N, M * N, L.NC_FP32 if c_dtype == "f32" else L.NC_BF16, 1.5, beta,
                   ws.data_ptr() if ws_bytes else 0, ws_bytes, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    opa = np.swapaxes(a, 1, 2) if ta else a
    opb = np.swapaxes(b, 1, 2) if tb else b
    ref = 1.5 * np.matmul(opa.astype(np.float64), np.swapaxes(opb, 1, 2).astype(np.float64)) + beta * c0
    got = C.float().cpu().numpy().astype(np.float64)
    return got, ref


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(304, 264, 200), (128, 128, 64), (72, 40, 24)])
def test_layouts_and_tails(M, N, K, ta, tb):
    got, ref = _run(M, N, K, ta, tb)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-4


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
def test_bf16_output_beta_and_batch(ta, tb):
    got, ref = _run(200, 520, 136, ta, tb, batch=3, c_dtype="bf16", beta=1.0)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 8e-3


def test_split_k_weight_gradient_shape():
    # small output, long reduction: the weight-gradient shape, split over K
    got, ref = _run(256, 384, 8192, 1, 1, ws_bytes=64 << 20, beta=1.0)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-4


def test_d20_projection_shape():
    got, ref = _run(1024, 3840, 1280, 0, 0, c_dtype="bf16")
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 8e-3


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_cta_pair_tiles_ragged(ta, tb):
    # M, N >= 256 run on CTA pairs (256 x 256 tiles); ragged in M, N and K
    got, ref = _run(520, 776, 200, ta, tb)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-4


def test_cta_pair_batched_square():
    # the Newton-Schulz shape class: batched square products, B stored [K, N]
    got, ref = _run(384, 384, 384, 0, 1, batch=3, c_dtype="bf16", beta=1.0)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 8e-3


@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,batch", [(520, 320, 1), (304, 448, 2), (520, 776, 1)])
def test_cta_pair_in_place_accumulate(M, N, ta, tb, batch):
    # C += alpha A B^T in fp32 in place (the residual stream, accumulated weight gradients):
    # C comes back in through the epilogue's auxiliary stream; ragged M and K, batched
    got, ref = _run(M, N, 200, ta, tb, batch=batch, beta=1.0)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-4
