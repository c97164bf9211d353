"""Degenerate shapes on the GPU, against the oracle: empty inputs at every
dtype (nothing enqueued, empty results, no error), a one-row weight (N = 1)
on the tile and split-K paths, the smallest product 1 x 1 x 64, and one
64-element block per row (K = 64) with a single activation row.  16-bit
results are checked with the row-normalised tolerance, fp32 (tf32 products)
with the per-element operand bound."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def rand(shape, std, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(DTYPES[dtype])


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_empty_inputs(dtype):
    dt = DTYPES[dtype]
    p, a = nf4.quantize(torch.empty(0, dtype=dt, device=DEV))
    assert p.numel() == 0 and a.numel() == 0
    y = nf4.dequantize(p, a, 0, dtype=dt)
    assert y.numel() == 0 and y.dtype == dt
    pw, aw = nf4.quantize(rand((64, 128), 0.02, 1, dtype).to(DEV))
    y = nf4.linear(torch.empty(0, 128, dtype=dt, device=DEV), pw, aw, 64)
    assert y.shape == (0, 64)
    y = nf4.linear_geglu(torch.empty(0, 128, dtype=dt, device=DEV), pw, aw, 32)
    assert y.shape == (0, 32)
    torch.cuda.synchronize()
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (200, 1, 64), (16, 1, 192), (300, 2, 64), (1, 640, 64),
                                   (256, 1, 1024)])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_degenerate_linear(M, N, K, dtype):
    w = rand((N, K), 0.02, N * K + M, dtype)
    x = rand((M, K), 1.0, M + 7, dtype)
    p, a = oracle.quantize(workloads.host(w), dtype=dtype)
    y = nf4.linear(x.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV), N)
    torch.cuda.synchronize()
    yref = oracle.linear(workloads.host(x), p, a, N, dtype=dtype)
    yg = y.float().cpu().numpy().astype(np.float64)
    if dtype == "f32":
        # tf32 products: each within 2^-9 relative (with N = 1 a row norm is one
        # element, so a cancelling dot product needs the per-element bound)
        wd = oracle.dequantize(p, a, N * K, dtype="f32").astype(np.float64).reshape(N, K)
        mag = np.abs(workloads.host(x).astype(np.float64)) @ np.abs(wd).T
        assert not (np.abs(yg - yref) > (2.0 ** -9 + K * 2.0 ** -23) * mag + 1e-30).any()
    else:
        nrm = np.maximum(np.linalg.norm(yref, axis=1, keepdims=True), 1e-30)
        assert np.max(np.abs(yg - yref) / nrm) <= 1e-2
    # quantize and dequantize of the same one-row / one-block tensors are bit-exact
    pq, aq = nf4.quantize(w.to(DEV))
    assert np.array_equal(pq.cpu().numpy(), p) and np.array_equal(aq.cpu().numpy().view(np.uint32), a.view(np.uint32))
    d = nf4.dequantize(pq, aq, N * K, dtype=DTYPES[dtype])
    want = oracle.dequantize(p, a, N * K, dtype=dtype)
    got = workloads.host(d)
    assert np.array_equal(got.view(want.dtype) if dtype != "f32" else got.view(np.uint32),
                          want if dtype != "f32" else want.view(np.uint32))


def test_no_error_recorded():
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
