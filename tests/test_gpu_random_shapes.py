"""Seeded random shapes through every route of nf4_linear and
nf4_linear_geglu at every compute dtype, against the oracle.

The shape draws span the routes a call can take -- the warp-MMA kernel
(M <= 16, bf16/fp16), the split tile kernel and its reduction (M < 128, and
fp32 skinny), the tile kernel and the CTA-pair kernel (M >= 128, which one by
the shape-only estimate) -- with ragged M and N (partial tiles, partial pairs,
partial row groups) and K from one NF4 block to 60.  The weights are quantized
by the library (bit-exactness of the quantizer is checked against the oracle
here too); each result is compared with the oracle's fp64 product on a sample
of rows within the row-normalised 1e-2 tolerance.  The draws are fixed by the
seed, so a failure names a reproducible case.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
TOL = 1e-2


def _draws(n=96, seed=20261203):
    rs = np.random.default_rng(seed)
    out = []
    for i in range(n):
        dtype = ["bf16", "f16", "f32"][i % 3]
        band = i % 4   # skinny, mid, tile-sized, pair-sized batches
        M = int([rs.integers(1, 17), rs.integers(17, 128), rs.integers(128, 513), rs.integers(513, 2600)][band])
        N = int(rs.integers(1, 160) * 2 if band < 2 else rs.integers(64, 5000) * 2)
        K = 64 * int(rs.integers(1, 61 if M * N < 4_000_000 else 20))
        geglu = bool(rs.integers(0, 4) == 0)
        out.append((dtype, M, N, K, geglu))
    return out


CASES = _draws()


@pytest.mark.parametrize("dtype,M,N,K,geglu", CASES,
                         ids=[f"{d}-M{m}-N{n}-K{k}{'-geglu' if g else ''}" for d, m, n, k, g in CASES])
def test_random_shape(dtype, M, N, K, geglu):
    seed = M * 7919 + N * 31 + K
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(N, K, generator=g) * 0.03).to(TORCH[dtype])
    x = torch.randn(M, K, generator=g).to(TORCH[dtype])
    p, a = nf4.quantize(w.to(DEV))
    torch.cuda.synchronize()
    op, oa = oracle.quantize(workloads.host(w), dtype=dtype)
    assert np.array_equal(p.cpu().numpy(), op) and np.array_equal(a.cpu().numpy().view(np.uint32), oa.view(np.uint32))
    xd = x.to(DEV)
    if geglu:
        F = N // 2
        y = nf4.linear_geglu(xd, p, a, F)
    else:
        y = nf4.linear(xd, p, a, N)
    torch.cuda.synchronize()
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
    rows = np.arange(M) if M <= 24 else np.sort(np.random.default_rng(seed).choice(M, 24, replace=False))
    yg = y.float().cpu().numpy().astype(np.float64)[rows]
    xb = workloads.host(x)[rows]
    yref = oracle.linear_geglu(xb, op, oa, N // 2, dtype=dtype) if geglu else oracle.linear(xb, op, oa, N, dtype=dtype)
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    err = float(np.max(np.abs(yg - yref) / np.maximum(nrm, 1e-300)))
    assert err <= TOL, f"row-normalised error {err}"
