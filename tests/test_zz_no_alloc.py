"""nf4_linear_noalloc: the skinny NF4 linear without a caller workspace.

Some callers cannot allocate device memory themselves (a plugin inside a host
application that owns the whole device memory pool, or a path that cannot
afford cudaMalloc's implicit synchronization).  For them the split-K scratch
lives in a fixed 16 MiB library-owned device array.  This file checks,
through the C ABI, that two calls in a row give exactly the bits nf4_linear
gives for the same arguments, that each is within the parity tolerance of the
CPU oracle, and that the entry point rejects what it cannot do.  It is collected last so that a run
stopping at its first failure has run every other test already; it also
passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2   # row-normalised max error, as for nf4_linear


def _case(m, n, k, seed):
    rs = np.random.default_rng(seed)
    w = torch.from_numpy((rs.standard_normal((n, k)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16)
    p, a = oracle.quantize(workloads.bits(w))
    return x.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV)


def _f32_of_bits(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("m,n,k", [(16, 3840, 15360), (7, 640, 1536), (127, 256, 512), (127, 32768, 64)],
                         ids=["down_proj_m16", "m7", "m127", "scratch_just_under_16MiB"])
def test_two_calls_match_nf4_linear(m, n, k):
    """Two calls in a row give exactly nf4_linear's bits (the same kernels on
    the same shape-only plan, partials summed in a fixed order) and each is
    within the parity tolerance of the oracle, plus the per-element bound of
    bf16 output rounding and fp32 summation; the last shape uses all but
    0.8 % of the fixed scratch array, so a mis-sized slice would show."""
    x, pd, ad = _case(m, n, k, m + n)
    p, a = pd.cpu().numpy(), ad.cpu().numpy()
    st, need = nf4.nf4_linear_workspace_size(m, n, k)
    assert st == nf4.NF4_OK and need <= nf4.NF4_NOALLOC_SCRATCH_BYTES
    if n == 32768:
        assert need > 0.99 * nf4.NF4_NOALLOC_SCRATCH_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    y_ref = nf4.linear(x, pd, ad, n)                 # the existing entry point, torch workspace
    xb = workloads.bits(x.cpu())
    yo = oracle.linear(xb, p, a, n)
    nrm = np.maximum(np.linalg.norm(yo, axis=1, keepdims=True), 1e-300)
    if n * k <= 1 << 22:
        wd = _f32_of_bits(oracle.dequantize(p, a, n * k)).astype(np.float64).reshape(n, k)
        mag = np.abs(_f32_of_bits(xb).astype(np.float64)) @ np.abs(wd).T
        bound = 2.0 ** -8 * np.abs(yo) + k * 2.0 ** -23 * mag + 1e-30
    for _ in range(2):
        y = torch.full((m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
        st = nf4.nf4_linear_noalloc(x.data_ptr(), m, k, pd.data_ptr(), ad.data_ptr(), n, 64,
                                    y.data_ptr(), stream)
        assert st == nf4.NF4_OK, nf4.nf4_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        yg = y.double().cpu().numpy()
        assert float(np.max(np.abs(yg - yo) / nrm)) <= TOL
        if n * k <= 1 << 22:
            assert not (np.abs(yg - yo) > bound).any()
    assert nf4.nf4_last_error(stream) == nf4.NF4_OK


def test_rejects_what_it_cannot_do():
    stream = torch.cuda.current_stream().cuda_stream
    x, pd, ad = _case(16, 64, 64, 1)
    y = torch.empty(16, 64, dtype=torch.bfloat16, device=DEV)
    args = (x.data_ptr(), 16, 64, pd.data_ptr(), ad.data_ptr(), 64, 64, y.data_ptr(), stream)
    assert nf4.nf4_linear_noalloc(*args) == nf4.NF4_OK
    # M >= 128: the tile path needs no scratch, use nf4_linear
    assert nf4.nf4_linear_noalloc(x.data_ptr(), 128, 64, pd.data_ptr(), ad.data_ptr(), 64, 64,
                                  y.data_ptr(), stream) == nf4.NF4_ERR_SHAPE
    # a shape whose split-K scratch exceeds the fixed array, rejected before any launch
    m, n, k = 100, 60000, 64
    st, need = nf4.nf4_linear_workspace_size(m, n, k)
    assert st == nf4.NF4_OK and need > nf4.NF4_NOALLOC_SCRATCH_BYTES
    assert nf4.nf4_linear_noalloc(x.data_ptr(), m, k, pd.data_ptr(), ad.data_ptr(), n, 64,
                                  y.data_ptr(), stream) == nf4.NF4_ERR_WORKSPACE
    assert nf4.nf4_linear_noalloc(x.data_ptr(), 16, 64, pd.data_ptr(), ad.data_ptr(), 64, 32,
                                  y.data_ptr(), stream) == nf4.NF4_ERR_BLOCKSIZE
    torch.cuda.synchronize()
