"""Failure detection on the GPU without a fault: a bounded wait that runs out.

A test build of the library (-DNF4_TEST_DROP_CONVERTED_ARRIVE
-DNF4_TEST_DROP_CONSUMED_ARRIVE, wait limit 50 ms) withholds two reports,
flags that nothing else sets: in the tcgen05 kernels the "converted" report
for the first K-slice, so the MMA issuer's wait on it expires (in the CTA-pair
kernel the odd CTA's waits for the MMAs then expire on their own); in the
warp-MMA kernel (M <= 16) one warp's "consumed" report for the first ring
slot, so the producer's wait to refill it expires.  The CTA must then record
the error word, drain its in-flight copies, release what it holds and return.
The host sees the launch succeed, nf4_last_error() report NF4_ERR_TIMEOUT
once (the word is cleared by the read), and the context stays usable: the
normal library computes a correct result right afterwards.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4
from nf4_weight_quantized_quantize_gb300 import build as nf4_build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def faulty_lib():
    path = nf4_build.build(extra=["-DNF4_TEST_DROP_CONVERTED_ARRIVE", "-DNF4_TEST_DROP_CONSUMED_ARRIVE",
                                  "-DNF4_WAIT_LIMIT_NS=50000000ull"],
                           out=os.path.join(nf4_build.BUILD, "libnf4_droparrive.so"))
    lib = ctypes.CDLL(path)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    lib.nf4_linear.argtypes = [P, I64, I64, P, P, I64, I32, P, P, SZ, P]
    lib.nf4_linear.restype = ctypes.c_int
    lib.nf4_linear_geglu.argtypes = [P, I64, I64, P, P, I64, I32, P, P, SZ, P]
    lib.nf4_linear_geglu.restype = ctypes.c_int
    lib.nf4_linear_ex.argtypes = [P, I32, I64, I64, P, P, I64, I32, P, P, SZ, P]
    lib.nf4_linear_ex.restype = ctypes.c_int
    lib.nf4_last_error.argtypes = [P]
    lib.nf4_last_error.restype = ctypes.c_int
    return lib


def _inputs(m, n, k, seed):
    rs = np.random.default_rng(seed)
    w = torch.from_numpy((rs.standard_normal((n, k)) * 0.02).astype(np.float32)).to(torch.bfloat16)
    x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16)
    p, a = oracle.quantize(workloads.bits(w))
    return x.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV), workloads.bits(x), p, a


@pytest.mark.parametrize("m,n,k", [(256, 512, 1024), (64, 512, 1024), (16, 19456, 1792), (1500, 10000, 192)],
                         ids=["tile_kernel", "split_kernel", "warp_mma_kernel", "pair_kernel"])
def test_bounded_wait_expires_and_reports(faulty_lib, m, n, k):
    # warp_mma_kernel: 152 tiles of 128 rows, no K split, 7 stages per CTA --
    # one more than its 6-slot ring, so the producer must wait for slot 0
    if m <= 16:
        rs = np.random.default_rng(5)
        x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16).to(DEV)
        pd = torch.from_numpy(rs.integers(0, 256, n * k // 2, dtype=np.uint8)).to(DEV)
        ad = torch.ones(n * k // 64, dtype=torch.float32, device=DEV)
    else:
        x, pd, ad, _, _, _ = _inputs(m, n, k, m)
    y = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    st, need = nf4.nf4_linear_workspace_size(m, n, k)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty_lib.nf4_linear(x.data_ptr(), m, k, pd.data_ptr(), ad.data_ptr(), n, 64, y.data_ptr(),
                               ws.data_ptr(), need, stream)
    assert st == nf4.NF4_OK                                  # the launch itself is fine
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_ERR_TIMEOUT
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_OK  # read-and-clear


@pytest.mark.parametrize("m,f,k", [(256, 256, 512), (1500, 5000, 192)], ids=["tile_kernel", "pair_kernel"])
def test_gate_up_pair_bounded_wait_expires(faulty_lib, m, f, k):
    """The fused gate/up forms: their epilogues meet at named barriers, which
    every converter thread must reach even when a wait ran out."""
    x, pd, ad, _, _, _ = _inputs(m, 2 * f, k, m + f)
    y = torch.empty(m, f, dtype=torch.bfloat16, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty_lib.nf4_linear_geglu(x.data_ptr(), m, k, pd.data_ptr(), ad.data_ptr(), f, 64, y.data_ptr(),
                                     None, 0, stream)
    assert st == nf4.NF4_OK
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_ERR_TIMEOUT
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_OK


def test_fp32_pair_bounded_wait_expires(faulty_lib):
    """The CTA-pair kernel's fp32 form: two ring slices per K-slice, each
    expanded by four converter warps per CTA; withholding the first stage's
    reports leaves four slices incomplete and the issuers' waits run out."""
    m, n, k = 1500, 10000, 192
    rs = np.random.default_rng(11)
    w = (rs.standard_normal((n, k)) * 0.02).astype(np.float32)
    x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32)).to(DEV)
    p, a = oracle.quantize(w.reshape(-1), dtype="f32")
    pd, ad = torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV)
    y = torch.empty(m, n, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = faulty_lib.nf4_linear_ex(x.data_ptr(), nf4.NF4_DTYPE_F32, m, k, pd.data_ptr(), ad.data_ptr(), n, 64,
                                  y.data_ptr(), None, 0, stream)
    assert st == nf4.NF4_OK
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_ERR_TIMEOUT
    assert faulty_lib.nf4_last_error(stream) == nf4.NF4_OK


def test_context_usable_after_timeouts(faulty_lib):
    m, n, k = 256, 512, 1024
    x, pd, ad, xb, p, a = _inputs(m, n, k, 99)
    y = nf4.linear(x, pd, ad, n)
    torch.cuda.synchronize()
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
    yref = oracle.linear(xb, p, a, n)
    yg = y.float().cpu().numpy().astype(np.float64)
    err = np.max(np.abs(yg - yref) / np.linalg.norm(yref, axis=1, keepdims=True))
    assert err < 1e-2
