"""GPU parity of the fp16 and fp32 compute dtypes (the _ex entry points)
against the oracle.

Quantize and dequantize have one correct answer at every dtype and are
compared bit for bit: whole Gemma3 projection weights, ragged sizes that
end in a partial tile or block, unaligned pointers (the element-wise
kernels), and blocks whose absmax is subnormal.  The fp16 linear and the
fp16 gate/up pair are compared with the oracle's fp64 result of the same
fp16 inputs within the row-normalised tolerance of the bf16 linear, plus a
per-element bound of fp16 output rounding and fp32 summation error; the fp32
ones (tf32 tensor-core products) the same way with the tf32 operand error
in the bound.
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


def rand_w(numel, std, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(numel, generator=g) * std).to(TORCH[dtype])


def special_blocks(dtype):
    """Blocks of zeros, -0.0, one outlier, subnormal-only magnitudes (the
    absmax below the smallest normal of the type, or of fp32) and a mix."""
    rs = np.random.default_rng(5)
    tiny = {"bf16": 2.0 ** -130, "f16": 2.0 ** -20, "f32": 2.0 ** -140}[dtype]
    rows = [np.zeros(64), -np.zeros(64), rs.normal(0, 0.02, 64), rs.normal(0, 1, 64) * tiny,
            rs.normal(0, 1, 64) * tiny * 64, np.concatenate([rs.normal(0, 1e-3, 63), [3.0]])]
    r = rs.normal(0, 0.02, 64)
    r[::5] = 0
    rows.append(r)
    return torch.from_numpy(np.concatenate(rows).astype(np.float32)).to(TORCH[dtype])


def check_quantize(w_cpu, dtype, offset=0):
    """nf4_quantize_ex on w (optionally at an element offset into a larger
    buffer, so the pointer loses its 16-byte alignment) against the oracle."""
    if offset:
        buf = torch.zeros(w_cpu.numel() + offset, dtype=w_cpu.dtype)
        buf[offset:] = w_cpu
        wd = buf.to(DEV)[offset:]
    else:
        wd = w_cpu.to(DEV)
    p, a = nf4.quantize(wd)
    torch.cuda.synchronize()
    op, oa = oracle.quantize(workloads.host(w_cpu), dtype=dtype)
    assert np.array_equal(p.cpu().numpy(), op), "packed bytes differ"
    assert np.array_equal(a.cpu().numpy().view(np.uint32), oa.view(np.uint32)), "absmax differs"
    return op, oa


def check_dequantize(p, a, numel, dtype, offset=0):
    out_full = torch.empty(numel + offset, dtype=TORCH[dtype], device=DEV)
    out = out_full[offset:]
    nf4.dequantize(torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV), numel, out=out)
    torch.cuda.synchronize()
    want = oracle.dequantize(p, a, numel, dtype=dtype)
    got = workloads.host(out)
    assert np.array_equal(got.view(np.uint16 if dtype != "f32" else np.uint32),
                          want.view(np.uint16 if dtype != "f32" else np.uint32)), "dequantized values differ"


# ---------------------------------------------------------------- quantize / dequantize


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("cfg", [workloads.Q_PROJ, workloads.DOWN], ids=lambda c: c.name)
def test_projection_weights_bit_exact(dtype, cfg):
    w = workloads.make_weight(cfg, dtype=TORCH[dtype]).reshape(-1)
    p, a = check_quantize(w, dtype)
    check_dequantize(p, a, w.numel(), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_special_blocks_bit_exact(dtype):
    w = special_blocks(dtype)
    p, a = check_quantize(w, dtype)
    check_dequantize(p, a, w.numel(), dtype)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
@pytest.mark.parametrize("numel", [2, 64, 100, 128, 64 * 33 + 2, 512 * 9 + 64 * 3 + 10, 1 << 20])
def test_ragged_sizes_bit_exact(dtype, numel):
    w = rand_w(numel, 0.02, numel % 9973, dtype)
    p, a = check_quantize(w, dtype)
    check_dequantize(p, a, numel, dtype)


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_unaligned_pointers_bit_exact(dtype):
    """w and out one element past a 16-byte boundary: the element-wise kernels."""
    w = rand_w(64 * 50, 0.02, 77, dtype)
    p, a = check_quantize(w, dtype, offset=1)
    check_dequantize(p, a, w.numel(), dtype, offset=1)


def test_same_values_same_bytes_across_dtypes():
    """bf16 weights widened to fp32 (exact) quantize to the same bytes and
    scales at both dtypes; likewise fp16 weights widened to fp32."""
    w16 = workloads.make_weight(workloads.TINY)
    for narrow in (w16, w16.to(torch.float16)):
        p1, a1 = nf4.quantize(narrow.to(DEV))
        p2, a2 = nf4.quantize(narrow.float().to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(p1, p2) and torch.equal(a1, a2)


# ---------------------------------------------------------------- fp16 linear


def f16_linear_check(x_cpu, w_cpu, fn, n_cols, oracle_fn, rows=None):
    """Run the fp16 GEMM `fn` and compare (the sampled `rows` of) its result
    with the oracle's fp64 result of the same rows."""
    p, a = oracle.quantize(workloads.host(w_cpu), dtype="f16")
    y = fn(x_cpu.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV))
    torch.cuda.synchronize()
    assert y.dtype == torch.float16 and y.shape == (x_cpu.shape[0], n_cols)
    yg = y.float().cpu().numpy().astype(np.float64)
    xb = workloads.host(x_cpu)
    if rows is not None:
        yg, xb = yg[rows], xb[rows]
    yref = oracle_fn(xb, p, a)
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    err = float(np.max(np.abs(yg - yref) / np.maximum(nrm, 1e-300)))
    assert err <= TOL, f"row-normalised error {err}"
    return yg, yref, xb, p, a


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 3840), (16, 3840, 15360), (257, 300, 128), (130, 640, 1536),
                                   (33, 1000, 64 * 50), (700, 30720, 128)])
def test_linear_f16(M, N, K):
    rs_seed = M + N + K
    w = rand_w(N * K, 0.02, rs_seed, "f16").reshape(N, K)
    x = rand_w(M * K, 1.0, rs_seed + 1, "f16").reshape(M, K)
    rows = None if M * N <= 1 << 20 else np.sort(np.random.default_rng(M).choice(M, 32, replace=False))
    ys, yref, xs, p, a = f16_linear_check(x, w, lambda xd, pd, ad: nf4.linear(xd, pd, ad, N), N,
                                          lambda xb, p, a: oracle.linear(xb, p, a, N, dtype="f16"), rows)
    # per element: fp16 rounding of Y plus fp32 summation error
    wd = oracle.dequantize(p, a, N * K, dtype="f16").view(np.float16).astype(np.float64).reshape(N, K)
    mag = np.abs(xs.view(np.float16).astype(np.float64)) @ np.abs(wd).T
    bound = 2.0 ** -11 * np.abs(yref) + K * 2.0 ** -23 * mag + 2.0 ** -24
    assert not (np.abs(ys - yref) > bound).any()


@pytest.mark.parametrize("M,F,K", [(300, 640, 1024), (16, 640, 1024), (2048, 2432, 256)],
                         ids=["tile_tcgen05", "warp_mma", "cta_pair"])
def test_linear_geglu_f16(M, F, K):
    w = rand_w(2 * F * K, 0.05, 90 + M, "f16").reshape(2 * F, K)
    x = rand_w(M * K, 1.0, 91 + M, "f16").reshape(M, K)
    rows = None if M * F <= 1 << 20 else np.sort(np.random.default_rng(M).choice(M, 32, replace=False))
    f16_linear_check(x, w, lambda xd, pd, ad: nf4.linear_geglu(xd, pd, ad, F), F,
                     lambda xb, p, a: oracle.linear_geglu(xb, p, a, F, dtype="f16"), rows)


@pytest.mark.parametrize("M,N", [(16, 256), (64, 256), (300, 256), (2048, 4864)],
                         ids=["warp_mma", "split_tcgen05", "tile_tcgen05", "cta_pair"])
def test_linear_f16_on_weights_quantized_at_f32(M, N):
    """The fp16 linear on a weight quantized from fp32 values: its absmax
    values are not fp16 values, and every 7th row is scaled so that the
    dequantized values land in fp16's subnormal range.  Every fused kernel
    must scale by the fp32 absmax and round once (the fp16 dequantizer's
    value, which the oracle uses) rather than round the absmax first
    (sampled rows for the large batch)."""
    K = 1024
    rs = np.random.default_rng(40 + M)
    w = (rs.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[::7] *= 1e-3
    p, a = oracle.quantize(w, dtype="f32")
    assert np.any(a.astype(np.float16).astype(np.float32) != a)
    x = rand_w(M * K, 1.0, 50 + M, "f16").reshape(M, K)
    y = nf4.linear(x.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV), N)
    torch.cuda.synchronize()
    yg = y.float().cpu().numpy().astype(np.float64)
    xb = workloads.host(x)
    if M > 300:
        rows = np.sort(np.random.default_rng(M).choice(M, 32, replace=False))
        yg, xb = yg[rows], xb[rows]
    yref = oracle.linear(xb, p, a, N, dtype="f16")
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    assert float(np.max(np.abs(yg - yref) / nrm)) <= TOL
    wd = oracle.dequantize(p, a, N * K, dtype="f16").view(np.float16).astype(np.float64).reshape(N, K)
    mag = np.abs(xb.view(np.float16).astype(np.float64)) @ np.abs(wd).T
    bound = 2.0 ** -11 * np.abs(yref) + K * 2.0 ** -23 * mag + 2.0 ** -24
    assert not (np.abs(yg - yref) > bound).any()


def test_f16_matches_bf16_path_on_shared_values():
    """Weights and activations exactly representable in both 16-bit types
    (small integers times powers of two): the fp16 and bf16 GEMMs agree to
    within their output roundings."""
    rs = np.random.default_rng(3)
    N, K, M = 256, 512, 256
    w = torch.from_numpy((rs.integers(-64, 64, (N, K)) * 2.0 ** -8).astype(np.float32))
    x = torch.from_numpy((rs.integers(-8, 8, (M, K)) * 2.0 ** -2).astype(np.float32))
    ys = []
    for dt in (torch.bfloat16, torch.float16):
        p, a = nf4.quantize(w.to(dt).to(DEV))
        ys.append(nf4.linear(x.to(dt).to(DEV), p, a, N).float())
    ref = ys[0].abs().amax(dim=1, keepdim=True)
    assert ((ys[0] - ys[1]).abs() / ref).max().item() < 1e-2


# ---------------------------------------------------------------- fp32 linear (tf32 MMA)


def linear_check(dtype, x_cpu, w_cpu, fn, n_cols, oracle_fn, rows=None):
    """Run the GEMM `fn` at `dtype` and compare (the sampled `rows` of) its
    result with the oracle's fp64 result of the same rows; returns the
    compared arrays."""
    p, a = oracle.quantize(workloads.host(w_cpu), dtype=dtype)
    y = fn(x_cpu.to(DEV), torch.from_numpy(p).to(DEV), torch.from_numpy(a).to(DEV))
    torch.cuda.synchronize()
    assert y.dtype == TORCH[dtype] and y.shape == (x_cpu.shape[0], n_cols)
    yg = y.float().cpu().numpy().astype(np.float64)
    xb = workloads.host(x_cpu)
    if rows is not None:
        yg, xb = yg[rows], xb[rows]
    yref = oracle_fn(xb, p, a)
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    err = float(np.max(np.abs(yg - yref) / np.maximum(nrm, 1e-300)))
    assert err <= TOL, f"row-normalised error {err}"
    return yg, yref, xb, p, a


@pytest.mark.parametrize("M,N,K", [(2048, 4096, 3840), (16, 3840, 15360), (257, 300, 128), (130, 640, 1536),
                                   (33, 1000, 64 * 50), (512, 256, 64),
                                   # CTA pairs at fp32 (two tf32 ring slices per K-slice): ragged M and
                                   # N, an odd number of K-slices, nx = 256 and 192
                                   (1500, 10000, 192), (2047, 4100, 320), (700, 30720, 128)])
def test_linear_f32(M, N, K):
    """fp32 compute dtype: the tensor cores read tf32 (X's 10-bit fraction,
    the weight rounded to tf32), accumulate in fp32 and write fp32.  Per
    element each product is within 2^-9 relative of the exact one, so
    |Y - Yref| <= (2^-9 + K 2^-23) sum_k |x_k| |w_k|."""
    seed = 7 * M + N + K
    w = rand_w(N * K, 0.02, seed, "f32").reshape(N, K)
    x = rand_w(M * K, 1.0, seed + 1, "f32").reshape(M, K)
    rows = None if M * N <= 1 << 20 else np.sort(np.random.default_rng(M).choice(M, 32, replace=False))
    ys, yref, xs, p, a = linear_check("f32", x, w, lambda xd, pd, ad: nf4.linear(xd, pd, ad, N), N,
                                      lambda xb, p, a: oracle.linear(xb, p, a, N, dtype="f32"), rows)
    wd = oracle.dequantize(p, a, N * K, dtype="f32").astype(np.float64).reshape(N, K)
    mag = np.abs(xs.astype(np.float64)) @ np.abs(wd).T
    bound = (2.0 ** -9 + K * 2.0 ** -23) * mag + 1e-30
    assert not (np.abs(ys - yref) > bound).any()


@pytest.mark.parametrize("M", [300, 16])
def test_linear_geglu_f32(M):
    F, K = 640, 1024
    w = rand_w(2 * F * K, 0.05, 190 + M, "f32").reshape(2 * F, K)
    x = rand_w(M * K, 1.0, 191 + M, "f32").reshape(M, K)
    linear_check("f32", x, w, lambda xd, pd, ad: nf4.linear_geglu(xd, pd, ad, F), F,
                 lambda xb, p, a: oracle.linear_geglu(xb, p, a, F, dtype="f32"))


@pytest.mark.parametrize("M,F,K", [(2048, 2432, 256), (1500, 2400, 320)])
def test_linear_geglu_f32_pair_kernel(M, F, K):
    """The fused gate/up pair at fp32 on CTA pairs (sampled rows)."""
    w = rand_w(2 * F * K, 0.05, 290 + M, "f32").reshape(2 * F, K)
    x = rand_w(M * K, 1.0, 291 + M, "f32").reshape(M, K)
    rows = np.sort(np.random.default_rng(M + F).choice(M, 24, replace=False))
    linear_check("f32", x, w, lambda xd, pd, ad: nf4.linear_geglu(xd, pd, ad, F), F,
                 lambda xb, p, a: oracle.linear_geglu(xb, p, a, F, dtype="f32"), rows)


def test_f32_close_to_bf16_on_shared_values():
    """Weights and activations exactly representable in bf16: the fp32 (tf32)
    and bf16 GEMMs agree to within the bf16 roundings."""
    rs = np.random.default_rng(4)
    N, K, M = 384, 768, 300
    w = torch.from_numpy((rs.integers(-64, 64, (N, K)) * 2.0 ** -8).astype(np.float32))
    x = torch.from_numpy((rs.integers(-8, 8, (M, K)) * 2.0 ** -2).astype(np.float32))
    ys = []
    for dt in (torch.bfloat16, torch.float32):
        p, a = nf4.quantize(w.to(dt).to(DEV))
        ys.append(nf4.linear(x.to(dt).to(DEV), p, a, N).float())
    ref = ys[1].abs().amax(dim=1, keepdim=True)
    assert ((ys[0] - ys[1]).abs() / ref).max().item() < 1e-2


def test_no_error_recorded():
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
