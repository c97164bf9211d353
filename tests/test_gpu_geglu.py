"""GPU parity of nf4_linear_geglu (the Gemma3 MLP's gate and up projections
with the GELU-gated product fused into the GEMM epilogue) against the oracle.

The weight is ONE NF4 tensor [2F, K]: gate rows, then up rows.  The oracle
gives gelu_tanh(g) * u with g, u from an fp64 matmul of the dequantized
weight.  Checked: the row-normalised tolerance of nf4_linear (1e-2), and a
per-element bound built from the fp32 summation error of g and u, the slope
of gelu (|gelu'| < 1.13) and one bf16 rounding, which a swapped half, a wrong
activation or a dropped K-slice breaks.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-2


def f32_of_bits(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def rand_bits(shape, std, seed):
    rs = np.random.default_rng(seed)
    t = torch.from_numpy((rs.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


class Pair:
    """Gate and up weights stacked as [2F, K] and quantized by the oracle."""

    def __init__(self, w_bits_2d):
        n2, self.k = w_bits_2d.shape
        assert n2 % 2 == 0
        self.f = n2 // 2
        self.p, self.a = oracle.quantize(w_bits_2d)
        self.pd = torch.from_numpy(self.p).to(DEV)
        self.ad = torch.from_numpy(self.a).to(DEV)


def run(x_bits, w):
    y = nf4.linear_geglu(workloads.from_bits(x_bits, DEV), w.pd, w.ad, w.f)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def check(x_bits, w, rows=None):
    y = run(x_bits, w)
    xs = x_bits if rows is None else x_bits[rows]
    ys = y if rows is None else y[rows]
    yref = oracle.linear_geglu(xs, w.p, w.a, w.f)
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    err = float(np.max(np.abs(ys - yref) / np.maximum(nrm, 1e-300)))
    assert err <= TOL, f"row-normalised error {err}"
    # element bound: g and u carry fp32 summation error e = K 2^-23 sum|x||w|
    G = oracle.linear(xs, w.p, w.a, 2 * w.f)
    g, u = G[:, :w.f], G[:, w.f:]
    wd = f32_of_bits(oracle.dequantize(w.p, w.a, 2 * w.f * w.k)).astype(np.float64).reshape(2 * w.f, w.k)
    mag = np.abs(f32_of_bits(xs).astype(np.float64)) @ np.abs(wd).T
    K = w.k
    eg, eu = K * 2.0 ** -23 * mag[:, :w.f], K * 2.0 ** -23 * mag[:, w.f:]
    act = oracle.gelu_tanh(g)
    bound = (1.13 * eg * (np.abs(u) + eu) + np.abs(act) * eu
             + 2.0 ** -20 * (np.abs(g) + 1) * np.abs(u)    # fp32 activation
             + 2.0 ** -8 * np.abs(yref) + 1e-30)
    viol = np.abs(ys - yref) > bound
    assert not viol.any(), f"{int(viol.sum())} elements exceed the rounding bound"
    return y


def test_gemma3_gate_up_m2048_sampled_rows():
    """The gate/up workload (F = 15360, K = 3840, M = 2048, 0.1 % outliers x20)."""
    cfg = workloads.GATE_UP
    w = Pair(workloads.bits(workloads.make_weight(cfg)))
    assert w.f == 15360
    x = workloads.bits(workloads.make_activation(cfg))
    rows = np.sort(np.random.default_rng(5).choice(cfg.m, 24, replace=False))
    rows[0], rows[-1] = 0, cfg.m - 1
    check(x, w, rows=rows)


def test_gemma3_gate_up_skinny_m16():
    cfg = workloads.GATE_UP
    w = Pair(workloads.bits(workloads.make_weight(cfg)))
    x = workloads.bits(workloads.make_activation(cfg))[:16]
    check(x, w)


@pytest.mark.parametrize("M,F,K", [
    (128, 64, 64), (130, 100, 192), (257, 200, 128), (256, 32, 256),
    (512, 1000, 320), (1000, 384, 1024), (384, 130, 640),
])
def test_tile_path_ragged_shapes(M, F, K):
    w = Pair(rand_bits((2 * F, K), 0.05, M + 11 * F))
    check(rand_bits((M, K), 1.0, 3 * M + K), w)


@pytest.mark.parametrize("M,F,K", [
    (2048, 2432, 128),   # 19 pair tiles of 128 outputs x 4 tiles of 512 activation rows
    (1500, 2400, 320),   # ragged M and F (the last CTA's outputs partly past F), 5 K-slices
    (640, 4800, 192),    # 160 activation rows per accumulator, 3 K-slices
])
def test_pair_kernel_shapes(M, F, K):
    """Shapes the CTA-pair kernel takes (64 gate and 64 up rows per CTA, the
    epilogue exchanging halves through shared memory), on sampled rows."""
    w = Pair(rand_bits((2 * F, K), 0.05, M + 7 * F))
    rows = np.sort(np.random.default_rng(M + F).choice(M, 48, replace=False))
    rows[0], rows[-1] = 0, M - 1
    y = check(rand_bits((M, K), 1.0, 5 * M + K), w, rows=rows)
    assert np.array_equal(y, run(rand_bits((M, K), 1.0, 5 * M + K), w))


@pytest.mark.parametrize("M", [1, 7, 16, 17, 64, 100, 127])
def test_skinny_path_widths(M):
    F, K = 320, 1536
    w = Pair(rand_bits((2 * F, K), 0.05, 500 + M))
    check(rand_bits((M, K), 1.0, 600 + M), w)


def test_fused_matches_unfused_within_bf16():
    """nf4_linear over the [2F, K] weight, then gelu(g) * u in torch from the
    bf16 outputs: the fused result differs only by rounding g and u to bf16."""
    F, K, M = 512, 1024, 384
    w = Pair(rand_bits((2 * F, K), 0.05, 77))
    x = workloads.from_bits(rand_bits((M, K), 1.0, 78), DEV)
    fused = nf4.linear_geglu(x, w.pd, w.ad, F).float()
    G = nf4.linear(x, w.pd, w.ad, 2 * F).float()
    ref = torch.nn.functional.gelu(G[:, :F], approximate="tanh") * G[:, F:]
    scale = ref.abs().amax(dim=1, keepdim=True)
    assert ((fused - ref).abs() / scale).max().item() < 2e-2
    assert ((fused - ref).abs() <= 2.0 ** -6 * ref.abs() + 2.0 ** -7 * scale).float().mean().item() > 0.999


def test_deterministic_and_zero_weight():
    F, K = 256, 512
    w = Pair(rand_bits((2 * F, K), 0.05, 3))
    for m in (16, 300):
        x = rand_bits((m, K), 1.0, m)
        assert np.array_equal(run(x, w), run(x, w))
    z = Pair(np.zeros((2 * F, K), np.uint16))
    assert np.all(run(rand_bits((200, K), 1.0, 4), z) == 0)


def test_no_error_recorded():
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
