"""GPU parity of nf4_linear against the CPU oracle.

nf4_linear accumulates in fp32 in its own order, so it is compared within a
tolerance: per output row m, max_n |Y - Yref| / ||Yref[m, :]||_2 <= 1e-2, with
Yref the oracle's fp64 product of X and the dequantized weight.  A second,
much tighter per-element bound is also checked -- bf16 output rounding plus
fp32 summation error:

    |Y - Yref| <= 2^-8 |Yref| + K * 2^-23 * sum_k |x_k| |w_k|   (+ tiny)

which a dropped K-slice, a wrong scale or a transposed tile would break.
W is always quantized by the oracle; the GPU only multiplies.  Large
workloads are checked on seeded row samples (rows of Y are independent).
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


def row_err(y, yref):
    nrm = np.linalg.norm(yref, axis=1, keepdims=True)
    return float(np.max(np.abs(y - yref) / np.maximum(nrm, 1e-300)))


def check_bound(y, yref, x_bits, wdeq_f64):
    K = x_bits.shape[1]
    ax = np.abs(f32_of_bits(x_bits).astype(np.float64))
    mag = ax @ np.abs(wdeq_f64).T
    bound = 2.0 ** -8 * np.abs(yref) + K * 2.0 ** -23 * mag + 1e-30
    viol = np.abs(y - yref) > bound
    assert not viol.any(), f"{int(viol.sum())} elements exceed the rounding bound"


class Quantized:
    def __init__(self, w_bits_2d):
        self.n, self.k = w_bits_2d.shape
        self.p, self.a = oracle.quantize(w_bits_2d)
        self.pd = torch.from_numpy(self.p).to(DEV)
        self.ad = torch.from_numpy(self.a).to(DEV)
        self._wdeq = None

    def wdeq(self):
        if self._wdeq is None:
            d = oracle.dequantize(self.p, self.a, self.n * self.k)
            self._wdeq = f32_of_bits(d).astype(np.float64).reshape(self.n, self.k)
        return self._wdeq


def run_linear(x_bits, q):
    x = workloads.from_bits(x_bits, DEV)
    y = nf4.linear(x, q.pd, q.ad, q.n)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64)


def check(x_bits, q, rows=None, bound=True):
    y = run_linear(x_bits, q)
    xs = x_bits if rows is None else x_bits[rows]
    ys = y if rows is None else y[rows]
    yref = oracle.linear(xs, q.p, q.a, q.n)
    err = row_err(ys, yref)
    assert err <= TOL, f"row-normalised error {err}"
    if bound:
        check_bound(ys, yref, xs, q.wdeq())
    return y, err


def rand_bits(shape, std, seed):
    rs = np.random.default_rng(seed)
    t = torch.from_numpy((rs.standard_normal(shape) * std).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- the five workloads


def test_tiny_full():
    cfg = workloads.TINY
    q = Quantized(workloads.bits(workloads.make_weight(cfg)))
    check(workloads.bits(workloads.make_activation(cfg)), q)


@pytest.mark.parametrize("cfg", [workloads.Q_PROJ, workloads.GATE_UP, workloads.DOWN], ids=lambda c: c.name)
def test_projection_m2048_sampled_rows(cfg):
    q = Quantized(workloads.bits(workloads.make_weight(cfg)))
    x = workloads.bits(workloads.make_activation(cfg))
    rs = np.random.default_rng(cfg.x_seed)
    rows = np.sort(rs.choice(cfg.m, 48, replace=False))
    rows[0] = 0
    rows[-1] = cfg.m - 1
    check(x, q, rows=rows, bound=(cfg.n * cfg.k <= 4096 * 3840 * 4))


def test_down_proj_skinny_full():
    cfg = workloads.DOWN_SKINNY
    q = Quantized(workloads.bits(workloads.make_weight(cfg)))
    x = workloads.bits(workloads.make_activation(cfg))
    check(x, q)


def test_skinny_rows_equal_rows_of_full_batch():
    """Batched-vs-solo: the 16-row call (warp-MMA kernel) matches the same 16
    rows of the 2048-row call (CTA-pair kernel) to within fp32 reordering +
    bf16 rounding."""
    q = Quantized(workloads.bits(workloads.make_weight(workloads.DOWN)))
    xf = workloads.bits(workloads.make_activation(workloads.DOWN))
    xs = workloads.bits(workloads.make_activation(workloads.DOWN_SKINNY))
    assert np.array_equal(xs, xf[:16])
    yf = run_linear(xf, q)[:16]
    ys = run_linear(xs, q)
    scale = np.linalg.norm(yf, axis=1, keepdims=True)
    assert np.max(np.abs(yf - ys) / scale) < 1e-3


# ---------------------------------------------------------------- shapes and edges


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64), (256, 256, 128), (130, 256, 192), (255, 512, 256), (257, 300, 128),
    (384, 264, 640), (512, 1000, 320), (129, 8, 64), (200, 200, 448), (1000, 768, 1024),
])
def test_tile_path_ragged_shapes(M, N, K):
    q = Quantized(rand_bits((N, K), 0.02, M * 7 + N))
    check(rand_bits((M, K), 1.0, M + K), q)


@pytest.mark.parametrize("M,N,K", [
    (500, 1250, 4096),     # 20 tiles, ragged M and N, 32 stages
    (1024, 2048, 3840),    # 64 tiles (k_proj-like)
    (2048, 640, 15360),    # long K: 40 tiles of 120 stages
])
def test_tile_path_larger_shapes(M, N, K):
    """Larger ragged shapes on the tile path, against the oracle (sampled rows
    for the larger ones), and determinism: two calls give identical bits."""
    q = Quantized(rand_bits((N, K), 0.02, M + 3 * N))
    x_bits = rand_bits((M, K), 1.0, K + M)
    rows = None if M * N * K <= 500 * 1250 * 4096 else np.sort(
        np.random.default_rng(M).choice(M, 40, replace=False))
    y1, _ = check(x_bits, q, rows=rows)
    y2 = run_linear(x_bits, q)
    assert np.array_equal(y1, y2)


@pytest.mark.parametrize("M,N,K", [
    (1500, 10000, 192),    # ragged M (the last tile's second accumulator half partly past M) and N, odd block count
    (2047, 4100, 320),     # 4 tiles of 512 rows, the last one ragged; a partial weight tile
    (4096, 2048, 128),     # 8 tiles of 512 rows, one stage
    (2000, 20000, 256),    # 316 pair tiles (632 CTAs, several waves), ragged M and N
    (300, 10000, 128),     # 160 activation rows per accumulator, the second one partly past M
    (700, 30720, 192),     # 192 rows per accumulator, 2 tiles of 350 rows
    (850, 30720, 128),     # 224 rows per accumulator, 2 tiles of 425 rows
    (2048, 4864, 64),      # one K-slice: one stage, its second half empty
])
def test_wide_path_shapes(M, N, K):
    """Shapes the CTA-pair kernel takes (expanded weights in shared memory,
    pair tiles of 256 x 512): against the oracle on sampled rows, plus
    determinism."""
    q = Quantized(rand_bits((N, K), 0.02, M + 5 * N))
    x_bits = rand_bits((M, K), 1.0, K + 2 * M)
    rows = np.sort(np.random.default_rng(M + 1).choice(M, 48, replace=False))
    rows[-1] = M - 1
    y1, _ = check(x_bits, q, rows=rows)
    assert np.array_equal(y1, run_linear(x_bits, q))


@pytest.mark.parametrize("M", [1, 2, 7, 15, 16, 17, 31, 33, 48, 64, 65, 100, 112, 127])
def test_skinny_path_all_widths(M):
    N, K = 640, 1536
    q = Quantized(rand_bits((N, K), 0.02, 1000 + M))
    check(rand_bits((M, K), 1.0, 2000 + M), q)


@pytest.mark.parametrize("N,K", [(64, 64), (72, 128), (1000, 64 * 50), (3840, 15360)])
def test_skinny_path_shapes(N, K):
    q = Quantized(rand_bits((N, K), 0.02, N + K))
    check(rand_bits((16, K), 1.0, K), q, bound=(N * K <= 1 << 22))


def test_outlier_weights_and_large_activations():
    w = rand_bits((512, 1024), 0.02, 5).copy()
    flat = w.reshape(-1)
    idx = np.arange(0, flat.size, 997)
    flat[idx] = rand_bits((idx.size,), 0.4, 6)
    q = Quantized(w)
    check(rand_bits((256, 1024), 30.0, 7), q)


def test_zero_weight_blocks_give_zero_output():
    w = np.zeros((256, 512), np.uint16)
    q = Quantized(w)
    y = run_linear(rand_bits((128, 512), 1.0, 8), q)
    assert np.all(y == 0)


def test_deterministic():
    cfg = workloads.TINY
    q = Quantized(workloads.bits(workloads.make_weight(cfg)))
    for m in (16, 300):
        x = rand_bits((m, cfg.k), 1.0, m)
        assert np.array_equal(run_linear(x, q), run_linear(x, q))


def test_matches_cublas_on_dequantized_weight():
    """Against torch.matmul (cuBLAS) of the same dequantized bf16 weight: both
    are fp32-accumulated, so they agree to about one bf16 rounding."""
    cfg = workloads.Q_PROJ
    q = Quantized(workloads.bits(workloads.make_weight(cfg)))
    x = workloads.make_activation(cfg).to(DEV)
    wd = workloads.from_bits(oracle.dequantize(q.p, q.a, q.n * q.k), DEV).view(q.n, q.k)
    y = nf4.linear(x, q.pd, q.ad, q.n).float()
    ref = torch.matmul(x, wd.t()).float()
    diff = (y - ref).abs()
    tol = 2.0 ** -7 * ref.abs() + 1e-3
    frac_bad = (diff > tol).float().mean().item()
    assert frac_bad < 1e-3, frac_bad


HEADER = 4096   # the skinny workspace's arrival counters: zero before a call, zero after it


@pytest.mark.parametrize("M", [16, 40])
def test_workspace_reuse_and_user_workspace(M):
    """A caller's workspace: zeroed once, then reused.  Every call leaves the
    counter header zero again (on both skinny kernels); the rest of it may hold
    anything (filled with 0xFF here) -- the partials are written before they
    are read.  Too small a workspace is refused before any launch."""
    N, K = 512, 2048
    q = Quantized(rand_bits((N, K), 0.02, 9))
    x_bits = rand_bits((M, K), 1.0, 10)
    x = workloads.from_bits(x_bits, DEV)
    st, need = nf4.nf4_linear_workspace_size(M, N, K)
    assert st == nf4.NF4_OK and need > HEADER
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    ws[:HEADER] = 0
    y1 = nf4.linear(x, q.pd, q.ad, N, workspace=ws)
    y2 = nf4.linear(x, q.pd, q.ad, N, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert int(ws[:HEADER].count_nonzero()) == 0
    yref = oracle.linear(x_bits, q.p, q.a, N)
    assert row_err(y1.float().cpu().numpy().astype(np.float64), yref) <= TOL
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(nf4.NF4Error):
        nf4.linear(x, q.pd, q.ad, N, workspace=small)


# ---------------------------------------------------------------- the M <= 16 warp-MMA kernel


@pytest.mark.parametrize("M,N,K", [
    (16, 1000, 64 * 37),    # ragged N, odd block count: a partial last stage, K split
    (5, 40000, 256),        # more tiles than SMs: two waves, no K split
    (8, 2048, 3840),        # k_proj shape, one activation octet
    (9, 4096, 3840),        # q_proj shape, two octets, ragged rows
    (16, 640, 64 * 3),      # fewer blocks than a stage
    (3, 130, 64 * 9),       # a tile larger than the weight
    (16, 3840, 4096),       # o_proj shape
    (16, 20480, 512),       # 256-row tiles (the 3-slot ring)
    (7, 20480, 512),        # 256-row tiles, one activation octet
])
def test_small_batch_kernel_shapes(M, N, K):
    q = Quantized(rand_bits((N, K), 0.02, 11 * M + N))
    x_bits = rand_bits((M, K), 1.0, M + 3 * K)
    y1, _ = check(x_bits, q, bound=(N * K <= 1 << 23))
    assert np.array_equal(y1, run_linear(x_bits, q))     # deterministic: fixed split order


@pytest.mark.parametrize("M,N", [(16, 384), (64, 384), (256, 384), (2048, 4864)],
                         ids=["warp_mma", "split_tcgen05", "tile_tcgen05", "cta_pair"])
def test_absmax_not_a_bf16_value(M, N):
    """Scales that are not bf16 values (a weight quantized at fp32, then used
    at bf16): every kernel path must still multiply by the exact fp32 absmax
    and round once, which is what nf4_dequantize (and the oracle) compute
    (sampled rows for the large batch)."""
    K = 1024
    q = Quantized(rand_bits((N, K), 0.02, 21))
    bumped = (q.a.view(np.uint32) | np.uint32(0x5a5)).view(np.float32)   # low fraction bits set
    q.a = bumped.copy()
    q.ad = torch.from_numpy(q.a).to(DEV)
    q._wdeq = None
    rows = None if M <= 256 else np.sort(np.random.default_rng(M).choice(M, 32, replace=False))
    check(rand_bits((M, K), 1.0, 22), q, rows=rows)


@pytest.mark.parametrize("cfg,reps", [(workloads.Q_PROJ, 100), (workloads.GATE_UP, 20)], ids=["q_proj", "gate_up"])
def test_pair_kernel_repeatable_under_load(cfg, reps):
    """Back-to-back calls of the CTA-pair kernel on the Gemma3 shapes at
    M = 2048 (one wave, and several), each into its own output: every result
    equals the first bit for bit.  The kernel is deterministic, so a read of
    an expanded-weight or activation slot before its writes were visible --
    the odd CTA signals the even one with a CTA-scope release -- would show
    here as a rare difference."""
    w = workloads.make_weight(cfg, device=DEV)
    p, a = nf4.quantize(w)
    del w
    x = workloads.make_activation(cfg, device=DEV)
    ref = nf4.linear(x, p, a, cfg.n)
    outs = [torch.empty_like(ref) for _ in range(4)]
    for i in range(reps):
        nf4.linear(x, p, a, cfg.n, out=outs[i % 4])
        if i % 4 == 3:
            torch.cuda.synchronize()
            for o in outs:
                assert torch.equal(o, ref)
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK


def test_no_error_recorded():
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK


@pytest.mark.parametrize("m,n,k", [(256, 640, 1536), (2048, 4864, 256)], ids=["tile_kernel", "cta_pair_kernel"])
def test_cuda_graph_replay_matches_eager(m, n, k):
    """The calls are stream-ordered with no host synchronisation, so a whole
    step (quantize, dequantize, linear at M = m and M = 16) captures into a
    CUDA graph -- the CTA-pair kernel's cluster launch included; replays give
    the eager results bit for bit (the kernels are deterministic) and match
    the oracle (on sampled rows for the large batch)."""
    rs = np.random.default_rng(7)
    w = torch.from_numpy((rs.standard_normal((n, k)) * 0.02).astype(np.float32)).to(torch.bfloat16).to(DEV)
    x = torch.from_numpy(rs.standard_normal((m, k)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    xs = x[:16].contiguous()
    p = torch.empty(n * k // 2, dtype=torch.uint8, device=DEV)
    a = torch.empty(n * k // 64, dtype=torch.float32, device=DEV)
    wd = torch.empty(n * k, dtype=torch.bfloat16, device=DEV)
    y = torch.empty(m, n, dtype=torch.bfloat16, device=DEV)
    ys = torch.empty(16, n, dtype=torch.bfloat16, device=DEV)
    _, ws_bytes = nf4.nf4_linear_workspace_size(16, n, k)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)

    def step():
        nf4.quantize(w, out=(p, a))
        nf4.dequantize(p, a, n * k, out=wd)
        nf4.linear(x, p, a, n, out=y)
        nf4.linear(xs, p, a, n, out=ys, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in (p, a, wd, y, ys)]
    for t in (p, a, wd, y, ys):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for t in (p, a, wd, y, ys):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for got, ref in zip((p, a, wd, y, ys), eager):
            assert torch.equal(got, ref)
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
    q = Quantized(workloads.bits(w.cpu()))
    assert np.array_equal(p.cpu().numpy(), q.p) and np.array_equal(a.cpu().numpy(), q.a)
    rows = np.arange(m) if m <= 256 else np.sort(np.random.default_rng(m).choice(m, 64, replace=False))
    yref = oracle.linear(workloads.bits(x.cpu())[rows], q.p, q.a, n)
    assert row_err(f32_of_bits(workloads.bits(y.cpu())[rows]).astype(np.float64), yref) < TOL
