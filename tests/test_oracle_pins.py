"""Pins for the CPU oracle: each checks it against something other than itself.

The oracle follows the diffuseR page "Gemma3 NF4 on GPU" (pull request #39,
Summary): NF4-packed projection weights, dequantized and multiplied at the
compute dtype, with forward parity checked by cosine > 0.99.  What the page
leaves open (codebook, block 64, fp32 absmax, nibble order, tie rule) is
fixed by the readings listed in the oracle's C file.  Each test below pins one
of those against a published table, a closed form, an invariant, a library
routine or a brute force, chosen so that a dropped term, a wrong index, a
swapped nibble or a transposed operand fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BLOCK = 64


def golden_codebook():
    vals = []
    with open(os.path.join(GOLDEN, "nf4_codebook.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return np.array(vals, dtype=np.float32)


def bf16_bits_of(values_f32):
    """bf16 bit patterns by torch's own fp32 -> bf16 cast (round to nearest even)."""
    t = torch.tensor(np.asarray(values_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f32_of_bits(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- codebook


def test_codebook_is_the_published_table():
    assert np.array_equal(oracle.codebook().view(np.uint32), golden_codebook().view(np.uint32))


def test_codebook_by_quantile_construction():
    """NF4 is built from normal quantiles: 8 positive points from
    linspace(offset, 0.5, 9) and 7 negative ones from linspace(offset, 0.5, 8),
    the 0.5 end dropped, plus zero, normalised by the largest (QLoRA appendix)."""
    from scipy.stats import norm
    offset = 0.9677083
    pos = norm.ppf(np.linspace(offset, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(offset, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, [0.0], neg]))
    v /= v.max()
    c = oracle.codebook().astype(np.float64)
    assert np.max(np.abs(c - v)) < 2e-7
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0
    assert np.all(np.diff(c) > 0)
    assert (c < 0).sum() == 7 and (c > 0).sum() == 8


# ---------------------------------------------------------------- code selection


def _midpoints():
    c = oracle.codebook().astype(np.float64)
    return (c[:-1] + c[1:]) / 2.0   # exact: fp32 sums and halves fit in fp64


def test_code_is_count_of_midpoints_below():
    """Nearest code with ties to the lower index equals the number of exact
    midpoints strictly below n.  Checked on every fp32 within 2^15 ulps of each
    midpoint, on each codebook value, on signed zeros and on a random sample."""
    mids = _midpoints()
    pieces = []
    for m in mids:
        # neighbouring bit patterns are neighbouring values on either side of m
        b = np.float32(m).view(np.int32).astype(np.int64)
        rng = np.arange(b - (1 << 15), b + (1 << 15), dtype=np.int64)
        pieces.append(rng.astype(np.uint32).view(np.float32))
    pieces.append(oracle.codebook())
    pieces.append(np.array([0.0, -0.0, 1e-30, -1e-30, 1.0, -1.0], dtype=np.float32))
    rs = np.random.default_rng(7)
    pieces.append(rs.uniform(-1, 1, 1 << 20).astype(np.float32))
    n = np.concatenate(pieces)
    n = n[np.abs(n) <= 1.0]
    got = oracle.nearest_code(n)
    want = np.searchsorted(mids, n.astype(np.float64), side="left")
    assert np.array_equal(got, want.astype(np.uint8))
    # each codebook value selects its own index
    assert np.array_equal(oracle.nearest_code(oracle.codebook()), np.arange(16, dtype=np.uint8))


@pytest.mark.slow
def test_code_selection_exhaustive_fp32():
    """Every fp32 in [-1, 1]: codes are monotone in n, step by one, and each of
    the 15 steps sits exactly at its midpoint (last value <= m_j, next > m_j)."""
    mids = _midpoints()
    chunk = 1 << 26
    for sign in (0, 1):
        top = int(np.float32(1.0).view(np.uint32))  # 0x3f800000
        start_code = 7
        prev_code = None
        prev_val = None
        jumps = []
        for lo in range(0, top + 1, chunk):
            hi = min(lo + chunk, top + 1)
            bits = np.arange(lo, hi, dtype=np.uint32)
            if sign:
                bits |= np.uint32(0x80000000)
            vals = bits.view(np.float32)
            codes = oracle.nearest_code(vals).astype(np.int16)
            if prev_code is None:
                assert codes[0] == start_code
            else:
                codes_ext = np.concatenate([[prev_code], codes])
                vals_ext = np.concatenate([[prev_val], vals])
                codes, vals = codes_ext, vals_ext
            d = np.diff(codes)
            step = -1 if sign else 1
            assert np.all((d == 0) | (d == step))
            for i in np.flatnonzero(d):
                jumps.append((float(vals[i]), float(vals[i + 1]), int(codes[i]), int(codes[i + 1])))
            prev_code = codes[-1]
            prev_val = vals[-1]
        if sign == 0:
            assert prev_code == 15 and len(jumps) == 8
            for j, (a, b, ca, cb) in enumerate(jumps):
                m = mids[7 + j]
                assert (ca, cb) == (7 + j, 8 + j)
                assert a <= m < b
        else:
            assert prev_code == 0 and len(jumps) == 7
            for j, (a, b, ca, cb) in enumerate(jumps):
                m = mids[6 - j]
                assert (ca, cb) == (7 - j, 6 - j)
                # values fall as bits rise: a > b; code 6-j is taken at and below m (tie -> lower)
                assert b <= m < a


# ---------------------------------------------------------------- quantize


def _brute_quantize(w_bits, block=BLOCK):
    """Independent restatement, one element at a time in Python."""
    cb = [float(v) for v in golden_codebook()]
    w = [float(v) for v in f32_of_bits(w_bits)]
    codes, scales = [], []
    for b0 in range(0, len(w), block):
        blk = w[b0:b0 + block]
        am = max(abs(v) for v in blk)
        scales.append(am)
        for v in blk:
            if am == 0.0:
                codes.append(7)
                continue
            n = float(np.float32(v) / np.float32(am))
            dists = [abs(n - c) for c in cb]
            codes.append(dists.index(min(dists)))   # first minimum = lower index on a tie
    packed = bytes((codes[2 * j] << 4) | codes[2 * j + 1] for j in range(len(codes) // 2))
    return np.frombuffer(packed, dtype=np.uint8), np.array(scales, dtype=np.float32)


def _special_weights():
    rs = np.random.default_rng(3)
    rows = []
    rows.append(np.zeros(64, np.float32))                                   # all-zero block
    rows.append(np.full(64, -0.0, np.float32))                              # negative zeros
    r = rs.normal(0, 0.02, 64).astype(np.float32); r[5] = -0.25; rows.append(r)   # max is negative
    cb = golden_codebook()
    mids = ((cb[:-1].astype(np.float64) + cb[1:]) / 2)
    r = np.zeros(64, np.float32); r[0] = 1.0; r[1:16] = mids.astype(np.float32); rows.append(r)
    r = rs.normal(0, 1e-3, 64).astype(np.float32); r[63] = 3.0; rows.append(r)      # one outlier
    r = np.array([(-1) ** i * 2.0 ** -(i % 30) for i in range(64)], np.float32); rows.append(r)
    w = np.concatenate(rows + [rs.normal(0, 0.02, 64 * 4).astype(np.float32)])
    return bf16_bits_of(w)


def test_quantize_brute_force_tiny():
    w = _special_weights()
    p, a = oracle.quantize(w)
    bp, ba = _brute_quantize(w)
    assert np.array_equal(p, bp)
    assert np.array_equal(a.view(np.uint32), ba.view(np.uint32))


def test_quantize_partial_last_block():
    rs = np.random.default_rng(11)
    w = bf16_bits_of(rs.normal(0, 0.02, 100))
    p, a = oracle.quantize(w)
    assert p.size == 50 and a.size == 2
    bp, ba = _brute_quantize(w)
    assert np.array_equal(p, bp) and np.array_equal(a, ba)


def test_zero_blocks():
    w = bf16_bits_of(np.array([0.0] * 64 + [-0.0] * 64, np.float32))
    p, a = oracle.quantize(w)
    assert np.all(p == 0x77)
    assert np.all(a.view(np.uint32) == 0)
    y = oracle.dequantize(p, a, w.size)
    assert np.all(y == 0)       # +0.0 everywhere


def test_tiny_config_against_brute_force():
    w = workloads.bits(workloads.make_weight(workloads.TINY))
    p, a = oracle.quantize(w)
    bp, ba = _brute_quantize(w.ravel()[: 64 * 64])
    assert np.array_equal(p[: bp.size], bp) and np.array_equal(a[: ba.size], ba)


# ---------------------------------------------------------------- dequantize


def test_dequant_absmax_one_is_the_bf16_codebook():
    """All 256 bytes with absmax 1: first element = bf16(C[hi]), second = bf16(C[lo])."""
    packed = np.arange(256, dtype=np.uint8)
    absmax = np.ones(512 // BLOCK, np.float32)
    y = oracle.dequantize(packed, absmax, 512)
    cbb = bf16_bits_of(golden_codebook())
    want = np.empty(512, np.uint16)
    want[0::2] = cbb[np.arange(256) >> 4]
    want[1::2] = cbb[np.arange(256) & 15]
    assert np.array_equal(y, want)


@pytest.mark.parametrize("e", [-20, -5, 0, 3, 60])
def test_dequant_power_of_two_scale_is_exact(e):
    """A power-of-two absmax scales bf16(C) without rounding."""
    packed = np.arange(256, dtype=np.uint8)
    absmax = np.full(512 // BLOCK, 2.0 ** e, np.float32)
    y = f32_of_bits(oracle.dequantize(packed, absmax, 512)).astype(np.float64)
    cb = f32_of_bits(bf16_bits_of(golden_codebook())).astype(np.float64)
    want = np.empty(512)
    want[0::2] = cb[np.arange(256) >> 4] * 2.0 ** e
    want[1::2] = cb[np.arange(256) & 15] * 2.0 ** e
    assert np.array_equal(y, want)


def test_dequant_matches_torch_rounding():
    """Arbitrary fp32 scales: y equals torch's bf16 cast of the fp32 product."""
    rs = np.random.default_rng(5)
    packed = rs.integers(0, 256, 64 * 32, dtype=np.uint8)
    absmax = rs.uniform(1e-3, 2.0, 64).astype(np.float32)
    y = oracle.dequantize(packed, absmax, packed.size * 2)
    cb = torch.tensor(golden_codebook()).to(torch.bfloat16).float()
    codes = np.empty(packed.size * 2, np.int64)
    codes[0::2] = packed >> 4
    codes[1::2] = packed & 15
    prod = cb[torch.from_numpy(codes)] * torch.from_numpy(np.repeat(absmax, BLOCK))
    want = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, want)


def _roundtrip_cases():
    t = workloads.bits(workloads.make_weight(workloads.TINY))
    g = workloads.bits(workloads.make_weight(workloads.GATE_UP, rows=slice(0, 64)))
    return [t.ravel(), g.ravel(), _special_weights()]


def test_max_element_is_exact():
    """In a nonzero block the largest |w| normalises to +-1, takes code 0 or 15
    and comes back bit-exact."""
    for w in _roundtrip_cases():
        p, a = oracle.quantize(w)
        y = oracle.dequantize(p, a, w.size)
        wf = np.abs(f32_of_bits(w)).reshape(-1, BLOCK)
        for b in range(wf.shape[0]):
            if a[b] == 0:
                continue
            i = b * BLOCK + int(np.argmax(wf[b]))
            code = (p[i // 2] >> 4) if i % 2 == 0 else (p[i // 2] & 15)
            assert code in (0, 15)
            assert y[i] == w[i]


def test_round_trip_error_bound():
    """|w - y| <= (half the largest codebook gap + 2^-9 + 2^-22) * absmax + half a bf16 ulp of y."""
    half_gap = (float(golden_codebook()[1]) - float(golden_codebook()[0])) / 2
    assert abs(half_gap - 0.15190359950065613) < 1e-9
    for w in _roundtrip_cases():
        p, a = oracle.quantize(w)
        y = oracle.dequantize(p, a, w.size)
        wf = f32_of_bits(w).astype(np.float64)
        yf = f32_of_bits(y).astype(np.float64)
        am = np.repeat(a.astype(np.float64), BLOCK)[: w.size]
        ulp = np.where(yf == 0, 0, 2.0 ** (np.floor(np.log2(np.abs(yf) + (yf == 0))) - 7))
        bound = (half_gap + 2.0 ** -9 + 2.0 ** -22) * am + ulp / 2
        assert np.all(np.abs(wf - yf) <= bound)


def test_requantize_is_idempotent():
    """quantize(dequantize(q)) == q: catches any mismatch in nibble order or
    scale handling between the two directions."""
    for w in _roundtrip_cases():
        p, a = oracle.quantize(w)
        y = oracle.dequantize(p, a, w.size)
        p2, a2 = oracle.quantize(y)
        assert np.array_equal(p, p2) and np.array_equal(a, a2)


# ---------------------------------------------------------------- linear


def test_linear_matches_library_matmul():
    cfg = workloads.TINY
    w = workloads.bits(workloads.make_weight(cfg))
    x = workloads.bits(workloads.make_activation(cfg))
    p, a = oracle.quantize(w)
    y = oracle.linear(x, p, a, cfg.n)
    wd = f32_of_bits(oracle.dequantize(p, a, w.size)).astype(np.float64).reshape(cfg.n, cfg.k)
    xd = f32_of_bits(x).astype(np.float64).reshape(cfg.m, cfg.k)
    ref = xd @ wd.T
    assert y.shape == (cfg.m, cfg.n)
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_linear_brute_force_small():
    rs = np.random.default_rng(9)
    M, N, K = 3, 2, 128
    w = bf16_bits_of(rs.normal(0, 0.02, N * K))
    x = bf16_bits_of(rs.normal(0, 1, M * K)).reshape(M, K)
    p, a = oracle.quantize(w)
    y = oracle.linear(x, p, a, N)
    wd = [float(v) for v in f32_of_bits(oracle.dequantize(p, a, N * K))]
    xf = [float(v) for v in f32_of_bits(x.ravel())]
    for m in range(M):
        for n in range(N):
            terms = [xf[m * K + k] * wd[n * K + k] for k in range(K)]   # exact in fp64
            assert abs(y[m, n] - math.fsum(terms)) <= 1e-13 * sum(abs(t) for t in terms)


def _cosine(a, b):
    a = a.ravel(); b = b.ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


@pytest.mark.parametrize("cfg,wrows,xrows", [
    (workloads.TINY, None, None),
    (workloads.Q_PROJ, slice(0, 256), 64),
    (workloads.GATE_UP, slice(0, 512), 64),
    (workloads.DOWN, slice(0, 128), 32),
])
def test_forward_parity_cosine(cfg, wrows, xrows):
    """Quantized vs unquantized forward: cosine > 0.99, the page's parity threshold."""
    w = workloads.bits(workloads.make_weight(cfg, rows=wrows))
    x = workloads.bits(workloads.make_activation(cfg))
    if xrows:
        x = x[:xrows]
    n = w.shape[0]
    p, a = oracle.quantize(w)
    yq = oracle.linear(x, p, a, n)
    wf = f32_of_bits(w).astype(np.float64)
    xf = f32_of_bits(x).astype(np.float64)
    y = xf @ wf.T
    assert _cosine(y, yq) > 0.99


def test_oracle_digest_is_stable():
    """The oracle's bits on two seeded cases equal the stored digests (written by
    tests/golden/make_oracle_digest.py, which calls only the oracle)."""
    import importlib.util
    import json
    spec = importlib.util.spec_from_file_location(
        "make_oracle_digest", os.path.join(GOLDEN, "make_oracle_digest.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "oracle_digest.json")) as f:
        want = json.load(f)
    got = mod.compute()
    for name, d in want.items():
        g = got[name]
        for key in ("input_w", "input_x", "packed", "absmax", "dequant"):
            assert g[key] == d[key], (name, key)
        assert np.allclose(g["linear_first_row"], d["linear_first_row"], rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- gate/up pair (GeGLU)


def test_gelu_tanh_closed_forms():
    """gelu(0) = 0; gelu(x) - gelu(-x) = x exactly in real arithmetic (the
    tanh terms cancel); for large |x| the tanh saturates so gelu(x) = x and
    gelu(-x) = 0; near zero gelu(x) = x/2 + sqrt(2/pi) x^2 / 2 + O(x^4)."""
    x = np.array([0.0, 1e-6, 0.25, 0.5, 1.0, 2.0, 3.0, 8.0, 30.0])
    g, gm = oracle.gelu_tanh(x), oracle.gelu_tanh(-x)
    assert g[0] == 0.0
    assert np.allclose(g - gm, x, rtol=4e-16, atol=0)
    assert g[-2] == 8.0 and g[-1] == 30.0 and gm[-2] == 0.0 and gm[-1] == 0.0
    small = 0.5e-6 + math.sqrt(2 / math.pi) * 0.5e-12
    assert abs(g[1] - small) <= 1e-18


def test_gelu_tanh_matches_torch():
    """torch's own tanh-approximate GELU in fp64 (a library routine)."""
    x = np.linspace(-10, 10, 20001)
    want = torch.nn.functional.gelu(torch.tensor(x, dtype=torch.float64), approximate="tanh").numpy()
    assert np.max(np.abs(oracle.gelu_tanh(x) - want)) <= 2e-15


def test_gelu_tanh_is_the_tanh_form_not_erf():
    """Against the exact GELU x * Phi(x): the tanh form stays within 5e-4 of
    it (largest gap near x = -2.7) but is not it."""
    x = np.linspace(-6, 6, 12001)
    exact = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in x])
    gap = np.max(np.abs(oracle.gelu_tanh(x) - exact))
    assert 4e-4 < gap < 5e-4


def test_linear_geglu_brute_force_small():
    """Gate rows first, up rows second, activation on the gate: a plain Python
    restatement with math.fsum and math.tanh on a tiny case."""
    rs = np.random.default_rng(21)
    M, F, K = 3, 3, 128
    w = bf16_bits_of(rs.normal(0, 0.05, 2 * F * K))
    x = bf16_bits_of(rs.normal(0, 1, M * K)).reshape(M, K)
    p, a = oracle.quantize(w)
    y = oracle.linear_geglu(x, p, a, F)
    wd = [float(v) for v in f32_of_bits(oracle.dequantize(p, a, 2 * F * K))]
    xf = [float(v) for v in f32_of_bits(x.ravel())]

    def dot(m, row):
        return math.fsum(xf[m * K + k] * wd[row * K + k] for k in range(K))

    def gelu(v):
        return 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))

    for m in range(M):
        for n in range(F):
            want = gelu(dot(m, n)) * dot(m, F + n)
            assert abs(y[m, n] - want) <= 1e-13 * max(1.0, abs(want))
    # swapping the halves gives a different answer on this case
    swapped = [[gelu(dot(m, F + n)) * dot(m, n) for n in range(F)] for m in range(M)]
    assert np.max(np.abs(y - np.array(swapped))) > 1e-3


# ---------------------------------------------------------------- fp16 and fp32 compute dtypes


def f16_bits_of(values):
    """binary16 bit patterns by numpy's fp32 -> fp16 cast (round to nearest even)."""
    return np.asarray(values, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_f16_widening_matches_numpy_on_every_pattern():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32_array(h)
    want = h.view(np.float16).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def test_f16_rounding_matches_numpy():
    """fp32 -> fp16 round to nearest even against numpy's cast: random bit
    patterns over the whole fp32 range, every fp16 value and the midpoints
    between neighbours (ties), the subnormal boundary and the overflow edge."""
    rs = np.random.default_rng(17)
    rand = rs.integers(0, 1 << 32, 400000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    rand = rand[np.isfinite(rand)]
    f16 = np.arange(0, 0x7c00, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    mids = ((f16[:-1] + f16[1:]) / 2).astype(np.float32)            # exact in fp32: ties
    edges = np.array([65504, 65519.996, 65520, 65536, 1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                      2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 6e-8, 1e-30, 0.0], np.float32)
    for v in (rand, mids, -mids, f16.astype(np.float32), edges, -edges):
        got = oracle.f32_to_f16_array(v)
        with np.errstate(over="ignore"):                 # numpy warns on values that round to inf
            want = v.astype(np.float16).view(np.uint16)
        assert np.array_equal(got, want)


def test_dequant_f16_absmax_one_is_the_f16_codebook():
    packed = np.arange(256, dtype=np.uint8)
    absmax = np.ones(8, np.float32)
    y = oracle.dequantize(packed, absmax, 512, dtype="f16")
    cb16 = f16_bits_of(golden_codebook())
    assert np.array_equal(y[0::2], cb16[packed >> 4]) and np.array_equal(y[1::2], cb16[packed & 15])


def test_dequant_f16_and_f32_match_numpy_products():
    """f16: numpy's fp16 of (fp32 of the fp16 codebook value) x absmax in fp32;
    f32: the fp32 codebook value x absmax in fp32, no rounding to a smaller type."""
    rs = np.random.default_rng(23)
    n = 64 * 300
    packed = rs.integers(0, 256, n // 2, dtype=np.uint16).astype(np.uint8)
    absmax = np.abs(rs.standard_normal(n // 64) * 10.0 ** rs.integers(-6, 4, n // 64)).astype(np.float32)
    absmax[::7] = f16_bits_of(absmax[::7]).view(np.float16).astype(np.float32)   # some fp16-exact scales
    codes = np.empty(n, np.int64)
    codes[0::2], codes[1::2] = packed >> 4, packed & 15
    am = np.repeat(absmax, 64)
    cb = golden_codebook()
    c16 = cb.astype(np.float16).astype(np.float32)
    want16 = (c16[codes] * am).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.dequantize(packed, absmax, n, dtype="f16"), want16)
    want32 = (cb[codes] * am).astype(np.float32)
    assert np.array_equal(oracle.dequantize(packed, absmax, n, dtype="f32").view(np.uint32), want32.view(np.uint32))


def _brute_quantize_values(w, block=BLOCK):
    """Independent restatement on plain Python floats (the element values)."""
    cb = [float(v) for v in golden_codebook()]
    w = [float(v) for v in w]
    codes, scales = [], []
    for b0 in range(0, len(w), block):
        blk = w[b0:b0 + block]
        am = max(abs(v) for v in blk)
        scales.append(am)
        for v in blk:
            if am == 0.0:
                codes.append(7)
                continue
            n = float(np.float32(v) / np.float32(am))
            dists = [abs(n - c) for c in cb]
            codes.append(dists.index(min(dists)))
    packed = bytes((codes[2 * j] << 4) | codes[2 * j + 1] for j in range(len(codes) // 2))
    return np.frombuffer(packed, dtype=np.uint8), np.array(scales, dtype=np.float32)


def test_quantize_f16_and_f32_brute_force():
    wb = _special_weights()                               # bf16 patterns of special blocks
    vals = f32_of_bits(wb)
    rs = np.random.default_rng(29)
    extra = (rs.standard_normal(64 * 6) * 0.03).astype(np.float32)
    extra[64:128] *= 1e-6                                 # fp16 subnormal range
    w32 = np.concatenate([vals, extra])
    w16 = f16_bits_of(w32)
    p, a = oracle.quantize(w16, dtype="f16")
    bp, ba = _brute_quantize_values(w16.view(np.float16).astype(np.float32))
    assert np.array_equal(p, bp) and np.array_equal(a.view(np.uint32), ba.view(np.uint32))
    p, a = oracle.quantize(w32, dtype="f32")
    bp, ba = _brute_quantize_values(w32)
    assert np.array_equal(p, bp) and np.array_equal(a.view(np.uint32), ba.view(np.uint32))


def test_quantize_is_dtype_blind_for_equal_values():
    """The same values quantize identically whatever type carries them: bf16
    and fp16 values widened exactly to fp32 give the bf16 / fp16 result."""
    rs = np.random.default_rng(31)
    v = (rs.standard_normal(64 * 40) * 0.02).astype(np.float32)
    b16 = bf16_bits_of(v)
    h16 = f16_bits_of(v)
    pb, ab = oracle.quantize(b16)
    assert all(np.array_equal(x, y) for x, y in zip((pb, ab), oracle.quantize(f32_of_bits(b16), dtype="f32")))
    ph, ah = oracle.quantize(h16, dtype="f16")
    assert all(np.array_equal(x, y) for x, y in
               zip((ph, ah), oracle.quantize(h16.view(np.float16).astype(np.float32), dtype="f32")))


def test_f16_round_trip_bound_and_exact_max():
    rs = np.random.default_rng(37)
    v = (rs.standard_normal(64 * 50) * 0.05).astype(np.float32)
    w16 = f16_bits_of(v)
    p, a = oracle.quantize(w16, dtype="f16")
    y = oracle.dequantize(p, a, v.size, dtype="f16").view(np.float16).astype(np.float64)
    w = w16.view(np.float16).astype(np.float64)
    am = np.repeat(a.astype(np.float64), 64)
    ulp = np.spacing(np.abs(y).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(w - y) <= (0.15190359950065613 + 2.0 ** -11) * am + ulp / 2 + 1e-12)
    blocks = w.reshape(-1, 64)
    idx = np.argmax(np.abs(blocks), axis=1)
    ymax = y.reshape(-1, 64)[np.arange(blocks.shape[0]), idx]
    assert np.array_equal(ymax, blocks[np.arange(blocks.shape[0]), idx])


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_linear_other_dtypes_brute_force(dtype):
    rs = np.random.default_rng(41)
    M, N, K = 3, 2, 128
    wv = (rs.standard_normal(N * K) * 0.02).astype(np.float32)
    xv = rs.standard_normal(M * K).astype(np.float32)
    w = f16_bits_of(wv) if dtype == "f16" else wv
    x = (f16_bits_of(xv) if dtype == "f16" else xv).reshape(M, K)
    p, a = oracle.quantize(w, dtype=dtype)
    y = oracle.linear(x, p, a, N, dtype=dtype)
    wd = oracle.dequantize(p, a, N * K, dtype=dtype)
    as_f = (lambda b: b.view(np.float16).astype(np.float64)) if dtype == "f16" else (lambda b: b.astype(np.float64))
    wd, xf = [float(t) for t in as_f(wd)], [float(t) for t in as_f(x.ravel())]
    for m in range(M):
        for n in range(N):
            terms = [xf[m * K + k] * wd[n * K + k] for k in range(K)]
            assert abs(y[m, n] - math.fsum(terms)) <= 1e-13 * sum(abs(t) for t in terms)
