"""GPU parity of nf4_quantize and nf4_dequantize against the CPU oracle.

Both operations have exactly one correct result, so the comparison is
bit-exact: packed bytes, absmax bits and dequantized bf16 bits.  Inputs are
the seeded synthetic workloads (Gemma3-12B projection shapes) plus edge
cases: empty, tiny, ragged (partial last block, sizes that are not a whole
number of kernel tiles), unaligned pointers, zero blocks, outliers.  The
dequant inputs come from the oracle's quantizer or from random bytes, never
from the GPU quantizer.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import nf4_weight_quantized_quantize_gb300 as nf4

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_dev_bits(a_u16):
    return workloads.from_bits(a_u16, DEV)


def gpu_quantize_bits(w_bits):
    w = to_dev_bits(w_bits)
    p, a = nf4.quantize(w)
    torch.cuda.synchronize()
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK
    return p.cpu().numpy(), a.cpu().numpy()


def gpu_dequantize(packed, absmax, numel):
    p = torch.from_numpy(np.ascontiguousarray(packed)).to(DEV)
    a = torch.from_numpy(np.ascontiguousarray(absmax)).to(DEV)
    y = nf4.dequantize(p, a, numel)
    torch.cuda.synchronize()
    return workloads.bits(y)


def check_quant_exact(w_bits):
    w_bits = np.ascontiguousarray(w_bits).ravel()
    p_ref, a_ref = oracle.quantize(w_bits)
    p, a = gpu_quantize_bits(w_bits)
    bad = np.flatnonzero(p != p_ref)
    assert bad.size == 0, f"{bad.size} packed bytes differ, first at {bad[:5]}: {p[bad[:5]]} vs {p_ref[bad[:5]]}"
    assert np.array_equal(a.view(np.uint32), a_ref.view(np.uint32))
    return p_ref, a_ref


def check_dequant_exact(packed, absmax, numel):
    y_ref = oracle.dequantize(packed, absmax, numel)
    y = gpu_dequantize(packed, absmax, numel)
    bad = np.flatnonzero(y != y_ref)
    assert bad.size == 0, f"{bad.size} outputs differ, first at {bad[:5]}"


@pytest.mark.parametrize("cfg", [workloads.TINY, workloads.Q_PROJ, workloads.DOWN, workloads.GATE_UP],
                         ids=lambda c: c.name)
def test_quantize_dequantize_bit_exact_full(cfg):
    w = workloads.bits(workloads.make_weight(cfg))
    p, a = check_quant_exact(w)
    check_dequant_exact(p, a, w.size)


@pytest.mark.parametrize("numel", [2, 62, 64, 66, 100, 128, 1000, 1024, 1026, 4096 + 64 + 2,
                                   64 * 8 * 37 + 10, 512 * 1024 + 64 * 3 + 6])
def test_ragged_sizes(numel):
    rs = np.random.default_rng(numel)
    w = torch.from_numpy(rs.normal(0, 0.02, numel).astype(np.float32)).to(torch.bfloat16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    p, a = check_quant_exact(wb)
    check_dequant_exact(p, a, numel)


def test_special_blocks():
    blocks = [np.zeros(64), np.full(64, -0.0), np.linspace(-1, 1, 64), np.full(64, 3.5),
              np.r_[np.full(63, 1e-3), -7.0], np.r_[1.0, np.full(63, 1e-30)]]
    rs = np.random.default_rng(1)
    r = rs.normal(0, 0.02, 64 * 50); r[::97] *= 40; blocks.append(r)
    w = torch.from_numpy(np.concatenate(blocks).astype(np.float32)).to(torch.bfloat16)
    p, a = check_quant_exact(w.view(torch.int16).numpy().view(np.uint16))
    check_dequant_exact(p, a, w.numel())


def test_codebook_on_device_with_unit_scale():
    """All 256 bytes, absmax 1: the device LUT must give bf16(C[hi]), bf16(C[lo])."""
    packed = np.tile(np.arange(256, dtype=np.uint8), 4)
    absmax = np.ones(packed.size * 2 // 64, np.float32)
    check_dequant_exact(packed, absmax, packed.size * 2)


def test_dequant_random_bytes_and_scales():
    rs = np.random.default_rng(2)
    numel = 2 * (1 << 20) + 4 * 64 + 2
    packed = rs.integers(0, 256, numel // 2, dtype=np.uint8)
    absmax = rs.uniform(-3, 3, (numel + 63) // 64).astype(np.float32)   # negative scales too
    absmax[::17] = 0.0
    absmax[5::23] = np.float32(1e-40)                                    # subnormal fp32 scale
    check_dequant_exact(packed, absmax, numel)


@pytest.mark.parametrize("offset", [2, 6, 10])
def test_unaligned_pointers(offset):
    """Sub-tensors at odd offsets take the element-wise kernels and agree bit-exactly."""
    rs = np.random.default_rng(offset)
    n = 64 * 40
    base = torch.from_numpy(rs.normal(0, 0.02, n + 64).astype(np.float32)).to(torch.bfloat16).to(DEV)
    w = base[offset: offset + n]                        # 2*offset bytes: not 16-byte aligned
    packed = torch.empty(n // 2 + 3, dtype=torch.uint8, device=DEV)[1:1 + n // 2]   # odd address
    absmax = torch.empty(n // 64, dtype=torch.float32, device=DEV)
    st = nf4.nf4_quantize(w.data_ptr(), n, 64, packed.data_ptr(), absmax.data_ptr(), 0)
    assert st == nf4.NF4_OK
    torch.cuda.synchronize()
    p_ref, a_ref = oracle.quantize(workloads.bits(w))
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(absmax.cpu().numpy(), a_ref)
    out = torch.empty(n + 8, dtype=torch.bfloat16, device=DEV)[1:1 + n]
    st = nf4.nf4_dequantize(packed.data_ptr(), absmax.data_ptr(), n, 64, out.data_ptr(), 0)
    assert st == nf4.NF4_OK
    torch.cuda.synchronize()
    assert np.array_equal(workloads.bits(out), oracle.dequantize(p_ref, a_ref, n))


@pytest.mark.parametrize("packed_offset", [4, 8])
def test_packed_alignment_picks_the_kernel(packed_offset):
    """The vectorized quantizer stores 8 packed bytes per lane: packed output
    at a 4-byte (not 8-byte) boundary takes the element-wise kernel, at an
    8-byte boundary the vectorized one; both are bit-exact."""
    rs = np.random.default_rng(packed_offset)
    n = 64 * 300
    w = torch.from_numpy(rs.normal(0, 0.02, n).astype(np.float32)).to(torch.bfloat16).to(DEV)
    packed = torch.empty(n // 2 + 16, dtype=torch.uint8, device=DEV)[packed_offset:packed_offset + n // 2]
    absmax = torch.empty(n // 64, dtype=torch.float32, device=DEV)
    st = nf4.nf4_quantize(w.data_ptr(), n, 64, packed.data_ptr(), absmax.data_ptr(), 0)
    assert st == nf4.NF4_OK
    torch.cuda.synchronize()
    p_ref, a_ref = oracle.quantize(workloads.bits(w))
    assert np.array_equal(packed.cpu().numpy(), p_ref)
    assert np.array_equal(absmax.cpu().numpy(), a_ref)


def test_empty_is_a_no_op():
    assert nf4.nf4_quantize(0, 0, 64, 0, 0, 0) == nf4.NF4_OK
    assert nf4.nf4_dequantize(0, 0, 0, 64, 0, 0) == nf4.NF4_OK


def test_stream_ordering_on_side_stream():
    """Calls run on the caller's stream: results are ready after that stream syncs."""
    cfg = workloads.Q_PROJ
    w = workloads.make_weight(cfg, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        p, a = nf4.quantize(w)
        y = nf4.dequantize(p, a, w.numel())
    s.synchronize()
    p_ref, a_ref = oracle.quantize(workloads.bits(w))
    assert np.array_equal(p.cpu().numpy(), p_ref)
    assert np.array_equal(workloads.bits(y), oracle.dequantize(p_ref, a_ref, w.numel()))


def test_stack_all_weights_sampled_rows():
    """All 336 projection weights of the 48-layer stack, quantized and
    dequantized on the GPU; 8 seeded rows of each are checked bit-exactly
    against the oracle (blocks never straddle rows since K % 64 == 0)."""
    rs = np.random.default_rng(0)
    for layer in range(workloads.LAYERS):
        for pi in range(len(workloads.PROJECTIONS)):
            cfg = workloads.stack_layer(layer, pi)
            w = workloads.make_weight(cfg, device=DEV)
            p, a = nf4.quantize(w)
            y = nf4.dequantize(p, a, w.numel()).view(cfg.n, cfg.k)
            rows = np.sort(rs.choice(cfg.n, 8, replace=False))
            ri = torch.from_numpy(rows).to(DEV)
            wr = workloads.bits(w[ri])
            p_ref, a_ref = oracle.quantize(wr)
            pg = p.view(cfg.n, cfg.k // 2)[ri].cpu().numpy().ravel()
            ag = a.view(cfg.n, cfg.k // 64)[ri].cpu().numpy().ravel()
            assert np.array_equal(pg, p_ref), (layer, pi)
            assert np.array_equal(ag.view(np.uint32), a_ref.view(np.uint32)), (layer, pi)
            assert np.array_equal(workloads.bits(y[ri]).ravel(), oracle.dequantize(p_ref, a_ref, wr.size))
    assert nf4.nf4_last_error(torch.cuda.current_stream().cuda_stream) == nf4.NF4_OK


def _near_threshold_pairs(rel):
    """bf16 (absmax, w) pairs whose fp32 quotient w / absmax lies within `rel`
    (relative) of a decision midpoint between neighbouring codebook values."""
    import numpy as np
    cb = np.array(oracle.codebook(), dtype=np.float64)
    mids = (cb[:-1] + cb[1:]) / 2
    pairs = []
    for am in (1 + np.arange(128) / 128).astype(np.float32):
        for t in mids:
            u = int(np.array([np.float32(t * am)]).view(np.uint32)[0])
            for d in (-1, 0, 1):
                w = np.array([(((u >> 16) + d) & 0xffff) << 16], dtype=np.uint32).view(np.float32)[0]
                n = np.float32(w) / np.float32(am)
                if abs(float(n) - t) <= rel * abs(t):
                    pairs.append((am, w))
    return pairs


def test_quotients_next_to_thresholds():
    """Blocks whose elements divide to within 2^-12 of a decision midpoint (the
    closest bf16 quotient lies 1.2e-6 from one): the quantizer's fast grid
    path and its exact fallback must both agree with the oracle."""
    pairs = _near_threshold_pairs(2.0 ** -12)
    assert len(pairs) > 100
    by_am = {}
    for a, w in pairs:
        by_am.setdefault(float(a), []).append(float(w))
    blocks = []
    for a, ws in by_am.items():
        vals = ws + [-w for w in ws]
        for i in range(0, len(vals), 63):
            blk = np.zeros(64, np.float32)
            blk[0] = a                                  # the block absmax
            chunk = vals[i:i + 63]
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
    t = torch.from_numpy(np.concatenate(blocks)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.concatenate(blocks))   # every value is a bf16
    p, a = check_quant_exact(t.view(torch.int16).numpy().view(np.uint16))
    check_dequant_exact(p, a, t.numel())
