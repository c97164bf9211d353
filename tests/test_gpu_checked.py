"""The bounds-checked build of the library (-DNF4_CHECKED) on the GPU.

In that build every kernel access to global memory that is not a TMA tensor
copy first tests its index against the extent of its buffer; an index outside
skips the access and records NF4_ERR_BOUNDS for nf4_last_error().  Two
properties, over every kernel the library launches:

* on valid arguments the checked build reports nothing and writes the same
  bits as the normal build (the tests themselves are not arithmetic);
* with the test switch NF4_TEST_SHRINK_EXTENT, which checks against one
  element less than each buffer holds, every kernel reports NF4_ERR_BOUNDS
  once (the word is read-and-clear) -- the check fires and the call returns
  while no access leaves its buffer -- and the context stays usable.
"""
import os

import numpy as np
import pytest
import torch

import nf4_weight_quantized_quantize_gb300 as nf4
from nf4_weight_quantized_quantize_gb300 import build as nf4_build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BF16, F16, F32 = nf4.NF4_DTYPE_BF16, nf4.NF4_DTYPE_F16, nf4.NF4_DTYPE_F32
TORCH_DT = {BF16: torch.bfloat16, F16: torch.float16, F32: torch.float32}


@pytest.fixture(scope="module")
def checked_lib():
    return nf4.load_library(nf4_build.build(extra=nf4_build.CHECKED_FLAGS, out=nf4_build.CHECKED_LIB))


@pytest.fixture(scope="module")
def shrunk_lib():
    path = nf4_build.build(extra=nf4_build.CHECKED_FLAGS + ["-DNF4_TEST_SHRINK_EXTENT"],
                           out=os.path.join(nf4_build.BUILD, "libnf4_shrunk.so"))
    return nf4.load_library(path)


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _weight(n, k, dt, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, k, generator=g) * 0.02).to(TORCH_DT[dt]).to(DEV)


def _act(m, k, dt, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(m, k, generator=g).to(TORCH_DT[dt]).to(DEV)


def _quantized(n, k, dt, seed):
    w = _weight(n, k, dt, seed)
    p = torch.empty(n * k // 2, dtype=torch.uint8, device=DEV)
    a = torch.empty(n * k // 64, dtype=torch.float32, device=DEV)
    assert nf4.lib().nf4_quantize_ex(w.data_ptr(), dt, n * k, 64, p.data_ptr(), a.data_ptr(), _stream()) == 0
    return p, a


# Each case: (inputs built once) -> fn(lib) that runs one call through `lib`
# and returns its outputs.  The ids name the kernels the call launches.

def _quantize_case(numel, dt, offset):
    def make():
        w_full = _weight(1, numel + offset, dt, numel)[0]
        w = w_full[offset:]                                   # offset 1: not 16-byte aligned -> scalar kernel

        def run(lib):
            p = torch.zeros(numel // 2, dtype=torch.uint8, device=DEV)
            a = torch.zeros((numel + 63) // 64, dtype=torch.float32, device=DEV)
            assert lib.nf4_quantize_ex(w.data_ptr(), dt, numel, 64, p.data_ptr(), a.data_ptr(), _stream()) == 0
            return [p, a]
        return run
    return make


def _dequantize_case(numel, dt, offset):
    def make():
        g = torch.Generator().manual_seed(numel)
        p = torch.randint(0, 256, (numel // 2,), generator=g, dtype=torch.uint8).to(DEV)
        a = torch.rand((numel + 63) // 64, generator=g).to(DEV)

        def run(lib):
            out_full = torch.zeros(numel + offset, dtype=TORCH_DT[dt], device=DEV)
            out = out_full[offset:]                           # offset 1: not 16-byte aligned -> scalar kernel
            assert lib.nf4_dequantize_ex(p.data_ptr(), a.data_ptr(), numel, 64, dt, out.data_ptr(), _stream()) == 0
            return [out]
        return run
    return make


def _linear_case(m, n, k, dt, geglu=False):
    def make():
        p, a = _quantized(n, k, dt, m * 7 + n)
        x = _act(m, k, dt, m + k)
        n_out = n // 2 if geglu else n
        _, need = nf4.nf4_linear_workspace_size(m, n, k)

        def run(lib):
            y = torch.zeros(m, n_out, dtype=TORCH_DT[dt], device=DEV)
            ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=DEV)
            fn = lib.nf4_linear_geglu_ex if geglu else lib.nf4_linear_ex
            assert fn(x.data_ptr(), dt, m, k, p.data_ptr(), a.data_ptr(), n_out, 64, y.data_ptr(), ws.data_ptr(),
                      need, _stream()) == 0
            return [y]
        return run
    return make


def _noalloc_case(m, n, k):
    def make():
        p, a = _quantized(n, k, BF16, 3)
        x = _act(m, k, BF16, 4)

        def run(lib):
            y = torch.zeros(m, n, dtype=torch.bfloat16, device=DEV)
            assert lib.nf4_linear_noalloc(x.data_ptr(), m, k, p.data_ptr(), a.data_ptr(), n, 64, y.data_ptr(),
                                          _stream()) == 0
            return [y]
        return run
    return make


CASES = {
    "quantize_vec_bf16": _quantize_case(64 * 1000, BF16, 0),
    "quantize_vec_f16": _quantize_case(64 * 777, F16, 0),
    "quantize_vec_f32": _quantize_case(64 * 513, F32, 0),
    "quantize_scalar_unaligned": _quantize_case(64 * 40 + 32, BF16, 1),
    "quantize_vec_and_scalar_tail": _quantize_case(64 * 300 + 18, BF16, 0),
    "dequant_vec_bf16": _dequantize_case(1024 * 300, BF16, 0),
    "dequant_vec_f32": _dequantize_case(256 * 301, F32, 0),
    "dequant_vec_and_scalar_tail": _dequantize_case(1024 * 20 + 66, F16, 0),
    "dequant_scalar_unaligned": _dequantize_case(64 * 50, BF16, 1),
    "warp_mma_split": _linear_case(16, 2048, 4096, BF16),
    "warp_mma_m5_f16": _linear_case(5, 1000, 1024, F16),
    "warp_mma_scales_by_copy": _linear_case(16, 1536, 1344, BF16),      # K / 64 = 21: no scale tensor map
    "warp_mma_gate_up": _linear_case(8, 2048, 1024, BF16, geglu=True),
    "tile_split_and_reduce": _linear_case(64, 512, 1024, BF16),
    "tile_split_f32": _linear_case(40, 384, 512, F32),
    "tile_split_gate_up_reduce": _linear_case(64, 512, 512, BF16, geglu=True),
    "tile_direct": _linear_case(256, 512, 1024, BF16),
    "tile_direct_f32": _linear_case(256, 384, 512, F32),
    "tile_gate_up": _linear_case(256, 512, 512, BF16, geglu=True),
    "cta_pair": _linear_case(1500, 10000, 192, BF16),
    "cta_pair_f16_ragged": _linear_case(700, 30720, 128, F16),
    "cta_pair_gate_up": _linear_case(1500, 10000, 192, BF16, geglu=True),
    "cta_pair_f32": _linear_case(1500, 10000, 192, F32),
    "noalloc_m16": _noalloc_case(16, 3840, 2048),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_checked_build_matches_and_reports_nothing(checked_lib, case):
    run = CASES[case]()
    want = run(nf4.lib())
    got = run(checked_lib)
    assert checked_lib.nf4_last_error(_stream()) == nf4.NF4_OK
    assert nf4.lib().nf4_last_error(_stream()) == nf4.NF4_OK
    for w, g in zip(want, got):
        assert torch.equal(w.view(torch.uint8) if w.dtype != torch.uint8 else w,
                           g.view(torch.uint8) if g.dtype != torch.uint8 else g), case


@pytest.mark.parametrize("case", sorted(CASES))
def test_shrunk_extent_reports_bounds(shrunk_lib, case):
    run = CASES[case]()
    run(shrunk_lib)
    assert shrunk_lib.nf4_last_error(_stream()) == nf4.NF4_ERR_BOUNDS
    assert shrunk_lib.nf4_last_error(_stream()) == nf4.NF4_OK       # read-and-clear


def test_context_usable_after_bounds_reports(shrunk_lib):
    run = CASES["tile_direct"]()
    run(shrunk_lib)
    assert shrunk_lib.nf4_last_error(_stream()) == nf4.NF4_ERR_BOUNDS
    a = run(nf4.lib())
    b = run(nf4.lib())
    assert nf4.lib().nf4_last_error(_stream()) == nf4.NF4_OK
    assert torch.equal(a[0].view(torch.uint8), b[0].view(torch.uint8))
    assert torch.isfinite(a[0].float()).all()
