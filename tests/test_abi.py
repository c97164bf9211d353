"""The C ABI without a GPU: the library loads, exports every function that
include/nf4.h declares, and rejects bad arguments on the host before touching
a device (the "hard error, never run on garbage" convention of the diffuseR
page "Gemma3 NF4 on GPU", #39, Summary: the loader hard-errors on unfilled
parameters)."""
import ctypes
import os
import re

import pytest

import nf4_weight_quantized_quantize_gb300 as nf4
from nf4_weight_quantized_quantize_gb300 import build as nf4_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    nf4_build.build()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^NF4_API\s+[\w\s\*]+?\b(nf4_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert {"nf4_quantize", "nf4_dequantize", "nf4_linear", "nf4_linear_workspace_size",
            "nf4_last_error", "nf4_status_string", "nf4_version", "nf4_launch_count"} <= set(names)
    lib = ctypes.CDLL(nf4.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_library_links_no_torch_and_no_libcuda():
    import subprocess
    out = subprocess.run(["ldd", nf4.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "libcuda.so" not in out and "libcudart" not in out


def test_status_strings_and_version():
    for code, name in [(0, "NF4_OK"), (1, "NF4_ERR_NULL"), (2, "NF4_ERR_SHAPE"), (3, "NF4_ERR_ALIGN"),
                       (4, "NF4_ERR_BLOCKSIZE"), (5, "NF4_ERR_WORKSPACE"), (6, "NF4_ERR_DEVICE"),
                       (7, "NF4_ERR_CUDA"), (8, "NF4_ERR_TIMEOUT"), (9, "NF4_ERR_DTYPE"),
                       (10, "NF4_ERR_BOUNDS")]:
        assert nf4.nf4_status_string(code) == name
    assert nf4.nf4_status_string(99) == "NF4_ERR_UNKNOWN"
    assert nf4.nf4_version() >= 100
    assert nf4.nf4_launch_count() >= 0


FAKE = 1 << 20   # a 16-byte aligned non-null address; never dereferenced by these calls


def test_quantize_argument_errors():
    assert nf4.nf4_quantize(FAKE, 128, 32, FAKE, FAKE) == nf4.NF4_ERR_BLOCKSIZE
    assert nf4.nf4_quantize(FAKE, 127, 64, FAKE, FAKE) == nf4.NF4_ERR_SHAPE
    assert nf4.nf4_quantize(FAKE, -2, 64, FAKE, FAKE) == nf4.NF4_ERR_SHAPE
    assert nf4.nf4_quantize(0, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_NULL
    assert nf4.nf4_quantize(FAKE, 128, 64, 0, FAKE) == nf4.NF4_ERR_NULL
    assert nf4.nf4_quantize(FAKE, 128, 64, FAKE, 0) == nf4.NF4_ERR_NULL
    assert nf4.nf4_quantize(FAKE + 1, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_quantize(FAKE, 128, 64, FAKE, FAKE + 2) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_quantize(0, 0, 64, 0, 0) == nf4.NF4_OK       # empty: nothing to do


def test_dequantize_argument_errors():
    assert nf4.nf4_dequantize(FAKE, FAKE, 128, 128, FAKE) == nf4.NF4_ERR_BLOCKSIZE
    assert nf4.nf4_dequantize(FAKE, FAKE, 3, 64, FAKE) == nf4.NF4_ERR_SHAPE
    assert nf4.nf4_dequantize(0, FAKE, 128, 64, FAKE) == nf4.NF4_ERR_NULL
    assert nf4.nf4_dequantize(FAKE, 0, 128, 64, FAKE) == nf4.NF4_ERR_NULL
    assert nf4.nf4_dequantize(FAKE, FAKE, 128, 64, 0) == nf4.NF4_ERR_NULL
    assert nf4.nf4_dequantize(FAKE, FAKE, 128, 64, FAKE + 1) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_dequantize(0, 0, 0, 64, 0) == nf4.NF4_OK


def test_linear_argument_errors():
    ok = dict(x=FAKE, M=256, K=128, packed=FAKE, absmax=FAKE, N=64, block=64, y=FAKE,
              workspace=0, workspace_bytes=0)

    def call(**kw):
        a = dict(ok, **kw)
        return nf4.nf4_linear(a["x"], a["M"], a["K"], a["packed"], a["absmax"], a["N"], a["block"],
                              a["y"], a["workspace"], a["workspace_bytes"])

    assert call(block=128) == nf4.NF4_ERR_BLOCKSIZE
    assert call(K=96) == nf4.NF4_ERR_SHAPE
    assert call(K=0) == nf4.NF4_ERR_SHAPE
    assert call(M=-1) == nf4.NF4_ERR_SHAPE
    assert call(N=-5) == nf4.NF4_ERR_SHAPE
    assert call(M=1 << 31) == nf4.NF4_ERR_SHAPE
    assert call(x=0) == nf4.NF4_ERR_NULL
    assert call(packed=0) == nf4.NF4_ERR_NULL
    assert call(absmax=0) == nf4.NF4_ERR_NULL
    assert call(y=0) == nf4.NF4_ERR_NULL
    assert call(x=FAKE + 2) == nf4.NF4_ERR_ALIGN
    assert call(packed=FAKE + 8) == nf4.NF4_ERR_ALIGN
    assert call(y=FAKE + 4) == nf4.NF4_ERR_ALIGN
    assert call(absmax=FAKE + 2) == nf4.NF4_ERR_ALIGN
    assert call(M=0) == nf4.NF4_OK and call(N=0) == nf4.NF4_OK
    st, need = nf4.nf4_linear_workspace_size(16, 3840, 15360)
    assert st == nf4.NF4_OK
    if need:
        assert call(M=16, N=3840, K=15360) == nf4.NF4_ERR_WORKSPACE
        assert call(M=16, N=3840, K=15360, workspace=FAKE, workspace_bytes=need - 1) == nf4.NF4_ERR_WORKSPACE
        assert call(M=16, N=3840, K=15360, workspace=FAKE + 4, workspace_bytes=need) == nf4.NF4_ERR_ALIGN


def test_linear_geglu_argument_errors():
    ok = dict(x=FAKE, M=256, K=128, packed=FAKE, absmax=FAKE, F=64, block=64, y=FAKE,
              workspace=0, workspace_bytes=0)

    def call(**kw):
        a = dict(ok, **kw)
        return nf4.nf4_linear_geglu(a["x"], a["M"], a["K"], a["packed"], a["absmax"], a["F"], a["block"],
                                    a["y"], a["workspace"], a["workspace_bytes"])

    assert call(block=32) == nf4.NF4_ERR_BLOCKSIZE
    assert call(K=100) == nf4.NF4_ERR_SHAPE
    assert call(F=-1) == nf4.NF4_ERR_SHAPE
    assert call(F=1 << 30) == nf4.NF4_ERR_SHAPE          # 2F weight rows must stay below 2^31
    assert call(x=0) == nf4.NF4_ERR_NULL
    assert call(y=0) == nf4.NF4_ERR_NULL
    assert call(y=FAKE + 2) == nf4.NF4_ERR_ALIGN
    assert call(M=0) == nf4.NF4_OK and call(F=0) == nf4.NF4_OK
    # the skinny path's workspace is that of the [2F, K] weight
    _, need = nf4.nf4_linear_workspace_size(16, 2 * 15360, 3840)
    assert need > 0
    assert call(M=16, F=15360, K=3840) == nf4.NF4_ERR_WORKSPACE
    assert call(M=16, F=15360, K=3840, workspace=FAKE, workspace_bytes=need - 1) == nf4.NF4_ERR_WORKSPACE


def test_dtype_argument_errors():
    """The _ex entry points: a dtype outside nf4_dtype is refused on the host
    and element alignment follows the dtype.  (No call here passes
    validation with its placeholder pointers.)"""
    BF16, F16, F32 = nf4.NF4_DTYPE_BF16, nf4.NF4_DTYPE_F16, nf4.NF4_DTYPE_F32
    for bad in (-1, 3, 99):
        assert nf4.nf4_quantize_ex(FAKE, bad, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_DTYPE
        assert nf4.nf4_dequantize_ex(FAKE, FAKE, 128, 64, bad, FAKE) == nf4.NF4_ERR_DTYPE
        assert nf4.nf4_linear_ex(FAKE, bad, 256, 128, FAKE, FAKE, 64, 64, FAKE, 0, 0) == nf4.NF4_ERR_DTYPE
        assert nf4.nf4_linear_geglu_ex(FAKE, bad, 256, 128, FAKE, FAKE, 64, 64, FAKE, 0, 0) == nf4.NF4_ERR_DTYPE
    assert nf4.nf4_linear_ex(FAKE + 4, F32, 256, 128, FAKE, FAKE, 64, 64, FAKE, 0, 0) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_linear_geglu_ex(FAKE, F32, 256, 128, FAKE, FAKE, 64, 64, FAKE + 8, 0, 0) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_quantize_ex(FAKE + 2, F32, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_quantize_ex(FAKE + 1, F16, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_dequantize_ex(FAKE, FAKE, 128, 64, F32, FAKE + 2) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_linear_ex(FAKE + 2, F16, 256, 128, FAKE, FAKE, 64, 64, FAKE, 0, 0) == nf4.NF4_ERR_ALIGN
    assert nf4.nf4_quantize_ex(FAKE, BF16, 127, 64, FAKE, FAKE) == nf4.NF4_ERR_SHAPE
    assert nf4.nf4_linear_ex(0, F16, 0, 128, 0, 0, 64, 64, 0, 0, 0) == nf4.NF4_OK


def test_workspace_size_rules():
    assert nf4.nf4_linear_workspace_size(2048, 4096, 3840) == (nf4.NF4_OK, 0)
    assert nf4.nf4_linear_workspace_size(16, 4096, 100)[0] == nf4.NF4_ERR_SHAPE
    assert nf4.nf4_linear_workspace_size(-1, 4096, 128)[0] == nf4.NF4_ERR_SHAPE
    st, b = nf4.nf4_linear_workspace_size(0, 4096, 128)
    assert st == nf4.NF4_OK and b == 0
    assert nf4.lib().nf4_linear_workspace_size(16, 16, 64, None) == nf4.NF4_ERR_NULL


def test_no_device_is_reported_not_crashed():
    """With arguments that pass validation and no usable GPU the call returns
    NF4_ERR_DEVICE (with a GPU present this test is skipped)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert nf4.nf4_quantize(FAKE, 128, 64, FAKE, FAKE) == nf4.NF4_ERR_DEVICE
    assert nf4.nf4_last_error(0) == nf4.NF4_ERR_DEVICE


def test_tensor_wrappers_refuse_host_tensors_and_wrong_dtypes():
    """The torch-level wrappers check device, dtype and layout before calling
    the library (no device needed to see the refusal)."""
    import torch
    with pytest.raises(TypeError):
        nf4.quantize(torch.zeros(128, dtype=torch.bfloat16))          # host tensor
    with pytest.raises(TypeError):
        nf4.quantize(torch.zeros(128, dtype=torch.float64))           # not a compute dtype
    with pytest.raises(TypeError):
        nf4.dequantize(torch.zeros(64, dtype=torch.uint8), torch.zeros(2, dtype=torch.float32))
    with pytest.raises(TypeError):
        nf4.linear(torch.zeros(2, 64, dtype=torch.int32), torch.zeros(32, dtype=torch.uint8),
                   torch.zeros(1, dtype=torch.float32), 1)


def test_kernel_hash_ignores_comments_and_layout():
    """The ncu traffic line is keyed to the GEMM code without comments and
    whitespace: editing a comment keeps it, editing code does not."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    a = "int f(int x) {  // the input\n    return x + 1; /* one */\n}\n"
    b = "/* header */\nint f(int x) {\n  return x + 1;\n}"
    assert bench.code_tokens(a) == bench.code_tokens(b) == "int f(int x) { return x + 1; }"
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("x + 1", "x + 2"))
    assert len(bench.kernel_source_hash()) == 16


def test_checked_build_loads_and_exports_every_symbol():
    """The bounds-checked build (-DNF4_CHECKED) compiles for sm_103a, loads
    without a GPU and exports the same entry points."""
    lib = nf4.load_library(nf4_build.build(extra=nf4_build.CHECKED_FLAGS, out=nf4_build.CHECKED_LIB))
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert lib.nf4_status_string(nf4.NF4_ERR_BOUNDS) == b"NF4_ERR_BOUNDS"
    assert lib.nf4_quantize(FAKE, 127, 64, FAKE, FAKE, None) == nf4.NF4_ERR_SHAPE   # same host checks
