"""Python binding of libnf4 (NF4 weight-only quantized linear for GB300).

Two layers, both argument marshalling only -- every step of the computation
runs in the library's CUDA kernels:

* ``nf4_quantize``, ``nf4_dequantize``, ``nf4_linear``, ``nf4_linear_geglu``,
  their ``_ex`` forms (an ``nf4_dtype`` argument: bf16, fp16, fp32),
  ``nf4_linear_noalloc``, ``nf4_linear_workspace_size``, ``nf4_last_error``,
  ``nf4_status_string``:
  the C entry points of ``include/nf4.h`` under the same names, taking plain
  integers (device addresses, sizes, a stream handle) and returning the
  status code.
* ``quantize``, ``dequantize``, ``linear``, ``linear_geglu``: the same calls on
  torch tensors, at the tensors' dtype (bf16, fp16; fp32 for quantize and
  dequantize).
  They check dtypes and devices, allocate the outputs with torch, pass the raw
  pointers and the current stream, and raise :class:`NF4Error` on a nonzero
  status.

The library must have been built (``build.build()``); importing this package
without it raises ImportError -- there is no fallback implementation.  The
environment variable ``NF4_LIBRARY`` selects another build of it (for
instance the bounds-checked one).
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

NF4_OK = 0
NF4_ERR_NULL = 1
NF4_ERR_SHAPE = 2
NF4_ERR_ALIGN = 3
NF4_ERR_BLOCKSIZE = 4
NF4_ERR_WORKSPACE = 5
NF4_ERR_DEVICE = 6
NF4_ERR_CUDA = 7
NF4_ERR_TIMEOUT = 8
NF4_ERR_DTYPE = 9
NF4_ERR_BOUNDS = 10
NF4_DTYPE_BF16 = 0
NF4_DTYPE_F16 = 1
NF4_DTYPE_F32 = 2
BLOCK = 64
# The environment variable NF4_LIBRARY names another build to load instead --
# the bounds-checked one (``build.CHECKED_LIB``), to run a whole program or
# test suite through it; unset, the in-tree libnf4.so.
LIB_PATH = os.environ.get("NF4_LIBRARY") or _build.LIB


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of libnf4 at `path` with every entry point's signature set
    (the bounds-checked build, for instance)."""
    lib = ctypes.CDLL(path)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    sigs = {
        "nf4_quantize": [P, I64, I32, P, P, P],
        "nf4_dequantize": [P, P, I64, I32, P, P],
        "nf4_linear": [P, I64, I64, P, P, I64, I32, P, P, SZ, P],
        "nf4_linear_workspace_size": [I64, I64, I64, ctypes.POINTER(SZ)],
        "nf4_last_error": [P],
        "nf4_status_string": [ctypes.c_int],
        "nf4_version": [],
        "nf4_launch_count": [],
        "nf4_linear_noalloc": [P, I64, I64, P, P, I64, I32, P, P],
        "nf4_linear_geglu": [P, I64, I64, P, P, I64, I32, P, P, SZ, P],
        "nf4_quantize_ex": [P, I32, I64, I32, P, P, P],
        "nf4_dequantize_ex": [P, P, I64, I32, I32, P, P],
        "nf4_linear_ex": [P, I32, I64, I64, P, P, I64, I32, P, P, SZ, P],
        "nf4_linear_geglu_ex": [P, I32, I64, I64, P, P, I64, I32, P, P, SZ, P],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.nf4_status_string.restype = ctypes.c_char_p
    lib.nf4_launch_count.restype = ctypes.c_uint64
    return lib


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libnf4 is not built ({LIB_PATH}); run "
            "`python -m nf4_weight_quantized_quantize_gb300.build` first")
    return load_library(LIB_PATH)


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libnf4 (loaded on first use; ImportError if it is not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


class NF4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {nf4_status_string(status)}")
        self.status = status


# ---------------------------------------------------------------- C entry points


def nf4_quantize(w: int, numel: int, block: int, packed: int, absmax: int, stream: int = 0) -> int:
    return lib().nf4_quantize(w, numel, block, packed, absmax, stream)


def nf4_dequantize(packed: int, absmax: int, numel: int, block: int, out: int, stream: int = 0) -> int:
    return lib().nf4_dequantize(packed, absmax, numel, block, out, stream)


def nf4_linear(x: int, M: int, K: int, packed: int, absmax: int, N: int, block: int, y: int,
               workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return lib().nf4_linear(x, M, K, packed, absmax, N, block, y, workspace, workspace_bytes, stream)


def nf4_linear_geglu(x: int, M: int, K: int, packed: int, absmax: int, F: int, block: int, y: int,
                     workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return lib().nf4_linear_geglu(x, M, K, packed, absmax, F, block, y, workspace, workspace_bytes, stream)


def nf4_quantize_ex(w: int, dtype: int, numel: int, block: int, packed: int, absmax: int, stream: int = 0) -> int:
    return lib().nf4_quantize_ex(w, dtype, numel, block, packed, absmax, stream)


def nf4_dequantize_ex(packed: int, absmax: int, numel: int, block: int, dtype: int, out: int,
                      stream: int = 0) -> int:
    return lib().nf4_dequantize_ex(packed, absmax, numel, block, dtype, out, stream)


def nf4_linear_ex(x: int, dtype: int, M: int, K: int, packed: int, absmax: int, N: int, block: int, y: int,
                  workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return lib().nf4_linear_ex(x, dtype, M, K, packed, absmax, N, block, y, workspace, workspace_bytes, stream)


def nf4_linear_geglu_ex(x: int, dtype: int, M: int, K: int, packed: int, absmax: int, F: int, block: int,
                        y: int, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    return lib().nf4_linear_geglu_ex(x, dtype, M, K, packed, absmax, F, block, y, workspace, workspace_bytes,
                                     stream)


def nf4_linear_noalloc(x: int, M: int, K: int, packed: int, absmax: int, N: int, block: int, y: int,
                       stream: int = 0) -> int:
    return lib().nf4_linear_noalloc(x, M, K, packed, absmax, N, block, y, stream)


NF4_NOALLOC_SCRATCH_BYTES = 16 << 20


def nf4_linear_workspace_size(M: int, N: int, K: int) -> tuple[int, int]:
    """Returns (status, bytes)."""
    out = ctypes.c_size_t(0)
    st = lib().nf4_linear_workspace_size(M, N, K, ctypes.byref(out))
    return st, out.value


def nf4_last_error(stream: int = 0) -> int:
    return lib().nf4_last_error(stream)


def nf4_status_string(status: int) -> str:
    return lib().nf4_status_string(status).decode()


def nf4_version() -> int:
    return lib().nf4_version()


def nf4_launch_count() -> int:
    return lib().nf4_launch_count()


# ---------------------------------------------------------------- torch tensors


def _torch():
    import torch
    return torch


def _stream(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, what: str) -> None:
    if status != NF4_OK:
        raise NF4Error(status, what)


def _need(t, dtypes, name):
    torch = _torch()
    dtypes = dtypes if isinstance(dtypes, tuple) else (dtypes,)
    if not isinstance(t, torch.Tensor) or t.dtype not in dtypes or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {' or '.join(map(str, dtypes))}")


def _compute_dtypes():
    torch = _torch()
    return {torch.bfloat16: NF4_DTYPE_BF16, torch.float16: NF4_DTYPE_F16, torch.float32: NF4_DTYPE_F32}


def quantize(w, out=None):
    """bf16, fp16 or fp32 CUDA tensor (any shape, even numel) ->
    (packed uint8 [numel/2], absmax fp32 [ceil(numel/64)])."""
    torch = _torch()
    codes = _compute_dtypes()
    _need(w, tuple(codes), "w")
    numel = w.numel()
    if out is None:
        packed = torch.empty(numel // 2, dtype=torch.uint8, device=w.device)
        absmax = torch.empty((numel + BLOCK - 1) // BLOCK, dtype=torch.float32, device=w.device)
    else:
        packed, absmax = out
    _check(nf4_quantize_ex(w.data_ptr(), codes[w.dtype], numel, BLOCK, packed.data_ptr(), absmax.data_ptr(),
                           _stream(w.device)), "nf4_quantize")
    return packed, absmax


def dequantize(packed, absmax, numel: int | None = None, out=None, dtype=None):
    """(packed uint8, absmax fp32) -> [numel] of `dtype` (bf16 by default, fp16, fp32; the
    dtype of `out` when given); numel defaults to 2 * packed.numel()."""
    torch = _torch()
    codes = _compute_dtypes()
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    numel = 2 * packed.numel() if numel is None else int(numel)
    if 2 * packed.numel() < numel or absmax.numel() * BLOCK < numel:
        raise ValueError("packed/absmax too small for numel")
    if out is None:
        out = torch.empty(numel, dtype=dtype or torch.bfloat16, device=packed.device)
    _need(out, tuple(codes), "out")
    _check(nf4_dequantize_ex(packed.data_ptr(), absmax.data_ptr(), numel, BLOCK, codes[out.dtype], out.data_ptr(),
                             _stream(packed.device)), "nf4_dequantize")
    return out


def linear(x, packed, absmax, n_out: int, out=None, workspace=None):
    """Y [M, n_out] = X [M, K] . deq(W)^T with W [n_out, K] in NF4; X and Y
    bf16, fp16 or fp32 (fp32 runs on the tf32 tensor cores: X's and the
    weight's fractions cut to 10 bits, fp32 output).  A given `workspace`
    (uint8, at least nf4_linear_workspace_size bytes) must start zeroed before
    its first use; each call leaves its counter header zero again, so it can
    be reused on one stream.  Without one, a zeroed workspace is allocated."""
    torch = _torch()
    codes = _compute_dtypes()
    _need(x, tuple(codes), "x")
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if packed.numel() * 2 != n_out * K or absmax.numel() * BLOCK != n_out * K:
        raise ValueError("packed/absmax do not match [n_out, K]")
    if out is None:
        out = torch.empty(M, n_out, dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out")
    st, ws_bytes = nf4_linear_workspace_size(M, n_out, K)
    _check(st, "nf4_linear_workspace_size")
    if ws_bytes and workspace is None:
        workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(nf4_linear_ex(x.data_ptr(), codes[x.dtype], M, K, packed.data_ptr(), absmax.data_ptr(), n_out, BLOCK,
                         out.data_ptr(), ws_ptr, ws_len, _stream(x.device)), "nf4_linear")
    return out


def linear_geglu(x, packed, absmax, n_ff: int, out=None, workspace=None):
    """Y [M, n_ff] = gelu_tanh(X . Wg^T) * (X . Wu^T), where (packed, absmax)
    is ONE NF4 weight [2 n_ff, K]: the gate rows, then the up rows.  X and Y
    bf16, fp16 or fp32 (tf32 tensor cores).  `workspace` as for linear()."""
    torch = _torch()
    codes = _compute_dtypes()
    _need(x, tuple(codes), "x")
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if packed.numel() * 2 != 2 * n_ff * K or absmax.numel() * BLOCK != 2 * n_ff * K:
        raise ValueError("packed/absmax do not match [2 n_ff, K]")
    if out is None:
        out = torch.empty(M, n_ff, dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out")
    st, ws_bytes = nf4_linear_workspace_size(M, 2 * n_ff, K)
    _check(st, "nf4_linear_workspace_size")
    if ws_bytes and workspace is None:
        workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(nf4_linear_geglu_ex(x.data_ptr(), codes[x.dtype], M, K, packed.data_ptr(), absmax.data_ptr(), n_ff,
                               BLOCK, out.data_ptr(), ws_ptr, ws_len, _stream(x.device)), "nf4_linear_geglu")
    return out
