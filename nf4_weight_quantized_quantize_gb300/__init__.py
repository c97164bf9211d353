"""Python binding of libnf4 (NF4 weight-only quantized linear for GB300).

Two layers, both argument marshalling only -- every step of the computation
runs in the library's CUDA kernels:

* ``nf4_quantize``, ``nf4_dequantize``, ``nf4_linear``, ``nf4_linear_geglu``,
  ``nf4_linear_noalloc``, ``nf4_linear_workspace_size``, ``nf4_last_error``,
  ``nf4_status_string``:
  the C entry points of ``include/nf4.h`` under the same names, taking plain
  integers (device addresses, sizes, a stream handle) and returning the
  status code.
* ``quantize``, ``dequantize``, ``linear``, ``linear_geglu``: the same calls on
  torch tensors.
  They check dtypes and devices, allocate the outputs with torch, pass the raw
  pointers and the current stream, and raise :class:`NF4Error` on a nonzero
  status.

The library must have been built (``build.build()``); importing this package
without it raises ImportError -- there is no fallback implementation.
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
BLOCK = 64
LIB_PATH = _build.LIB


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libnf4.so is not built ({LIB_PATH}); run "
            "`python -m nf4_weight_quantized_quantize_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
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
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.nf4_status_string.restype = ctypes.c_char_p
    lib.nf4_launch_count.restype = ctypes.c_uint64
    return lib


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


def _need(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")


def quantize(w, out=None):
    """bf16 CUDA tensor (any shape, even numel) -> (packed uint8 [numel/2], absmax fp32 [ceil(numel/64)])."""
    torch = _torch()
    _need(w, torch.bfloat16, "w")
    numel = w.numel()
    if out is None:
        packed = torch.empty(numel // 2, dtype=torch.uint8, device=w.device)
        absmax = torch.empty((numel + BLOCK - 1) // BLOCK, dtype=torch.float32, device=w.device)
    else:
        packed, absmax = out
    _check(nf4_quantize(w.data_ptr(), numel, BLOCK, packed.data_ptr(), absmax.data_ptr(),
                        _stream(w.device)), "nf4_quantize")
    return packed, absmax


def dequantize(packed, absmax, numel: int | None = None, out=None):
    """(packed uint8, absmax fp32) -> bf16 [numel] (numel defaults to 2 * packed.numel())."""
    torch = _torch()
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    numel = 2 * packed.numel() if numel is None else int(numel)
    if 2 * packed.numel() < numel or absmax.numel() * BLOCK < numel:
        raise ValueError("packed/absmax too small for numel")
    if out is None:
        out = torch.empty(numel, dtype=torch.bfloat16, device=packed.device)
    _check(nf4_dequantize(packed.data_ptr(), absmax.data_ptr(), numel, BLOCK, out.data_ptr(),
                          _stream(packed.device)), "nf4_dequantize")
    return out


def linear(x, packed, absmax, n_out: int, out=None, workspace=None):
    """Y [M, n_out] bf16 = X [M, K] bf16 . deq(W)^T with W [n_out, K] in NF4."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if packed.numel() * 2 != n_out * K or absmax.numel() * BLOCK != n_out * K:
        raise ValueError("packed/absmax do not match [n_out, K]")
    if out is None:
        out = torch.empty(M, n_out, dtype=torch.bfloat16, device=x.device)
    st, ws_bytes = nf4_linear_workspace_size(M, n_out, K)
    _check(st, "nf4_linear_workspace_size")
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(nf4_linear(x.data_ptr(), M, K, packed.data_ptr(), absmax.data_ptr(), n_out, BLOCK,
                      out.data_ptr(), ws_ptr, ws_len, _stream(x.device)), "nf4_linear")
    return out


def linear_geglu(x, packed, absmax, n_ff: int, out=None, workspace=None):
    """Y [M, n_ff] bf16 = gelu_tanh(X . Wg^T) * (X . Wu^T), where (packed, absmax)
    is ONE NF4 weight [2 n_ff, K]: the gate rows, then the up rows."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    _need(packed, torch.uint8, "packed")
    _need(absmax, torch.float32, "absmax")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    M, K = x.shape
    if packed.numel() * 2 != 2 * n_ff * K or absmax.numel() * BLOCK != 2 * n_ff * K:
        raise ValueError("packed/absmax do not match [2 n_ff, K]")
    if out is None:
        out = torch.empty(M, n_ff, dtype=torch.bfloat16, device=x.device)
    st, ws_bytes = nf4_linear_workspace_size(M, 2 * n_ff, K)
    _check(st, "nf4_linear_workspace_size")
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(nf4_linear_geglu(x.data_ptr(), M, K, packed.data_ptr(), absmax.data_ptr(), n_ff, BLOCK,
                            out.data_ptr(), ws_ptr, ws_len, _stream(x.device)), "nf4_linear_geglu")
    return out
