"""CPU oracle for NF4 weight-only quantization (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package imports nothing from it: the two share no code, header, table or
constant.

The arithmetic lives in ``nf4_oracle.c`` (plain C, compiled with gcc, no fast
math, no FMA contraction).  This module compiles it on first use, loads it
with ctypes and marshals numpy arrays.  Every function here is a thin call;
the definitions, and the readings of the diffuseR page "Gemma3 NF4 on GPU"
(pull request #39, Summary) they follow, are documented in the C file.

bf16 and fp16 data cross this interface as ``uint16`` bit patterns, fp32 as
``float32``; every array function takes ``dtype`` ("bf16" by default, "f16",
"f32").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nf4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``nf4_oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.oracle_codebook.restype = ctypes.POINTER(ctypes.c_float)
        lib.oracle_codebook.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_nearest_code.argtypes = [P, I64, P]
        lib.oracle_quantize.argtypes = [P, I64, I32, P, P]
        lib.oracle_dequantize.argtypes = [P, P, I64, I32, P]
        lib.oracle_linear.argtypes = [P, I64, I64, P, P, I64, I32, P]
        lib.oracle_gelu_tanh.argtypes = [P, I64, P]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_f16_array.argtypes = [P, I64, P]
        lib.oracle_f16_to_f32_array.argtypes = [P, I64, P]
        lib.oracle_f32_to_f16_array.restype = None
        lib.oracle_f16_to_f32_array.restype = None
        lib.oracle_quantize_dt.argtypes = [P, ctypes.c_int, I64, I32, P, P]
        lib.oracle_dequantize_dt.argtypes = [P, P, I64, I32, ctypes.c_int, P]
        lib.oracle_linear_dt.argtypes = [P, ctypes.c_int, I64, I64, P, P, I64, I32, P]
        lib.oracle_linear_geglu_dt.argtypes = [P, ctypes.c_int, I64, I64, P, P, I64, I32, P]
        lib.oracle_linear_geglu.argtypes = [P, I64, I64, P, P, I64, I32, P]
        for f in (lib.oracle_nearest_code, lib.oracle_quantize,
                  lib.oracle_dequantize, lib.oracle_linear, lib.oracle_set_num_threads,
                  lib.oracle_gelu_tanh, lib.oracle_linear_geglu, lib.oracle_quantize_dt,
                  lib.oracle_dequantize_dt, lib.oracle_linear_dt, lib.oracle_linear_geglu_dt):
            f.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


BLOCK = 64

# Element types: name -> (code in nf4_oracle.c, numpy storage dtype).  bf16
# and fp16 travel as uint16 bit patterns, fp32 as float32.
DTYPES = {"bf16": (0, np.uint16), "f16": (1, np.uint16), "f32": (2, np.float32)}


def _dt(dtype: str):
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    return DTYPES[dtype]


def codebook() -> np.ndarray:
    """The oracle's 16 fp32 codebook values, ascending."""
    lib = _load()
    return np.ctypeslib.as_array(lib.oracle_codebook(), shape=(16,)).copy()


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def f32_to_bf16_bits(v: float) -> int:
    return int(_load().oracle_f32_to_bf16(ctypes.c_float(v)))


def nearest_code(n: np.ndarray) -> np.ndarray:
    """Code chosen for each normalised fp32 value ``n``."""
    n = np.ascontiguousarray(n, dtype=np.float32).ravel()
    out = np.empty(n.size, dtype=np.uint8)
    _load().oracle_nearest_code(_ptr(n), n.size, _ptr(out))
    return out


def f32_to_f16_bits(v: float) -> int:
    return int(_load().oracle_f32_to_f16(ctypes.c_float(v)))


def f16_bits_to_f32(h: int) -> float:
    return float(_load().oracle_f16_to_f32(ctypes.c_uint16(h)))


def f32_to_f16_array(v: np.ndarray) -> np.ndarray:
    """fp32 values -> binary16 bit patterns (round to nearest even)."""
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, dtype=np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(v), v.size, _ptr(out))
    return out


def f16_to_f32_array(h: np.ndarray) -> np.ndarray:
    """binary16 bit patterns -> fp32 values."""
    h = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    out = np.empty(h.size, dtype=np.float32)
    _load().oracle_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


def quantize(w_bits: np.ndarray, block: int = BLOCK, dtype: str = "bf16"):
    """Weights (any shape, even size) -> (packed uint8 [numel/2], absmax fp32 [ceil(numel/block)]).
    bf16/f16 weights are uint16 bit patterns, f32 weights float32."""
    code, store = _dt(dtype)
    w = np.ascontiguousarray(w_bits, dtype=store).ravel()
    if w.size % 2:
        raise ValueError("numel must be even")
    packed = np.empty(w.size // 2, dtype=np.uint8)
    absmax = np.empty((w.size + block - 1) // block, dtype=np.float32)
    _load().oracle_quantize_dt(_ptr(w), code, w.size, block, _ptr(packed), _ptr(absmax))
    return packed, absmax


def dequantize(packed: np.ndarray, absmax: np.ndarray, numel: int, block: int = BLOCK,
               dtype: str = "bf16") -> np.ndarray:
    """(packed, absmax) -> [numel] values of `dtype` by nibble unpack (bit patterns for bf16/f16)."""
    code, store = _dt(dtype)
    p = np.ascontiguousarray(packed, dtype=np.uint8).ravel()
    a = np.ascontiguousarray(absmax, dtype=np.float32).ravel()
    if p.size * 2 < numel or a.size * block < numel:
        raise ValueError("packed/absmax too small for numel")
    out = np.empty(numel, dtype=store)
    _load().oracle_dequantize_dt(_ptr(p), _ptr(a), numel, block, code, _ptr(out))
    return out


def linear(x_bits: np.ndarray, packed: np.ndarray, absmax: np.ndarray, n_out: int,
           block: int = BLOCK, dtype: str = "bf16") -> np.ndarray:
    """Y = X . deq(W)^T in fp64.  X is [M, K] of `dtype`; W is NF4 over [n_out, K]."""
    code, store = _dt(dtype)
    x = np.ascontiguousarray(x_bits, dtype=store)
    if x.ndim != 2:
        raise ValueError("x must be 2-D")
    M, K = x.shape
    p = np.ascontiguousarray(packed, dtype=np.uint8).ravel()
    a = np.ascontiguousarray(absmax, dtype=np.float32).ravel()
    if p.size * 2 != n_out * K or a.size != (n_out * K + block - 1) // block:
        raise ValueError("packed/absmax do not match [n_out, K]")
    y = np.empty((M, n_out), dtype=np.float64)
    _load().oracle_linear_dt(_ptr(x), code, M, K, _ptr(p), _ptr(a), n_out, block, _ptr(y))
    return y


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU (tanh form) of each value, fp64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_gelu_tanh(_ptr(x), x.size, _ptr(y))
    return y


def linear_geglu(x_bits: np.ndarray, packed: np.ndarray, absmax: np.ndarray, n_ff: int,
                 block: int = BLOCK, dtype: str = "bf16") -> np.ndarray:
    """gelu_tanh(X . Wg^T) * (X . Wu^T) in fp64, [M, n_ff], where the NF4 weight
    covers [2 n_ff, K]: the gate rows, then the up rows.  X is of `dtype`."""
    code, store = _dt(dtype)
    x = np.ascontiguousarray(x_bits, dtype=store)
    if x.ndim != 2:
        raise ValueError("x must be 2-D")
    M, K = x.shape
    p = np.ascontiguousarray(packed, dtype=np.uint8).ravel()
    a = np.ascontiguousarray(absmax, dtype=np.float32).ravel()
    if p.size * 2 != 2 * n_ff * K or a.size != (2 * n_ff * K + block - 1) // block:
        raise ValueError("packed/absmax do not match [2 n_ff, K]")
    y = np.empty((M, n_ff), dtype=np.float64)
    _load().oracle_linear_geglu_dt(_ptr(x), code, M, K, _ptr(p), _ptr(a), n_ff, block, _ptr(y))
    return y
