"""Build libnf4.so in-tree with nvcc for sm_103a.

Each .cu file under csrc/ compiles to an object in parallel (one -gencode:
compute_103a -> sm_103a), then nvcc links them with the static CUDA runtime
into ``libnf4.so`` beside this file.  No cmake, no setuptools; the CUDA driver API
is reached through cudaGetDriverEntryPointByVersion, so the library has no
link-time dependency on libcuda and loads on a machine without a GPU.

``--checked`` builds ``_build/libnf4_checked.so`` instead (-DNF4_CHECKED):
every kernel access that is not a TMA tensor copy tests its index against its
buffer and reports NF4_ERR_BOUNDS through nf4_last_error() instead of
touching memory outside it.  A debugging build, never the default library.

    python -m nf4_weight_quantized_quantize_gb300.build [--force] [--checked]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnf4.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
CHECKED_LIB = os.path.join(BUILD, "libnf4_checked.so")
CHECKED_FLAGS = ["-DNF4_CHECKED"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, extra: list[str], build_dir: str) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          out: str | None = None) -> str:
    """Compile csrc/*.cu into libnf4.so (skipped when up to date).

    `extra` adds nvcc flags (e.g. -D test switches) and then `out` must name a
    different library path, so the product library is never built with them."""
    lib = out or LIB
    if extra and lib == LIB:
        raise ValueError("a build with extra flags needs its own output path")
    if not force and lib == LIB and up_to_date():
        return LIB
    if not force and lib != LIB and os.path.exists(lib) and \
            all(os.path.getmtime(d) <= os.path.getmtime(lib) for d in _deps()):
        return lib
    build_dir = BUILD if lib == LIB else os.path.join(BUILD, os.path.basename(lib) + ".d")
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra or [], build_dir), srcs))
    if verbose:
        for obj, log in results:
            print(f"== {os.path.basename(obj)}\n{log}")
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results],
           "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        for obj, log in results:
            f.write(f"== {os.path.basename(obj)}\n{log}\n")
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true", help="build the bounds-checked library")
    a = ap.parse_args()
    if a.checked:
        print(build(force=a.force, verbose=a.verbose, extra=CHECKED_FLAGS, out=CHECKED_LIB))
    else:
        print(build(force=a.force, verbose=a.verbose))
    sys.exit(0)
