"""Build the CUDA library ``libw4a16.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into one
shared library next to this file.  Only nvcc and the host compiler are used.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libw4a16.so")
DEBUG_OUT_DIR = os.path.join(ROOT, "_build", "debug")
DEBUG_LIB = os.path.join(PKG, "libw4a16_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    inc = os.path.join(ROOT, "include")
    hs += [os.path.join(inc, f) for f in os.listdir(inc) if f.endswith(".h")]
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, extra: list[str], verbose: bool, out_dir: str = OUT_DIR,
             cacheable: bool = True) -> str:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()) \
            and cacheable:
        return obj
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr.strip():
        print(r.stderr, file=sys.stderr)
    return obj


def build_library(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
                  debug: bool = False) -> str:
    """Compile libw4a16.so (or, with debug=True, libw4a16_debug.so: the same
    sources with -DW4A16_DEBUG, whose kernels bounds-check their global
    accesses and report W4A16_ERR_BOUNDS instead of trapping)."""
    out_dir, lib = (DEBUG_OUT_DIR, DEBUG_LIB) if debug else (OUT_DIR, LIB)
    os.makedirs(out_dir, exist_ok=True)
    extra = list(extra or [])
    cacheable = not extra
    if debug:
        extra.append("-DW4A16_DEBUG")
    srcs = sources()
    newest = max([os.path.getmtime(s) for s in srcs] + [_headers_mtime()])
    if not force and cacheable and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose, out_dir, cacheable), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True,
                        extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None,
                        debug="--debug" in sys.argv))
