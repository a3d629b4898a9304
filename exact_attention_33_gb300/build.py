"""Build libfa.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit is compiled to an object in parallel, then linked into
``exact_attention_33_gb300/libfa.so``.  No cmake; only nvcc and the host
compiler.  Run as ``python -m exact_attention_33_gb300.build`` or through
``__graft_entry__.build()``.

``--checked`` (``build(checked=True)``) builds the same sources with
FA_DEBUG_CHECKS into ``libfa_checked.so``: every plain global load and store of
the kernels is checked against its buffer's extent, and a failing access is
skipped and reported in the status word (FA_DEV_BAD_INDEX).  The binding loads
that library when the environment sets FA_CHECKED=1.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libfa_checked.so")
SOURCES = ["fa_api.cu", "prefill.cu", "decode.cu", "backward.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put /usr/local/cuda/bin on PATH)")


def common_flags():
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                   "-I" + os.path.join(PKG, "..", "include"), "--expt-relaxed-constexpr"]


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)
    return r.stdout


def build(verbose: bool = False, ptxas_verbose: bool = False, force: bool = False,
          checked: bool = False) -> str:
    """Compile every CUDA source and link libfa.so (libfa_checked.so with
    ``checked``); returns the library path."""
    nvcc = nvcc_path()
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    defines = ["-DFA_DEBUG_CHECKS"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(PKG, "..", "include", "fa.h"))
    if not force and os.path.exists(lib):
        lib_t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return lib

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc] + common_flags() + defines + ["-c", src, "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        out = _run(cmd, verbose)
        if ptxas_verbose and out:
            print(out, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, verbose)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv, force="-f" in sys.argv,
                checked="--checked" in sys.argv))
