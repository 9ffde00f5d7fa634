"""Build the USP CUDA library (libusp.so) in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in parallel with nvcc and the
objects are linked into ``_build/libusp.so`` with the CUDA runtime linked
statically, so the library loads on hosts without a GPU driver (its symbols
can be inspected there) and on the GPU host without extra runtime libraries.

``build(debug=True)`` makes ``_build_debug/libusp.so`` with USP_DEBUG_BOUNDS:
every global index a kernel computes is checked against the extent usp_dims
implies for its buffer, and an out-of-range one is reported through the
device status word instead of being accessed.  The binding loads it when
USP_DEBUG_BOUNDS=1 is set in the environment.

Usage:  python -m ulysses_sequence_attention_usp_gb300.build [-v] [-f] [-d]
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libusp.so")
OUT_DEBUG = os.path.join(PKG, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the USP CUDA library cannot be built")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _digest(paths, flags) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as f:
            h.update(p.encode() + f.read())
    h.update(" ".join(ARCH + flags).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    out = OUT_DEBUG if debug else OUT
    lib = os.path.join(out, "libusp.so")
    flags = CFLAGS + (["-DUSP_DEBUG_BOUNDS"] if debug else [])
    srcs = _sources()
    deps = srcs + sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    deps.append(os.path.join(INCLUDE, "usp.h"))
    stamp = os.path.join(out, "stamp")
    dig = _digest(deps, flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == dig:
                return lib
    os.makedirs(out, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(out, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(dig)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="-d" in sys.argv))
