"""In-tree build of libmxq.so for sm_103a (GB300).

Each translation unit under ``csrc/`` is compiled in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``) and linked into
``mx_block_scaled_mxq_gb300/libmxq.so`` next to this file.  The CUDA runtime is
linked statically and the driver entry point for tensor maps is fetched at run
time, so the library loads on a machine without a GPU driver (symbol checks)
and needs no libcuda at link time.

``build(debug=True)`` makes ``libmxq_debug.so`` with ``-DMXQ_DEBUG``: the same
kernels with every computed global address of their plain loads and stores
checked against its buffer's extent (an access outside is skipped and
reported through the device error word) -- the bounds checking that stands in
for a memory-checking tool.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_obj")
LIB = os.path.join(HERE, "libmxq.so")
DEBUG_LIB = os.path.join(HERE, "libmxq_debug.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + \
        [os.path.join(INCLUDE, "mxq.h"), os.path.abspath(__file__)]


def up_to_date(debug: bool = False) -> bool:
    lib = DEBUG_LIB if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if needed) and return the path of libmxq.so (or, with debug,
    of libmxq_debug.so)."""
    lib = DEBUG_LIB if debug else LIB
    if not force and up_to_date(debug):
        return lib
    obj_dir = OBJ + ("_debug" if debug else "")
    os.makedirs(obj_dir, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc(), *ARCH, *FLAGS, *(["-DMXQ_DEBUG"] if debug else []), "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if failed:
        raise RuntimeError("libmxq build failed:\n" + "\n".join(failed))
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lpthread"])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
