"""Build liblocks.so in-tree with nvcc for sm_103a (GB300).

    python -m sparse_kv_page_rank_gb300.build_lib [--verbose]

Each .cu file compiles to an object in parallel; the objects link into
``sparse_kv_page_rank_gb300/_lib/liblocks.so`` with the CUDA runtime linked
statically, so the library depends on neither torch nor libcuda at link time
(the TMA descriptor encoder is looked up through the runtime's driver entry
point at first use).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "liblocks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr"]
SOURCES = ["api.cu", "scan.cu", "topk.cu", "attend.cu", "build.cu", "static_ws.cu"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"command failed ({p.returncode}): {' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
    return p.stdout + p.stderr


def build(verbose: bool = False, extra_flags=(), force: bool = False) -> str:
    """Compile and link; returns the library path.  Skips work when the library
    is newer than every source and header."""
    os.makedirs(OUT_DIR, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "locks.h"))
    if not force and os.path.exists(LIB):
        lib_t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) < lib_t for d in deps):
            return LIB
    cc = nvcc()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([cc, *ARCH, *CFLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj])
    outputs = []
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        for out in ex.map(lambda c: _run(c, verbose), cmds):
            outputs.append(out)
    tmp = LIB + ".tmp"
    _run([cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], verbose)
    os.replace(tmp, LIB)
    if verbose:
        for o in outputs:
            if o.strip():
                print(o)
    return LIB


if __name__ == "__main__":
    v = "--verbose" in sys.argv
    flags = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(verbose=v or bool(flags), extra_flags=flags, force=bool(flags) or "--force" in sys.argv))
