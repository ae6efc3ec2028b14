"""Compile the CUDA library (libqe.so) in-tree for sm_103a.

Each translation unit is compiled in its own nvcc process (in parallel) and then linked
into ``tiered_quantize_evict_gb300/_lib/libqe.so``.  No cmake, no torch extension machinery:
the library is a plain C-ABI shared object.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
BUILD = os.path.join(HERE, "_build")
SOURCES = ["qe_attn.cu", "qe_route.cu", "qe_host.cu", "qe_noalloc.cu", "qe_tok.cu", "qe_tok_host.cu", "qe_verify.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def compile_units(sources, out_so, include_dirs, extra=()):
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(os.path.dirname(out_so), exist_ok=True)
    inc = [f"-I{d}" for d in include_dirs]
    objs, jobs = [], []
    with cf.ThreadPoolExecutor(max_workers=len(sources)) as ex:
        for src in sources:
            obj = os.path.join(BUILD, os.path.basename(src) + ".o")
            objs.append(obj)
            jobs.append(ex.submit(_run, [nvcc(), *ARCH, *FLAGS, *extra, *inc, "-c", src, "-o", obj]))
        for j in jobs:
            j.result()
    tmp = out_so + ".tmp"
    _run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
    os.replace(tmp, out_so)
    return out_so


def build_library() -> str:
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    return compile_units(srcs, os.path.join(LIBDIR, "libqe.so"), [os.path.join(ROOT, "include"), CSRC])


if __name__ == "__main__":
    print(build_library())
    sys.exit(0)
