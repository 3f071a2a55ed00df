"""Build the AirCache CUDA library in-tree: csrc/*.cu -> libaircache.so (sm_103a).

Plain nvcc, one translation unit per kernel file compiled in parallel, linked
into one shared library with the CUDA runtime linked statically.  Usage:
``python -m lvlm_kv_cache_gb300.build`` (or ``build()`` from Python).
``build(timeline=True)`` makes the separate measurement build
``libaircache_timeline.so`` (kernels compiled with -DAIRCACHE_TIMELINE: each
compression kernel's CTAs record their entry and exit times; see
csrc/timeline.cuh and ``bench.py --timeline``).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libaircache.so")
OBJ_TIMELINE = os.path.join(HERE, "_build_timeline")
LIB_TIMELINE = os.path.join(HERE, "libaircache_timeline.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", os.path.join(ROOT, "include"), "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(ROOT, "include", "aircache.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, verbose: bool, timeline: bool = False) -> str:
    obj = os.path.join(OBJ_TIMELINE if timeline else OBJ, os.path.basename(src)[:-3] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()):
        return obj
    cmd = [_nvcc(), *ARCH, *FLAGS, *(["-DAIRCACHE_TIMELINE"] if timeline else []), "-c", src, "-o", obj + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip() and verbose:
        print(res.stderr, file=sys.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, timeline: bool = False) -> str:
    obj_dir, lib = (OBJ_TIMELINE, LIB_TIMELINE) if timeline else (OBJ, LIB)
    os.makedirs(obj_dir, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, timeline), srcs))
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs):
        return lib
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", lib + ".tmp", *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
