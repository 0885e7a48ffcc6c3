"""Build libidx.so in-tree with nvcc for sm_103a (no cmake).

Each ``csrc/*.cu`` compiles to an object in parallel; the objects link into
``sparse_attention_top_paged_gb300/libidx.so``. Objects are rebuilt only when a
source or header is newer.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libidx.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libidx")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose: bool = False, extra_flags=()) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if (not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_hdr)):
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for log in ex.map(lambda j: _compile(nvcc, j[0], j[1], list(extra_flags)), jobs):
                if verbose and log:
                    print(log)
    if jobs or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-lpthread", "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libidx.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines=(), sources=None) -> str:
    """Build ``libidx_<name>.so`` beside libidx.so with extra preprocessor
    ``defines`` (e.g. the failure-path test's short wait limit): the listed
    ``sources`` (default: every ``csrc/*.cu``) are recompiled with them into
    ``_build/<name>/`` and linked with the in-tree objects of the others.
    Used by tests only; the product library is ``build()``'s."""
    build()
    nvcc = _nvcc()
    vdir = os.path.join(BUILD, name)
    os.makedirs(vdir, exist_ok=True)
    flags = [f"-D{d}" for d in defines]
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    chosen = set(sources) if sources is not None else {os.path.basename(x) for x in srcs}
    objs, jobs = [], []
    for src in srcs:
        base = os.path.basename(src)[:-3] + ".o"
        if os.path.basename(src) in chosen:
            obj = os.path.join(vdir, base)
            jobs.append((src, obj))
        else:
            obj = os.path.join(BUILD, base)
        objs.append(obj)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda j: _compile(nvcc, j[0], j[1], flags), jobs))
    lib = os.path.join(PKG, f"libidx_{name}.so")
    cmd = [nvcc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart_static", "-lrt", "-lpthread", "-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
