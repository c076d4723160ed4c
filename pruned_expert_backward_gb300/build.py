"""Build liblrm.so (the C ABI of include/lrm.h) for sm_103a with nvcc.

Each .cu under csrc/ compiles to an object in parallel; the objects link into
pruned_expert_backward_gb300/liblrm.so (static CUDA runtime, no other dependency).
The same sources compiled with -DLRM_DEBUG link into liblrm_debug.so: every index the
kernels form themselves is checked as well (a failed check records LRM_ERR_BAD_INDEX in the
status word and skips the access).  Both builds run side by side by default.
Run: python -m pruned_expert_backward_gb300.build [--release-only] [-v]
(or __graft_entry__.build()).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "liblrm.so")
LIB_DEBUG = os.path.join(PKG, "liblrm_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build liblrm.so")


def _newest_dep_mtime() -> float:
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(p) for p in deps)


def _compile(src: str, extra: list[str], verbose_ptxas: bool, outdir: str = BUILD) -> str:
    obj = os.path.join(outdir, os.path.basename(src).replace(".cu", ".o"))
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _newest_dep_mtime()) \
            and not verbose_ptxas:
        return obj
    cmd = [nvcc()] + ARCH + FLAGS + extra + (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _link(objs: list[str], lib: str, force: bool) -> str:
    if os.path.exists(lib) and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs) and not force:
        return lib
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(verbose_ptxas: bool = False, extra: list[str] | None = None, debug: bool = True) -> str:
    """Compile and link liblrm.so (and, with debug, liblrm_debug.so); returns the release path."""
    dbg_dir = os.path.join(BUILD, "debug")
    os.makedirs(dbg_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = [(s, extra or [], BUILD) for s in srcs]
    if debug:
        jobs += [(s, (extra or []) + ["-DLRM_DEBUG"], dbg_dir) for s in srcs]
    # the largest translation unit first, so it does not start last
    jobs.sort(key=lambda j: -os.path.getsize(j[0]))
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 8, len(jobs))) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], j[1], verbose_ptxas, j[2]), jobs))
    rel = sorted(o for o in objs if os.path.dirname(o) == BUILD)
    _link(rel, LIB, bool(extra))
    if debug:
        _link(sorted(o for o in objs if os.path.dirname(o) == dbg_dir), LIB_DEBUG, bool(extra))
    return LIB


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv, debug="--release-only" not in sys.argv))
