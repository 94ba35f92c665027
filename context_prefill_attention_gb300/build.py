"""Build libpcp.so in-tree for sm_103a (nvcc, no CMake).

Each translation unit under ``csrc/`` is compiled in parallel into
``_build/``, then linked into ``libpcp.so`` next to this file. Rebuilds only
what is older than its sources.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpcp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: libpcp needs the CUDA 13 toolkit")


def _flags(verbose_ptxas: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
                "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _deps():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, sources) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _compile(src: str, verbose_ptxas: bool, build_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if not verbose_ptxas and not extra and not _stale(obj, [src] + _deps()):
        return obj
    cmd = [_nvcc(), "-c", src, "-o", obj + ".tmp"] + _flags(verbose_ptxas) + list(extra)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose_ptxas: bool = False, jobs: int = 0, defines=(), out: str = LIB) -> str:
    """Compile and link ``libpcp.so``; returns its path. ``defines`` (e.g.
    ``["PCP_POLY_EXP_EVERY=8"]``) override the kernels' compile-time tuning
    knobs; such a build goes to ``out`` through a build folder of its own."""
    extra = [f"-D{d}" for d in defines]
    build_dir = BUILD if not extra else out + ".build"
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    jobs = jobs or min(len(srcs), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, build_dir, extra), srcs))
    LIB_OUT = out
    if extra or _stale(LIB_OUT, objs):
        tmp = LIB_OUT + f".tmp{os.getpid()}"
        cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libpcp.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB_OUT)
    return LIB_OUT


if __name__ == "__main__":
    print(build(verbose_ptxas="-v" in sys.argv))
