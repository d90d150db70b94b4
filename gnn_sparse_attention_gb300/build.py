"""Build the CUDA library ``_build/libgattn.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel to an object file,
then the objects are linked into one shared library that exports the C ABI of
``include/gattn.h``.  Rebuilds only what is older than its sources.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libgattn.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build gattn")


def flags(extra=()):
    return [ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
            f"-I{INCLUDE}", f"-I{CSRC}", *extra]


def _deps():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build(verbose: bool = False, jobs: int | None = None) -> str:
    os.makedirs(OUT, exist_ok=True)
    units = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = _deps()
    objs = []
    todo = []
    for cu in units:
        obj = os.path.join(OUT, os.path.basename(cu)[:-3] + ".o")
        objs.append(obj)
        if _stale(obj, [cu, *deps]):
            todo.append((cu, obj))

    def compile_one(job):
        cu, obj = job
        cmd = [nvcc(), *flags(), "-c", cu, "-o", obj + ".tmp"]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(cu)}:\n{r.stdout}{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return r.stderr

    if todo:
        n = jobs or min(len(todo), os.cpu_count() or 4)
        with ThreadPoolExecutor(max_workers=n) as ex:
            for msg in ex.map(compile_one, todo):
                if verbose and msg:
                    print(msg, file=sys.stderr)
    if todo or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc(), ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
