"""Build the CUDA library (libmoe_gb300.so) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel; the objects link into
one shared library next to this file.  No CMake, no torch extension machinery.
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
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_gb300.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


FLAGS_FILE = os.path.join(BUILD, "libmoe_gb300.flags")


def _built_flags() -> str:
    try:
        return open(FLAGS_FILE).read()
    except OSError:
        return ""


def up_to_date(extra_flags=()) -> bool:
    """The library exists, is newer than every source, and was built with these extra flags."""
    if not os.path.exists(LIB) or _built_flags() != " ".join(extra_flags):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    # MOE_CHECKED=1 in the environment selects the bounds-checked build for
    # every caller (the tests, the bench) that builds with default flags
    if not extra_flags and os.environ.get("MOE_CHECKED") == "1":
        extra_flags = ("-DMOE_CHECKED",)
    if not force and up_to_date(extra_flags):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(FLAGS_FILE, "w") as f:
        f.write(" ".join(extra_flags))
    return LIB


if __name__ == "__main__":
    # --checked: the bounds-checked build (-DMOE_CHECKED), a debugging build
    # whose kernels check computed indices before they access memory
    flags = ["-DMOE_CHECKED"] if "--checked" in sys.argv else []
    print(build(force="--force" in sys.argv or bool(flags), verbose=True, extra_flags=flags))
