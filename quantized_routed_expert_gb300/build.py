"""Build libmoe (``csrc/*.cu``) for sm_103a into ``_build/libmoe.so``.

One nvcc process per translation unit, run in parallel, then one link. The
library is built in-tree so that the Python binding loads exactly this file.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                "-I", INCLUDE, "-I", SRC]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(SRC, "*.cu")))


def _deps():
    return (sorted(glob.glob(os.path.join(SRC, "*"))) + [os.path.join(INCLUDE, "moe.h")])


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), profile: bool = False) -> str:
    """Compile every csrc/*.cu and link _build/libmoe.so. profile=True builds the
    phase-stamp variant (-DMOE_PROFILE, exporting moe_profile_stamps) into
    _build_profile/libmoe.so instead; the product library never has it."""
    build_dir = os.path.join(HERE, "_build_profile" + os.environ.get("MOE_PROFILE_TAG", "")) \
        if profile else BUILD
    lib = os.path.join(build_dir, "libmoe.so")
    if profile:
        extra_flags = tuple(extra_flags) + ("-DMOE_PROFILE",)
    os.makedirs(build_dir, exist_ok=True)
    deps = _deps()
    if not force and not _stale(lib, deps):
        return lib
    objs = []

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc(), *FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    srcs = _sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [],
                profile="--profile" in sys.argv))
