"""Build libft.so (the C-ABI library) from csrc/ with nvcc for sm_103a.

Each .cu file compiles to an object in parallel; the objects link into
``_build/libft.so`` with the CUDA runtime linked statically, so the library
loads next to any PyTorch build without sharing its runtime.  The checked
build (``-DFT_CHECKED``: kernels bounds-check the table and plan indices they
dereference and report FT_ERR_CHECKED instead of touching memory out of
range) goes to ``_build_checked/libft.so``; the package loads it when the
environment has FT_CHECKED=1.

    python expert_cache_host_layer_gb300/build.py [--force] [--checked]
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libft.so")
OUT_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(OUT_CHECKED, "libft.so")
OUT_UBSAN = os.path.join(HERE, "_build_ubsan")
LIB_UBSAN = os.path.join(OUT_UBSAN, "libft.so")
UBSAN = ["-Xcompiler", "-fsanitize=undefined", "-Xcompiler", "-fno-sanitize-recover=all"]
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.h"))) + [os.path.join(INCLUDE, "ft.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False, ubsan: bool = False) -> str:
    """checked: the bounds-checked build; ubsan: the host code compiled with
    UndefinedBehaviorSanitizer (loaded with FT_SANITIZE=1; the host-sanitizer
    test runs the CPU tests of the ABI against it)."""
    out, lib = (OUT_CHECKED, LIB_CHECKED) if checked else (OUT_UBSAN, LIB_UBSAN) if ubsan else (OUT, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    cc = nvcc()
    srcs = _sources()
    objs = [os.path.join(out, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = (["-DFT_CHECKED"] if checked else []) + (UBSAN if ubsan else [])

    def compile_one(src_obj):
        src, obj = src_obj
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return r.stderr

    workers = max(1, min(len(srcs), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        for msg in ex.map(compile_one, zip(srcs, objs)):
            if verbose and msg.strip():
                print(msg, file=sys.stderr)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", *(UBSAN if ubsan else []), "-o", tmp, *objs, "-lpthread",
           "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv,
                ubsan="--ubsan" in sys.argv))
