"""Builds libfr.so (the sm_103a kernels and the C ABI) in-tree.

Each ``csrc/*.cu`` file is compiled to an object in parallel with one
``-gencode arch=compute_103a,code=sm_103a``; the objects are linked into
``_lib/libfr.so`` against the shared CUDA runtime (so the library and PyTorch
share one runtime and context).  ``-Xptxas -v`` register/spill lines go to
``_lib/ptxas.log``.  No cmake, no torch extension machinery.

Usage: ``python -m reduction_pointwise_row_gb300.buildlib [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libfr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfr.so")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(CSRC, "*.h"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "-I", INCLUDE, *ARCH]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        r = subprocess.run([nvcc, *common, "-c", src, "-o", obj], capture_output=True, text=True)
        return src, obj, r

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    log = []
    for src, obj, r in results:
        log.append(f"== {os.path.basename(src)}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}{r.stderr}")
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp,
                        *[o for _, o, _ in results], "-L", libdir,
                        f"-Xlinker=-rpath={libdir}"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print("\n".join(log))
    return LIB


def build_variant(name: str, defines: list[str], recompile=("layernorm.cu",)) -> str:
    """A test-only variant of the library: the sources named in `recompile`
    compiled again with `defines` (e.g. ``["-DFR_TEST_WAIT_BUDGET=1"]``) and
    linked with the main build's other objects into ``_lib/<name>/libfr.so``.
    Nothing in the product loads it."""
    build()
    nvcc = _nvcc()
    out_dir = os.path.join(OUT_DIR, name)
    os.makedirs(out_dir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, *ARCH]
    objs = []
    for src in _sources():
        base = os.path.basename(src)
        if base in recompile:
            obj = os.path.join(out_dir, base + ".o")
            r = subprocess.run([nvcc, *common, *defines, "-c", src, "-o", obj],
                               capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}{r.stderr}")
        else:
            obj = os.path.join(OUT_DIR, "obj", base + ".o")
        objs.append(obj)
    lib = os.path.join(out_dir, "libfr.so")
    libdir = _cuda_lib_dir(nvcc)
    r = subprocess.run([nvcc, "-shared", *ARCH, "-cudart", "shared", "-o", lib, *objs, "-L",
                        libdir, f"-Xlinker=-rpath={libdir}"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
