"""Build libflux_gb300.so (the C-ABI library) in place with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into a shared library beside this file.  The CUDA runtime is linked
dynamically so the library shares one runtime instance with PyTorch.

Usage:  python -m reducescatter_tcgen05_tmem_gb300.build  [--verbose]
"""
from __future__ import annotations

import fcntl
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libflux_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
# the checked build: the same sources with every kernel access checked
# (-DFLUX_CHECKS=1; loaded by the binding when FLUX_CHECKED=1)
CHECKED_LIB_PATH = os.path.join(HERE, "libflux_gb300_checked.so")

SOURCES = ["flux_core.cu", "flux_dense.cu", "flux_moe.cu", "flux_noalloc.cu", "flux_tune.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "-diag-suppress", "550", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def _run(cmd, verbose):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd[:3])} ...")
    return r.stdout + r.stderr


def _up_to_date() -> bool:
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "flux_gb300.h"))
    deps.append(__file__)
    newest = max(os.path.getmtime(d) for d in deps)
    return all(os.path.exists(lib) and os.path.getmtime(lib) >= newest
               for lib in (LIB_PATH, CHECKED_LIB_PATH))


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link; returns the path of the shared library.

    Several processes may call this at once (one per rank of a multi-GPU
    launch): they take turns on a lock file, and whoever comes after a
    finished build finds the library up to date and returns."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    if not force and _up_to_date():
        return LIB_PATH
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        if not force and _up_to_date():
            return LIB_PATH
        return _build_locked(nvcc, verbose)


def _build_locked(nvcc: str, verbose: bool) -> str:
    # both libraries' translation units compile in parallel
    variants = ((LIB_PATH, BUILD, []), (CHECKED_LIB_PATH, os.path.join(BUILD, "checked"), ["-DFLUX_CHECKS=1"]))
    jobs = []
    for lib, bdir, defs in variants:
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            jobs.append((src, os.path.join(bdir, src.replace(".cu", ".o")), defs))

    def compile_one(job):
        src, obj, defs = job
        _run([nvcc, *ARCH, *CFLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj], verbose)
        return obj

    with ThreadPoolExecutor(len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    libdir = _cuda_lib_dir(nvcc)
    for i, (lib, _, _) in enumerate(variants):
        tmp = f"{lib}.tmp{os.getpid()}"
        _run([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
              *objs[i * len(SOURCES):(i + 1) * len(SOURCES)],
              f"-L{libdir}", "-Xlinker", f"-rpath={libdir}"], verbose)
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))
