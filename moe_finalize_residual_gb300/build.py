"""Build the CUDA library libmoe_finalize.so in-tree with nvcc (sm_103a only).

Each translation unit compiles in parallel; the objects link into one shared library next to this
file, against the shared CUDA runtime (the one PyTorch already loaded, when it did).
"""
from __future__ import annotations

import concurrent.futures
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_finalize.so")
SOURCES = ["api.cu", "kernel_cluster.cu", "kernel_stream.cu", "kernel_bulk.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    f += os.environ.get("MFR_NVCC_FLAGS", "").split()  # e.g. -DMFR_STREAM_COMPUTE_WARPS=24
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src, os.path.join(INCLUDE, "moe_finalize.h")] + [
        os.path.join(CSRC, n) for n in os.listdir(CSRC) if n.endswith((".cuh", ".h"))]
    return any(os.path.getmtime(d) > os.path.getmtime(obj) for d in deps)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    """Compile (only what changed, unless ``force``) and link.  Returns the library path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "MACHINE")
    machine = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != machine:
        force = True  # objects from another architecture must not be linked here
        with open(stamp, "w") as f:
            f.write(machine + "\n")
    jobs = []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name.replace(".cu", ".o"))
        if force or ptxas_verbose or _stale(obj, src):
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc()] + _flags(ptxas_verbose) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        return r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(compile_one, jobs))
    if not quiet:
        for log in logs:
            print(log)
    objs = [os.path.join(BUILD, n.replace(".cu", ".o")) for n in SOURCES]
    if jobs or force or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc())), "lib64")
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-Xlinker", "-rpath," + cuda_lib, "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv, quiet=False))
