"""Build libfadam.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process, in parallel, then
the objects are linked into one shared library with the CUDA runtime linked
statically.  Set FADAM_PTXAS_VERBOSE=1 to print register and shared-memory
use per kernel.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libfadam.so")

SOURCES = ["fadam_plan.cu"] + [f"fadam_kernels_s{s}_g{g}.cu"
                               for s in ("f32", "bf16", "f16", "f32mbf16", "f32mf16")
                               for g in ("f32", "bf16", "f16")] + [
    f"fadam_kernels_{kind}s{s}_g{g}.cu" for kind in ("scaled_", "recip_", "recip_scaled_")
    for s in ("bf16", "f16") for g in ("f32", "bf16", "f16")]
HEADERS = ["fadam_internal.h", "fadam_kernel.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
    "--ftz=false", "--prec-div=true", "--prec-sqrt=true",
]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "fadam.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), lib: str = LIB) -> str:
    """Compile and link libfadam.so if it is missing or out of date.

    `defines` (e.g. ["FADAM_UNROLL=4"]) override the kernel's compile-time
    tuning defaults; `lib` puts such a build elsewhere.
    """
    if not force and not defines and not _stale(lib):
        return lib
    out_dir = os.path.dirname(os.path.abspath(lib))
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if os.environ.get("FADAM_PTXAS_VERBOSE") == "1" else []
    extra += [f"-D{d}" for d in defines]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or extra or p.returncode):
            sys.stdout.write(out)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
           "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
