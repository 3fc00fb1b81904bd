"""In-tree build of libcpt.so for sm_103a.

Each CUDA translation unit is compiled by nvcc in parallel, then linked into
one shared library next to this file. The CUDA runtime is linked statically
and the driver API is reached through the runtime's entry-point query, so
the library needs no libcuda at link time.

Floating-point flags: -fmad=false -ftz=false -prec-div=true -prec-sqrt=true.
The kernels use explicit round-to-nearest adds anyway; the flags keep any
other arithmetic IEEE as well.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["cpt_api.cu", "index_map.cu", "gather.cu", "grad_return.cu", "slot_reduce.cu", "ceiling.cu"]
HEADERS = ["cpt_internal.h", "cpt_device.cuh"]

# The two builds of the library: the product, and the same sources with
# every device index checked before use (CPT_CHECK_BOUNDS), for debugging and
# for running the parity suite against.
VARIANTS = {
    "release": ("libcpt.so", []),
    "checked": ("libcpt_checked.so", ["-DCPT_CHECK_BOUNDS"]),
}
LIB = os.path.join(PKG, VARIANTS["release"][0])

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE, "-I", CSRC,
]


def library_path(variant: str = "release") -> str:
    return os.path.join(PKG, VARIANTS[variant][0])


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcpt.so")
    return path


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in HEADERS]
            + [os.path.join(INCLUDE, "cpt.h"), os.path.abspath(__file__)])


def is_stale(variant: str = "release") -> bool:
    lib = library_path(variant)
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variants=("release", "checked")) -> str:
    """Compile (where stale) the given variants, every translation unit of
    every variant in one parallel pool, and return the path of libcpt.so."""
    todo = [v for v in variants if force or is_stale(v)]
    if not todo:
        return LIB
    cc = nvcc()

    def compile_one(job):
        variant, src = job
        out_dir = os.path.join(ROOT, "_build", "cpt" if variant == "release" else f"cpt_{variant}")
        os.makedirs(out_dir, exist_ok=True)
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + NVCC_FLAGS + VARIANTS[variant][1] + list(extra_flags) + [
            "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    jobs = [(v, s) for v in todo for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in todo:
        lib = library_path(v)
        tmp = lib + f".tmp{os.getpid()}"
        mine = [o for (vv, _), o in zip(jobs, objs) if vv == v]
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + mine + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({v}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else []))
