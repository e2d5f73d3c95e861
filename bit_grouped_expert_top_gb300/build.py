"""Builds liblily_moe.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu file is compiled in parallel with nvcc into an object, then the
objects are linked into one shared library under ``_build/``.  The build is
skipped when the library is newer than every source and header.

Besides the product library there is one test-only variant,
``liblily_moe_stalltest.so``, built from the same sources with two macros: the
pipeline waits of the grouped GEMM give up after 1 ms instead of 2 s, and for
T == 77 the epilogue first waits on a barrier that nothing completes.  The
failure-path tests use it to make a bounded wait run out on purpose and check
that the kernel reports LILY_ERR_DEVICE_TIMEOUT, drains its in-flight work and
leaves the GPU usable.  The product library is never built with these macros.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
from typing import Dict, List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

# variant name -> (library file, extra nvcc flags)
STALL_TEST_T = 77
VARIANTS: Dict[str, tuple] = {
    "product": ("liblily_moe.so", []),
    "stalltest": ("liblily_moe_stalltest.so",
                  ["-DLILY_WAIT_LIMIT_NS=1000000ull", f"-DLILY_TEST_STALL_T={STALL_TEST_T}"]),
}


def lib_path(variant: str = "product") -> str:
    return os.path.join(OUT_DIR, VARIANTS[variant][0])


def _nvcc() -> str:
    cand = [shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources() -> List[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> List[str]:
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(variant: str = "product") -> bool:
    p = lib_path(variant)
    if not os.path.exists(p):
        return False
    t = os.path.getmtime(p)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile_jobs(variant: str):
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
    flags += VARIANTS[variant][1]
    return [(variant, src, flags) for src in _sources()]


def _compile_one(job, verbose: bool) -> str:
    variant, src, flags = job
    obj = os.path.join(OUT_DIR, f"{os.path.basename(src)}.{variant}.{os.getpid()}.o")
    r = subprocess.run([_nvcc()] + flags + ["-c", src, "-o", obj], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout, r.stderr)
    return obj


def _link(variant: str, objs: List[str]) -> str:
    tmp = lib_path(variant) + f".{os.getpid()}.tmp"
    r = subprocess.run([_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcuda"], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed ({variant}):\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path(variant))
    return lib_path(variant)


def build(force: bool = False, verbose: bool = False, variants=("product",)) -> str:
    """Compile and link the requested variants (all translation units of all
    variants in parallel); returns the path of the first one."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if todo:
        os.makedirs(OUT_DIR, exist_ok=True)
        jobs = [j for v in todo for j in _compile_jobs(v)]
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            objs = list(ex.map(lambda j: _compile_one(j, verbose), jobs))
        for v in todo:
            _link(v, [o for j, o in zip(jobs, objs) if j[0] == v])
    return lib_path(variants[0])


def build_all(force: bool = False, verbose: bool = False) -> str:
    """The product library and the test-only variant."""
    return build(force=force, verbose=verbose, variants=tuple(VARIANTS))


if __name__ == "__main__":
    print(build_all(force=True, verbose=True))
