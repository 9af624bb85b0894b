"""Build the C-ABI shared library ``libskinny_gemm.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc in parallel, then linked into
``skinny_bf16_projection_gb300/libskinny_gemm.so`` against the shared CUDA
runtime.  Rebuilds only when a source or header is newer than the library.

The same sources built with ``-DSKG_DEVICE_CHECKS=1`` give
``libskinny_gemm_checked.so``: every guarded shared-memory, TMEM, DSMEM and
global access is tested against its bounds first, and a failed test is reported
through the handle's status word instead of being performed (the stand-in for a
memory checker).  ``build_all`` builds both, their translation units in one pool.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(ROOT, "_build", "obj")
LIB_PATH = os.path.join(PKG, "libskinny_gemm.so")
CHECKED_OBJ_DIR = os.path.join(ROOT, "_build", "obj_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libskinny_gemm_checked.so")
CHECKED_FLAGS = ["-DSKG_DEVICE_CHECKS=1"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libskinny_gemm.so")


def _cuda_lib_dir(nvcc: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        d = os.path.join(root, sub)
        if os.path.exists(os.path.join(d, "libcudart.so")):
            return d
    return os.path.join(root, "lib64")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    deps += glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _variants(checked: bool) -> list[tuple[str, str, list[str]]]:
    out = [(LIB_PATH, OBJ_DIR, [])]
    if checked:
        out.append((CHECKED_LIB_PATH, CHECKED_OBJ_DIR, CHECKED_FLAGS))
    return out


def _build(variants, force: bool, verbose: bool, ptxas_verbose: bool) -> None:
    todo = [v for v in variants if force or _stale(v[0])]
    if not todo:
        return
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(job: tuple[str, str, list[str]]) -> str:
        src, obj_dir, flags = job
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *CFLAGS, *flags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose or ptxas_verbose:
            sys.stderr.write(r.stderr)
        return obj

    jobs = []
    for _, obj_dir, flags in todo:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, obj_dir, flags) for src in sources()]
    # the longest translation units first, so they do not finish last
    jobs.sort(key=lambda j: -os.path.getsize(j[0]))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, jobs))
    libdir = _cuda_lib_dir(nvcc)
    for lib, obj_dir, _ in todo:
        mine = [o for o in objs if os.path.dirname(o) == obj_dir]
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *mine,
               "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link the library; returns its path."""
    _build(_variants(False), force, verbose, ptxas_verbose)
    return LIB_PATH


def build_all(force: bool = False, verbose: bool = False) -> tuple[str, str]:
    """Build the library and its checked variant; returns both paths."""
    _build(_variants(True), force, verbose, False)
    return LIB_PATH, CHECKED_LIB_PATH


if __name__ == "__main__":
    if "--checked" in sys.argv:
        print(build_all(force="--force" in sys.argv, verbose="-v" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                    ptxas_verbose="--ptxas" in sys.argv))
