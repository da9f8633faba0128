"""Builds libsptp.so in-tree from csrc/*.cu for sm_103a with nvcc.

Each translation unit is compiled in parallel to an object under _build/ and
the objects are linked into sequence_tensor_transformer_gb300/libsptp.so.  An
object is rebuilt when its source or any header is newer.

build(checked=True) builds the bounds-checked library libsptp_check.so
(objects under _build/check/): the same kernels compiled with
-DSPTP_BOUNDS_CHECK, which check every index and address they compute
against its buffer and report a failure as SPTP_ERR_BOUNDS in the workspace
status words.  It is a debug build for the tests, slower than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libsptp.so")
CHECKED_LIB = os.path.join(PKG, "libsptp_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
         "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compile every CUDA source and link libsptp.so (checked: the
    bounds-checked libsptp_check.so); returns its path."""
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "check") if checked else BUILD
    lib_path = CHECKED_LIB if checked else LIB
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = _headers()
    flags = FLAGS + (["-DSPTP_BOUNDS_CHECK"] if checked else []) + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        if _stale(obj, [src] + hdrs) or extra_flags:
            cmd = [nvcc] + ARCH + flags + ["-c", src, "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    if _stale(lib_path, objs) or extra_flags:
        tmp = lib_path + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(verbose=True, checked="--checked" in sys.argv[1:]))
