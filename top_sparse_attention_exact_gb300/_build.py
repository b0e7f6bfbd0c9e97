"""In-tree build of the CUDA library (sm_103a only).

Compiles every ``csrc/*.cu`` file in parallel with nvcc and links them into
``_build/libretopk.so``.  No cmake, no torch extension machinery: the library
exposes a plain C ABI (include/retopk.h) that the ctypes binding loads.

``build(checked=True)`` makes ``_build/checked/libretopk_checked.so``, the same
library compiled with ``RETOPK_CHECKED`` defined: every K / V row a kernel
gathers is range-checked against the sequence length first (a violation sets
RETOPK_STATUS_GATHER and the row is skipped).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libretopk.so")
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
LIB_CHECKED = os.path.join(CHECKED_DIR, "libretopk_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libretopk")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I", os.path.join(ROOT, "include"), *extra]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "retopk.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = False) -> str:
    """Compile (if stale) and return the path of libretopk.so (of
    libretopk_checked.so with checked=True)."""
    lib, out_dir = (LIB_CHECKED, CHECKED_DIR) if checked else (LIB, OUT_DIR)
    if checked:
        extra = (*extra, "-DRETOPK_CHECKED")
    if not force and not _stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    objs = []

    def one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *_flags(extra), "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(one, sources()))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
