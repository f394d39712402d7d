"""Builds libbkv.so in-tree with nvcc for sm_103a (GB300).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
kv_cache_eviction_head_gb300/libbkv.so with the static CUDA runtime. A stamp of
the sources, the flags and the compiler version skips the build when nothing
changed.

build(checked=True) makes the bounds-checked variant, libbkv_checked.so
(-DBKV_CHECKED: every computed index is tested before use and a failure
latches BKV_ERR_INTERNAL); the binding loads it when BKV_LIBRARY=checked.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libbkv.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libbkv_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libbkv")
    return cand


def _stamp(sources: list[str], nvcc: str) -> str:
    h = hashlib.sha256()
    for p in sorted(sources + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "bkv.h")]):
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + CFLAGS).encode())
    h.update(subprocess.run([nvcc, "--version"], capture_output=True, text=True).stdout.encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(verbose: bool = False, extra_flags: list[str] | None = None, checked: bool = False) -> str:
    """Compile every csrc/*.cu and link libbkv.so (libbkv_checked.so with
    checked=True); returns the library path."""
    nvcc = _nvcc()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra_flags or []) + (["-DBKV_CHECKED=1"] if checked else [])
    flags = CFLAGS + extra
    lib, bdir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    stamp = _stamp(sources, nvcc) + ("|" + " ".join(extra) if extra else "")
    stamp_path = os.path.join(bdir, "stamp")
    if os.path.exists(lib) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return lib
    os.makedirs(bdir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        objs = list(ex.map(compile_one, sources))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


def build_all(verbose: bool = False) -> list[str]:
    """The regular and the bounds-checked library."""
    return [build(verbose=verbose), build(verbose=verbose, checked=True)]


if __name__ == "__main__":
    print(build_all(verbose="-v" in sys.argv))
