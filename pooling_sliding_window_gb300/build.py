"""Build libfusedwin.so in-tree (``pooling_sliding_window_gb300/_build/``).

Every CUDA translation unit under ``csrc/`` is compiled in parallel by nvcc for
sm_103a only (``-gencode arch=compute_103a,code=sm_103a``) and linked into one
shared library with the CUDA runtime linked statically.  Rebuilds are
incremental on source / header modification times.

``checked=True`` builds the bounds-checked variant (``-DFW_CHECKED=1``) into
``_build/checked/libfusedwin_checked.so``: every kernel tests the address range of
its memory accesses and reports a range violation through the device error word
instead of making the access.  The binding loads it when FUSEDWIN_CHECKED=1.

Usage: ``python -m pooling_sliding_window_gb300.build [--verbose-ptxas] [--checked]``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libfusedwin.so")
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
LIB_CHECKED = os.path.join(CHECKED_DIR, "libfusedwin_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: libfusedwin needs the CUDA toolkit to build")


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + [os.path.join(ROOT, "include", "fusedwin.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose_ptxas: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compile and link libfusedwin.so (or the bounds-checked variant); returns its path."""
    out_dir, lib = (CHECKED_DIR, LIB_CHECKED) if checked else (OUT_DIR, LIB)
    os.makedirs(out_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
    if checked:
        flags += ["-DFW_CHECKED=1"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    flags += list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max(1, min(len(sources), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, sources))
    for src, _, r in results:
        if verbose_ptxas or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
    tmp = lib + f".{os.getpid()}.tmp"
    link = [cc, *ARCH, "-shared", "-o", tmp] + [o for _, o, _ in results]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"linking {os.path.basename(lib)} failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose_ptxas="--verbose-ptxas" in sys.argv, checked="--checked" in sys.argv))
