"""Builds libcsa_gb300.so in-tree with nvcc for sm_103a only.

A built library is stamped with a SHA-256 of its sources (``<lib>.sha256``); it is
rebuilt whenever the sources differ from the stamp, and the binding refuses to
load a library whose stamp does not match the sources beside it.

Each ``csrc/*.cu`` is compiled to an object in parallel, then linked into a
shared library with the CUDA runtime linked statically (so loading the
library needs no GPU and no libcuda; the driver is reached at first use).
``build(debug=True)`` makes libcsa_gb300_debug.so from the same sources with
-DCSA_DEBUG: the kernels then check tile indices, ring indices and TMEM column
ranges on the device and report a failed check as CSA_ERR_CHECK.
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
LIBNAME = "libcsa_gb300.so"
LIBPATH = os.path.join(PKG, LIBNAME)
DEBUG_LIBPATH = os.path.join(PKG, "libcsa_gb300_debug.so")
DEBUG_BUILD = os.path.join(PKG, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cand, "bin", "nvcc")
    return p if os.path.exists(p) else (shutil.which("nvcc") or "nvcc")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                   "-I", INCLUDE, "-I", CSRC, *extra]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def source_hash(debug: bool = False) -> str:
    """SHA-256 of every source the library is built from (csrc/, include/, this file)
    and of the compiler flags: what a built library is stamped with."""
    h = hashlib.sha256()
    for f in sorted(_deps()):
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(ARCH + ["debug" if debug else "release"]).encode())
    return h.hexdigest()


def stamp_path(path: str) -> str:
    """The file beside a built library that holds the source hash it was built from."""
    return path + ".sha256"


def up_to_date(path: str = LIBPATH, debug: bool = False) -> bool:
    """True when the library exists and was built from the current sources."""
    if not os.path.exists(path) or not os.path.exists(stamp_path(path)):
        return False
    with open(stamp_path(path)) as f:
        return f.read().strip() == source_hash(debug)


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(DEBUG_BUILD if debug else BUILD,
                       os.path.basename(src).replace(".cu", ".o"))
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DCSA_DEBUG"] if debug else [])
    cmd = [nvcc(), *_flags(extra), "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link the library (or, with debug=True, its checking variant) if any
    source changed; returns its path."""
    path = DEBUG_LIBPATH if debug else LIBPATH
    if not force and up_to_date(path, debug):
        return path
    digest = source_hash(debug)
    os.makedirs(DEBUG_BUILD if debug else BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), srcs))
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, path)
    with open(stamp_path(path) + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(stamp_path(path) + f".tmp{os.getpid()}", stamp_path(path))
    return path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                debug="--debug" in sys.argv))
