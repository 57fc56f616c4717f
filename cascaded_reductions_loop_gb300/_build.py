"""Builds the C-ABI shared library (librf_gb300.so) from csrc/ with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
with the static CUDA runtime into ``_lib/librf_gb300.so`` inside the package.
The same sources are also built with RF_DEBUG_BOUNDS into
``_lib/librf_gb300_dbg.so``: the bounds-checked debug build, in which every
global load or store a kernel thread issues is checked against its tensor
(an access outside is skipped and reported as RF_ERR_DEVICE_BOUNDS).  A
rebuild happens only when a source or header is newer than a library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG_DIR, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB_NAME = "librf_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "librf_gb300_dbg.so")
DEBUG_OBJ_DIR = os.path.join(OUT_DIR, "obj_dbg")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE]
# (library, object directory, extra flags) of each build
VARIANTS = [(LIB_PATH, OBJ_DIR, []), (DEBUG_LIB_PATH, DEBUG_OBJ_DIR, ["-DRF_DEBUG_BOUNDS"])]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librf_gb300.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def is_stale(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles and links both libraries if needed (all objects in one
    parallel pool); returns the path of the normal one."""
    todo = [v for v in VARIANTS if force or is_stale(v[0])]
    if not todo:
        return LIB_PATH
    nvcc = nvcc_path()
    srcs = _sources()
    cmds, links = [], []
    for lib, obj_dir, flags in todo:
        os.makedirs(obj_dir, exist_ok=True)
        objs = [os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o") for src in srcs]
        cmds += [[nvcc, *ARCH, *NVCC_FLAGS, *flags, "-c", src, "-o", o] for src, o in zip(srcs, objs)]
        links.append((lib, objs))
    with ThreadPoolExecutor(max_workers=min(len(cmds), os.cpu_count() or 4)) as ex:
        outs = list(ex.map(_run, cmds))
    if verbose:
        for o in outs:
            if o.strip():
                print(o, file=sys.stderr)
    for lib, objs in links:
        tmp = lib + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
