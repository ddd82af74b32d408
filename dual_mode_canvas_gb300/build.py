"""Builds the dg_attn shared library in-tree with nvcc for sm_103a.

``python -m dual_mode_canvas_gb300.build`` (or ``build_all()``) compiles
``csrc/dg_attn.cu`` twice, in parallel:

* ``dual_mode_canvas_gb300/lib/libdg_attn.so``: the library;
* ``dual_mode_canvas_gb300/lib/libdg_attn_debug.so``: the same sources with
  ``-DDG_ATTN_DEBUG``, whose kernels check every TMA coordinate, shared-memory
  destination, TMEM column and global index before the access and report a
  failed check as DG_ERR_DEVICE_BOUNDS in the status word.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "dg_attn.cu")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libdg_attn.so")
LIB_DEBUG = os.path.join(LIB_DIR, "libdg_attn_debug.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    csrc = os.path.join(PKG, "csrc")
    return [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith((".cu", ".cuh"))] + [
        os.path.join(INCLUDE, "dg_attn.h")]


def lib_path(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB


def up_to_date(debug: bool = False) -> bool:
    lib = lib_path(debug)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in sources())


def _command(out: str, debug: bool, verbose: bool, extra_flags) -> list:
    cmd = [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", os.path.join(PKG, "csrc"), SRC, "-o", out]
    if debug:
        cmd.insert(2, "-DDG_ATTN_DEBUG")
    if verbose:
        cmd.insert(2, "-Xptxas=-v")
    cmd.extend(extra_flags)
    return cmd


def _start(debug: bool, verbose: bool, extra_flags):
    lib = lib_path(debug)
    tmp = lib + ".tmp"
    cmd = _command(tmp, debug, verbose, extra_flags)
    return lib, tmp, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)


def _finish(lib, tmp, cmd, proc, verbose):
    out, err = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out + err)
    if verbose:
        sys.stderr.write(out + err)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Builds one library (the checking build with ``debug=True``)."""
    if not force and up_to_date(debug):
        return lib_path(debug)
    os.makedirs(LIB_DIR, exist_ok=True)
    return _finish(*_start(debug, verbose, extra_flags), verbose)


def build_all(force: bool = False, verbose: bool = False) -> list:
    """Builds the library and the checking build, the two nvcc runs in parallel."""
    os.makedirs(LIB_DIR, exist_ok=True)
    jobs = [_start(d, verbose, ()) for d in (False, True) if force or not up_to_date(d)]
    for job in jobs:
        _finish(*job, verbose)
    return [LIB, LIB_DEBUG]


if __name__ == "__main__":
    print(build_all(force=True, verbose="-v" in sys.argv))
