"""Builds the loss-head shared library (libflce.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
``lm_head_linear_fwd_gb300/_lib/<machine>/libflce.so`` (static CUDA runtime, no torch
dependency).  ``python lm_head_linear_fwd_gb300/build.py [--checked]`` runs it.
"""
from __future__ import annotations

import concurrent.futures
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
# per machine architecture, so that objects built on one host are never linked on another
LIBDIR = os.path.join(PKG, "_lib", platform.machine())
LIB = os.path.join(LIBDIR, "libflce.so")
SOURCES = ["ce_logits.cu", "flce.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libflce.so")
    return cand


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compiles (if needed) and returns the path of libflce.so.

    ``checked=True`` builds the debug variant ``libflce_checked.so`` instead,
    with device-side index checks (``FLCE_DEVICE_CHECKS=1``): an index that
    leaves its range records FLCE_EBOUNDS in the status word and the access is
    skipped.  It is a separate file; the package always loads libflce.so."""
    nvcc = _nvcc()
    os.makedirs(LIBDIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    suffix = "_checked" if checked else ""
    defs = ["-DFLCE_DEVICE_CHECKS=1"] if checked else []
    lib = os.path.join(LIBDIR, f"libflce{suffix}.so")
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(LIBDIR, src.replace(".cu", f"{suffix}.o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *ARCH, *FLAGS, *defs, "-c", s, "-o", o])
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for out in ex.map(_run, jobs):
                if verbose and out.strip():
                    print(out)
    if force or jobs or _stale(lib, objs):
        _run([nvcc, *ARCH, "-shared", "-o", lib, *objs, "-ldl"])
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
