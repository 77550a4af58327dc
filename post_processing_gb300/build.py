"""Builds the in-tree CUDA library ``libws.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` compiles to an object in parallel, then one shared link.
The same sources compiled with ``-DWS_BOUNDS_CHECK`` (in the same parallel
batch) give ``libws_bounds.so``, the checked build: its kernels test their
shared-memory and tap indices, set an error bit and clamp instead of reading
or writing out of range.  Nothing is installed: the libraries sit next to
this file and the binding loads one of them from there (the checked one when
the environment sets WS_BOUNDS_CHECK=1).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJS = os.path.join(HERE, "_objs")
LIBRARY = os.path.join(HERE, "libws.so")
BOUNDS_OBJS = os.path.join(HERE, "_objs_bounds")
BOUNDS_LIBRARY = os.path.join(HERE, "libws_bounds.so")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCCFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY) or not os.path.exists(BOUNDS_LIBRARY):
        return False
    t = min(os.path.getmtime(LIBRARY), os.path.getmtime(BOUNDS_LIBRARY))
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (when stale) both libraries and return the path of libws.so."""
    if not force and up_to_date():
        return LIBRARY
    procs = []
    for objdir, extra in ((OBJS, []), (BOUNDS_OBJS, ["-DWS_BOUNDS_CHECK"])):
        os.makedirs(objdir, exist_ok=True)
        for src in sources():
            obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
            cmd = [NVCC, *ARCH, *NVCCFLAGS, *extra, "-c", src, "-o", obj]
            if verbose_ptxas and not extra:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((objdir, obj, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs, failed = {OBJS: [], BOUNDS_OBJS: []}, []
    for objdir, obj, cmd, proc in procs:
        out, _ = proc.communicate()
        if out:
            sys.stderr.write(out.decode(errors="replace"))
        if proc.returncode != 0:
            failed.append(" ".join(cmd))
        objs[objdir].append(obj)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    for objdir, lib in ((OBJS, LIBRARY), (BOUNDS_OBJS, BOUNDS_LIBRARY)):
        tmp = lib + ".tmp%d" % os.getpid()
        subprocess.run([NVCC, *ARCH, "-shared", *objs[objdir], "-o", tmp], check=True)
        os.replace(tmp, lib)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
