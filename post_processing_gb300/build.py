"""Builds the in-tree CUDA library ``libws.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` compiles to an object in parallel, then one shared link.
Nothing is installed: the library sits next to this file and the binding
loads it from there.
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

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCCFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if not os.path.exists(LIBRARY):
        return False
    t = os.path.getmtime(LIBRARY)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile (when stale) and return the path of libws.so."""
    if not force and up_to_date():
        return LIBRARY
    os.makedirs(OBJS, exist_ok=True)
    procs = []
    for src in sources():
        obj = os.path.join(OBJS, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH, *NVCCFLAGS, "-c", src, "-o", obj]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((obj, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    objs, failed = [], []
    for obj, cmd, proc in procs:
        out, _ = proc.communicate()
        if out:
            sys.stderr.write(out.decode(errors="replace"))
        if proc.returncode != 0:
            failed.append(" ".join(cmd))
        objs.append(obj)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIBRARY + ".tmp%d" % os.getpid()
    subprocess.run([NVCC, *ARCH, "-shared", *objs, "-o", tmp], check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
