"""cudaMemcpy through ctypes, for tests that read lane-owned buffers.

The CUDA runtime is already loaded by torch; dlopen of its soname returns
that copy.  cudaMemcpyDefault lets unified addressing pick the direction.
"""
import ctypes
import glob
import os

import torch  # noqa: F401  (loads the CUDA runtime)

_lib = None


def _cudart():
    global _lib
    if _lib is None:
        names = ["libcudart.so.13", "libcudart.so"]
        import torch as _t
        names += glob.glob(os.path.join(os.path.dirname(_t.__file__), "..", "nvidia", "*", "lib",
                                        "libcudart.so*"))
        names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
        for n in names:
            try:
                _lib = ctypes.CDLL(n)
                break
            except OSError:
                continue
        if _lib is None:
            raise RuntimeError("no CUDA runtime library found")
        _lib.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        _lib.cudaMemcpy.restype = ctypes.c_int
    return _lib


def memcpy(dst: int, src: int, nbytes: int) -> None:
    rc = _cudart().cudaMemcpy(dst, src, nbytes, 4)   # cudaMemcpyDefault
    if rc != 0:
        raise RuntimeError(f"cudaMemcpy failed with {rc}")
