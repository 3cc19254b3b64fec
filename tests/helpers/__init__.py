"""Test-only GPU helpers (compiled on demand, never part of the product)."""
import ctypes
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_lib = None


def blocker():
    """ctypes handle with occupy_one_sm(ns, smem_bytes, started_ptr, stream)."""
    global _lib
    if _lib is None:
        os.makedirs(_BUILD, exist_ok=True)
        so = os.path.join(_BUILD, "libblocker.so")
        src = os.path.join(_HERE, "blocker.cu")
        if not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src):
            tmp = so + f".tmp{os.getpid()}"
            subprocess.check_call(["nvcc", "-gencode=arch=compute_103a,code=sm_103a", "-O2", "-Xcompiler", "-fPIC",
                                   "-shared", src, "-o", tmp])
            os.replace(tmp, so)
        lib = ctypes.CDLL(so)
        lib.occupy_one_sm.argtypes = [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.occupy_one_sm.restype = ctypes.c_int
        _lib = lib
    return _lib
