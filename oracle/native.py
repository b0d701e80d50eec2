"""ctypes wrapper around gdr_oracle.c (oracle; test infrastructure only).

``build()`` compiles the C oracle with gcc into ``oracle/liboracle.so``;
``recurrence(...)`` runs the float64 token recurrence on [B, T, H, d] arrays
with OpenMP over (batch, head). See gdr_oracle.c for the passages followed.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile the C oracle (gcc, -O2, OpenMP). Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.gdr_oracle_recurrence.argtypes = (
            [ctypes.c_int] * 5 + [ctypes.c_uint, ctypes.c_double] + [dp] * 11 + [ctypes.c_int])
        lib.gdr_oracle_recurrence.restype = ctypes.c_int
        lib.gdr_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads():
    return _load().gdr_oracle_max_threads()


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _c64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def recurrence(q, k, v, g, beta=None, lam=None, b=None, w=None, h0=None,
               scale=1.0, flags=0, nthreads=0):
    """Float64 token recurrence over [B, T, H, d] arrays.

    Returns (o [B, T, H, d_v], hT [B, H, d_k, d_v]).
    """
    q, k, v, g, beta, lam, b, w, h0 = map(_c64, (q, k, v, g, beta, lam, b, w, h0))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = np.empty((B, T, H, dv))
    hT = np.empty((B, H, dk, dv))
    rc = _load().gdr_oracle_recurrence(
        B, T, H, dk, dv, flags, float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
        _ptr(beta), _ptr(lam), _ptr(b), _ptr(w), _ptr(h0), _ptr(o), _ptr(hT), int(nthreads))
    if rc != 0:
        raise ValueError("gdr_oracle_recurrence rejected its arguments (rc=%d)" % rc)
    return o, hT
