"""ctypes wrapper of O2, the streaming two-pass C oracle (``twopass.c``).

TEST INFRASTRUCTURE ONLY.  ``build()`` compiles ``twopass.c`` with gcc into
``oracle/_twopass.so`` (plain C, no CUDA, same result on x86_64 and aarch64).
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twopass.c")
_LIB = os.path.join(_HERE, "_twopass.so")
_lib = None


def build(force=False):
    """Compile the C oracle (fast: one small translation unit)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_twopass_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i64,
                                           ctypes.c_double, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int64), i64, i64, ctypes.c_int]
        lib.oracle_twopass_fwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def forward(q, k, v, scale, causal=False, rows=None, Nq=None, block=16, nthreads=None):
    """Two-pass forward.  q [BH..., R, d], k [BH..., Nk, d], v [BH..., Nk, dv].

    Leading axes are flattened to BH.  ``rows`` (length R) gives the query index
    of each given query row, with ``Nq`` the total query count (causal offset).
    Returns O [..., R, dv] and LSE [..., R] in fp64.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    lead = q.shape[:-2]
    R, d = q.shape[-2:]
    Nk, dv = k.shape[-2], v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    if rows is None:
        Nq = R
        rows_p = None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows.size == R and Nq is not None
        rows_p = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    o = np.empty(lead + (R, dv))
    lse = np.empty(lead + (R,))
    nthreads = nthreads or os.cpu_count() or 1
    dp = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
    rc = lib.oracle_twopass_fwd(dp(q), dp(k), dp(v), dp(o), dp(lse), BH, Nq, Nk, d, dv,
                                float(scale), int(bool(causal)), rows_p, R, block, nthreads)
    if rc != 0:
        raise ValueError("oracle_twopass_fwd failed with %d" % rc)
    return o, lse
