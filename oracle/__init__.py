"""CPU fp64 oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library.

The arithmetic lives in ``gdn_oracle.c`` (plain token-by-token recurrence in
fp64, compiled with gcc + OpenMP on first use).  This module only converts
arrays to fp64 numpy and calls it.

Pins (tests/test_oracle_*.py): brute-force dense products of the per-token
factors, closed forms (alpha=1/beta=0 identity state, single token, exact
recall with orthonormal keys, memoryless alpha=0), the affine start-state
identity, continuation, central finite differences of the backward, Euler
homogeneity identities, a hand-worked example under tests/golden/, and the
window bound.  No function here is left without a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (plain C, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.gdn_oracle_fwd.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, P, P, P, P, P, P, P, ctypes.c_int,
                                           ctypes.c_double, P, P, ctypes.c_int]
            lib.gdn_oracle_bwd.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, P, P, P, P, P, P, P, P, P, ctypes.c_int,
                                           ctypes.c_double, P, P, P, P, P, P, ctypes.c_int]
            lib.gdn_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):          # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _pack(q, k, v, g, beta, cu_seqlens):
    """Flatten [B, T, H, D] to the packed [B*T, H, D] layout + int64 offsets."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
        assert B == 1
    return (q.reshape(B * T, H, Dk), k.reshape(B * T, H, Dk), v.reshape(B * T, H, Dv),
            g.reshape(B * T, H), beta.reshape(B * T, H), cu, B, T, H, Dk, Dv)


def fwd(q, k, v, g, beta, S0=None, cu_seqlens=None, *, scale=1.0, l2norm=False, nthreads=None):
    """Token recurrence.  Returns (o [B,T,H,Dv], S_T [N,H,Dv,Dk]) as fp64 numpy."""
    lib = _load()
    q, k, v, g, beta, cu, B, T, H, Dk, Dv = _pack(q, k, v, g, beta, cu_seqlens)
    N = len(cu) - 1
    S0 = _f64(S0)
    o = np.zeros((B * T, H, Dv))
    ST = np.zeros((N, H, Dv, Dk))
    nt = nthreads or os.cpu_count() or 1
    lib.gdn_oracle_fwd(B * T, H, Dk, Dv, N, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                       _ptr(S0), int(bool(l2norm)), float(scale), _ptr(o), _ptr(ST), int(nt))
    return o.reshape(B, T, H, Dv), ST


def bwd(q, k, v, g, beta, dO, S0=None, dST=None, cu_seqlens=None, *, scale=1.0, l2norm=False,
        nthreads=None):
    """Back-propagation through the token loop.

    Returns dict(dq, dk, dv [B,T,H,D], dg, dbeta [B,T,H], dS0 [N,H,Dv,Dk]) fp64.
    """
    lib = _load()
    q, k, v, g, beta, cu, B, T, H, Dk, Dv = _pack(q, k, v, g, beta, cu_seqlens)
    N = len(cu) - 1
    dO = _f64(dO).reshape(B * T, H, Dv)
    S0, dST = _f64(S0), _f64(dST)
    dq = np.zeros((B * T, H, Dk)); dk = np.zeros((B * T, H, Dk)); dv = np.zeros((B * T, H, Dv))
    dg = np.zeros((B * T, H)); db = np.zeros((B * T, H)); dS0 = np.zeros((N, H, Dv, Dk))
    nt = nthreads or os.cpu_count() or 1
    lib.gdn_oracle_bwd(B * T, H, Dk, Dv, N, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                       _ptr(S0), _ptr(dO), _ptr(dST), int(bool(l2norm)), float(scale),
                       _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db), _ptr(dS0), int(nt))
    return dict(dq=dq.reshape(B, T, H, Dk), dk=dk.reshape(B, T, H, Dk), dv=dv.reshape(B, T, H, Dv),
                dg=dg.reshape(B, T, H), dbeta=db.reshape(B, T, H), dS0=dS0)
