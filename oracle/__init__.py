"""Parallax attention oracle (fp64, CPU) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it.

The arithmetic lives in ``plx_oracle.c`` (plain loops, fp64, one definition per
line, see its header for the definition and its sources).  This module only
compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "plx_oracle.c")
_LIB = os.path.join(_HERE, "libplx_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.plx_oracle_fwd.argtypes = [dp, dp, dp, dp, i, i, i, i, i, dp, dp, dp, i]
        lib.plx_oracle_fwd_rows.argtypes = [dp, dp, dp, dp, i, i, i, i,
                                            ctypes.POINTER(ctypes.c_int64), i, dp, dp, dp, i]
        lib.plx_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, i, i, i, i,
                                       ctypes.POINTER(ctypes.c_int32), i, dp, dp, dp, dp, i]
        lib.plx_oracle_fwd_probe.argtypes = [dp, dp, dp, dp, i, i, i, i, dp, dp, i]
        lib.plx_oracle_fwd_probe_rows.argtypes = [dp, dp, dp, dp, i, i, i, i,
                                                  ctypes.POINTER(ctypes.c_int64), i, dp, dp, i]
        for f in (lib.plx_oracle_fwd, lib.plx_oracle_fwd_rows, lib.plx_oracle_bwd, lib.plx_oracle_fwd_probe,
                  lib.plx_oracle_fwd_probe_rows):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def forward(q, k, v, P, nthreads: int | None = None):
    """Full forward.  q,k,v: [B,H,T,d]; P: [H,d,d] or per-query [B,H,T,d,d].

    Returns (out [B,H,T,d], lse [B,H,T], mu_k [B,H,T,d]) in float64.
    """
    q, k, v, P = _f64(q), _f64(k), _f64(v), _f64(P)
    B, H, T, d = q.shape
    per_query = 1 if P.ndim == 5 else 0
    if per_query:
        assert P.shape == (B, H, T, d, d)
    else:
        assert P.shape == (H, d, d)
    out = np.empty((B, H, T, d))
    lse = np.empty((B, H, T))
    mu_k = np.empty((B, H, T, d))
    rc = _load().plx_oracle_fwd(_p(q), _p(k), _p(v), _p(P), per_query, B, H, T, d,
                                _p(out), _p(lse), _p(mu_k), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"plx_oracle_fwd failed ({rc})")
    return out, lse, mu_k


def forward_rows(q, k, v, P, rows, nthreads: int | None = None):
    """Forward at selected (b, h, t) rows: returns (out [n,d], lse [n], mu_k [n,d])."""
    q, k, v, P = _f64(q), _f64(k), _f64(v), _f64(P)
    B, H, T, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, d))
    lse = np.empty((n,))
    mu_k = np.empty((n, d))
    rc = _load().plx_oracle_fwd_rows(_p(q), _p(k), _p(v), _p(P), B, H, T, d,
                                     rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                                     _p(out), _p(lse), _p(mu_k), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"plx_oracle_fwd_rows failed ({rc})")
    return out, lse, mu_k


def forward_probe(q, k, v, rho, nthreads: int | None = None):
    """One-pass form with a given probe: o = o^SA - Sigma_KV rho.

    q, k, v, rho: [B,H,T,d].  Returns (out [B,H,T,d], lse [B,H,T]) in float64.
    """
    q, k, v, rho = _f64(q), _f64(k), _f64(v), _f64(rho)
    B, H, T, d = q.shape
    out = np.empty((B, H, T, d))
    lse = np.empty((B, H, T))
    rc = _load().plx_oracle_fwd_probe(_p(q), _p(k), _p(v), _p(rho), B, H, T, d, _p(out), _p(lse),
                                      nthreads or default_threads())
    if rc:
        raise RuntimeError(f"plx_oracle_fwd_probe failed ({rc})")
    return out, lse


def forward_probe_rows(q, k, v, rho, rows, nthreads: int | None = None):
    """The given-probe form at selected (b, h, t) rows: returns (out [n,d], lse [n])."""
    q, k, v, rho = _f64(q), _f64(k), _f64(v), _f64(rho)
    B, H, T, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = rows.shape[0]
    out = np.empty((n, d))
    lse = np.empty((n,))
    rc = _load().plx_oracle_fwd_probe_rows(_p(q), _p(k), _p(v), _p(rho), B, H, T, d,
                                           rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                                           _p(out), _p(lse), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"plx_oracle_fwd_probe_rows failed ({rc})")
    return out, lse


def backward(q, k, v, P, dout, heads=None, nthreads: int | None = None):
    """Gradients (dq, dk, dv, dP) of sum(dout * out).

    ``heads``: optional list of (b, h) pairs; only those heads' dq/dk/dv are
    computed (others are zero) and dP[h] sums over the listed heads only.
    """
    q, k, v, P, dout = _f64(q), _f64(k), _f64(v), _f64(P), _f64(dout)
    B, H, T, d = q.shape
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    hs = np.ascontiguousarray(np.asarray(heads, dtype=np.int32).reshape(-1, 2))
    dq = np.zeros((B, H, T, d))
    dk = np.zeros((B, H, T, d))
    dv = np.zeros((B, H, T, d))
    dP = np.zeros((H, d, d))
    rc = _load().plx_oracle_bwd(_p(q), _p(k), _p(v), _p(P), _p(dout), B, H, T, d,
                                hs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), hs.shape[0],
                                _p(dq), _p(dk), _p(dv), _p(dP), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"plx_oracle_bwd failed ({rc})")
    return dq, dk, dv, dP
