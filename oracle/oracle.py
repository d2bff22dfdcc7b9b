"""ctypes wrapper over the float64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg use this module; the CUDA library never does, and nothing here
touches a GPU.  Inputs are float64 numpy arrays shaped [B, H, N, d] (callers upcast
the exact bf16 values they also hand to the GPU).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test build)."""

    def __init__(self, path: str | None = None):
        if path is None:
            if _build.needs_build():
                _build.build()
            path = _build.OUT
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                   ctypes.c_long, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _lp, ctypes.c_long, _dp, _dp,
                                        ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_fwd_rows.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                      ctypes.c_long, ctypes.c_long, ctypes.c_double, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_long,
                                   ctypes.c_long, ctypes.c_long, ctypes.c_int, ctypes.c_double,
                                   ctypes.c_int]
        lib.oracle_bwd.restype = ctypes.c_int
        lib.oracle_bwd_rows.argtypes = [_dp, _dp, _dp, _dp, _lp, ctypes.c_long, _dp, _dp, _dp,
                                        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_int]
        lib.oracle_bwd_rows.restype = ctypes.c_int
        self.lib = lib

    @staticmethod
    def _f64(x):
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        if a.ndim != 4:
            raise ValueError("expected a [B, H, N, d] array")
        return a

    @staticmethod
    def _ptr(a):
        return a.ctypes.data_as(_dp)

    def fwd(self, q, k, v, causal=False, scale=None, nthreads=None):
        """Return (O [B,H,N,d], L [B,H,N]) in float64."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        B, H, N, d = q.shape
        if k.shape != q.shape or v.shape != q.shape:
            raise ValueError("q, k, v must share one shape")
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        o = np.empty_like(q)
        lse = np.empty((B, H, N), dtype=np.float64)
        rc = self.lib.oracle_fwd(self._ptr(q), self._ptr(k), self._ptr(v), self._ptr(o),
                                 self._ptr(lse), B * H, N, d, int(bool(causal)), scale,
                                 nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_fwd failed ({rc})")
        return o, lse

    def decode(self, q, k, v, scale=None, nthreads=None):
        """Decode shapes: q [B,H,Nq,d] against k, v [B,H,Nk,d], no mask.
        Return (O [B,H,Nq,d], L [B,H,Nq]) in float64."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        B, H, Nq, d = q.shape
        if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
            raise ValueError("k and v must be [B, H, Nk, d] with q's B, H and d")
        Nk = k.shape[2]
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        o = np.empty_like(q)
        lse = np.empty((B, H, Nq), dtype=np.float64)
        rc = self.lib.oracle_decode(self._ptr(q), self._ptr(k), self._ptr(v), self._ptr(o),
                                    self._ptr(lse), B * H, Nq, Nk, d, scale,
                                    nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_decode failed ({rc})")
        return o, lse

    def fwd_rows(self, q, k, v, rows, causal=False, scale=None, nthreads=None):
        """O and L for the given query rows of every head: [B,H,R,d], [B,H,R]."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        B, H, N, d = q.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.dtype("l"))
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        R = rows.shape[0]
        o = np.empty((B, H, R, d), dtype=np.float64)
        lse = np.empty((B, H, R), dtype=np.float64)
        rc = self.lib.oracle_fwd_rows(self._ptr(q), self._ptr(k), self._ptr(v),
                                      rows.ctypes.data_as(_lp), R, self._ptr(o),
                                      self._ptr(lse), B * H, N, d, int(bool(causal)), scale,
                                      nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_fwd_rows failed ({rc})")
        return o, lse

    def bwd(self, q, k, v, do, causal=False, scale=None, nthreads=None):
        """Return (dQ, dK, dV), each [B,H,N,d] float64."""
        q, k, v, do = self._f64(q), self._f64(k), self._f64(v), self._f64(do)
        B, H, N, d = q.shape
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        rc = self.lib.oracle_bwd(self._ptr(q), self._ptr(k), self._ptr(v), self._ptr(do),
                                 self._ptr(dq), self._ptr(dk), self._ptr(dv), B * H, N, d,
                                 int(bool(causal)), scale, nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_bwd failed ({rc})")
        return dq, dk, dv

    def bwd_rows(self, q, k, v, do, rows, causal=False, scale=None, nthreads=None):
        """Backward restricted to query rows `rows`: dQ of those rows [B,H,R,d] and
        their contributions to dK, dV [B,H,N,d]."""
        q, k, v, do = self._f64(q), self._f64(k), self._f64(v), self._f64(do)
        B, H, N, d = q.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.dtype("l"))
        scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
        R = rows.shape[0]
        dq = np.empty((B, H, R, d), dtype=np.float64)
        dk, dv = np.empty_like(q), np.empty_like(q)
        rc = self.lib.oracle_bwd_rows(self._ptr(q), self._ptr(k), self._ptr(v), self._ptr(do),
                                      rows.ctypes.data_as(_lp), R, self._ptr(dq), self._ptr(dk),
                                      self._ptr(dv), B * H, N, d, int(bool(causal)), scale,
                                      nthreads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_bwd_rows failed ({rc})")
        return dq, dk, dv


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def fwd(*a, **kw):
    return default().fwd(*a, **kw)


def fwd_rows(*a, **kw):
    return default().fwd_rows(*a, **kw)


def bwd(*a, **kw):
    return default().bwd(*a, **kw)


def bwd_rows(*a, **kw):
    return default().bwd_rows(*a, **kw)
