"""Oracle for tree/DAG-packed attention: plain, slow, fp64, on the CPU.

TEST INFRASTRUCTURE ONLY.  The library never imports, links or runs anything in this
package.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
use it.  It shares no code with the CUDA path: the DAG semantics are in ``oracle.dag``
(Python, from the definitions), the attention arithmetic in ``attn_oracle.c`` (plain C,
fp64, POSIX threads), compiled here with gcc.

Pins (the tests in ``tests/test_oracle_*.py``) tie it to what the pages fix rather than to
itself: packed = per-trajectory causal attention (a library routine) on expanded trees,
gradients at shared rows = the sum over trajectories, zero-length mounts change nothing,
closed forms at Q = 0, finite differences of the backward, the Eq. 2 worked example, the
Eq. 5 compact-row count and the Eq. 21-22 visible-pair count.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import dag  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C part of the oracle (gcc, -O2, no machine-specific flags)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-shared", "-fPIC",
                               "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_forward.argtypes = [i64, i32, i32, i32, dbl, vp, vp, vp, i64, vp, vp, vp, vp,
                                       vp, vp, i32]
        lib.oracle_forward.restype = i32
        lib.oracle_backward.argtypes = [i64, i32, i32, i32, dbl, vp, vp, vp, vp, i64, vp, vp, vp,
                                        vp, vp, vp, vp, vp, vp, vp, i32]
        lib.oracle_backward.restype = i32
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


class Result:
    """Oracle outputs for a set of listed query rows (all fp64)."""

    def __init__(self, rows):
        self.rows = rows
        self.o = self.lse = self.delta = self.dq = self.dk = self.dv = None
        self.threads = 0


def forward(branches, mounts, q, k, v, scale, rows=None, intervals=None, n_threads=0,
            view="mounted") -> Result:
    """O and lse (natural log) of the listed rows (default: all rows); ``view`` selects the
    visibility (see ``dag.VIEWS``)."""
    N, Hq, D = q.shape
    Hkv = k.shape[1]
    if intervals is None:
        intervals = dag.visible_intervals(branches, mounts, rows) if view == "mounted" else \
            dag.visible_intervals(branches, mounts, rows, view=view)
    rws, ptr, lo, hi = (_c(x, np.int64) for x in intervals)
    n = len(rws)
    res = Result(rws)
    res.o = np.zeros((n, Hq, D), dtype=np.float64)
    res.lse = np.zeros((n, Hq), dtype=np.float64)
    q, k, v = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    res.threads = _load().oracle_forward(N, Hq, Hkv, D, float(scale), _p(q), _p(k), _p(v), n,
                                         _p(rws), _p(ptr), _p(lo), _p(hi), _p(res.o),
                                         _p(res.lse), int(n_threads))
    res.intervals = (rws, ptr, lo, hi)
    return res


def backward(branches, mounts, q, k, v, do, scale, fwd: Result, with_dkdv=True,
             n_threads=0) -> Result:
    """delta, dQ of the listed rows and (optionally) dK, dV [N, Hkv, D] summed over the
    listed rows' contributions.  ``fwd`` is the oracle forward of the same rows."""
    N, Hq, D = q.shape
    Hkv = k.shape[1]
    rws, ptr, lo, hi = fwd.intervals
    n = len(rws)
    res = Result(rws)
    res.o, res.lse, res.intervals = fwd.o, fwd.lse, fwd.intervals
    res.delta = np.zeros((n, Hq), dtype=np.float64)
    res.dq = np.zeros((n, Hq, D), dtype=np.float64)
    if with_dkdv:
        res.dk = np.zeros((N, Hkv, D), dtype=np.float64)
        res.dv = np.zeros((N, Hkv, D), dtype=np.float64)
    q, k, v, do = (_c(x, np.uint16) for x in (q, k, v, do))
    o_in, lse_in = _c(fwd.o, np.float64), _c(fwd.lse, np.float64)
    res.threads = _load().oracle_backward(N, Hq, Hkv, D, float(scale), _p(q), _p(k), _p(v),
                                          _p(do), n, _p(rws), _p(ptr), _p(lo), _p(hi),
                                          _p(o_in), _p(lse_in), _p(res.delta), _p(res.dq),
                                          _p(res.dk), _p(res.dv), int(n_threads))
    return res


def run(branches, mounts, q, k, v, do, scale, rows=None, with_dkdv=True, n_threads=0,
        view="mounted") -> Result:
    """Forward then backward for the listed rows (default: all rows)."""
    f = forward(branches, mounts, q, k, v, scale, rows=rows, n_threads=n_threads, view=view)
    return backward(branches, mounts, q, k, v, do, scale, f, with_dkdv=with_dkdv,
                    n_threads=n_threads)
