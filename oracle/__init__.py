"""fp64 CPU oracle for the quaternion cumulative-product scan.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library: the arithmetic lives in
``quat_oracle.c`` (plain C, fp64, sequential per lane), this module only
compiles it with gcc, widens inputs to fp64 and marshals arrays through ctypes.

What it computes follows burn-mamba ``mamba3/quat_scan/backward.rs``, module
documentation, section "Gradient math":

* :func:`fwd` -- the scan ``cum[t] = q_t (x) cum[t-1]`` with ``cum[-1] = init``;
* :func:`bwd` -- the literal reverse recurrence
  ``G[t] = d_cum[t] + conj(q_{t+1}) (x) G[t+1]``, then
  ``d_q[t] = G[t] (x) conj(cum[t-1])`` and ``d_init = conj(q_0) (x) G[0]``
  (the per-factor VJP rule applied to every step);
* :func:`bwd_closed_form` -- the page's unit-quaternion closed form
  ``S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s]``, ``G[t] = P_t (x) S[t]``,
  ``d_init = S[0]`` (used only to pin :func:`bwd` against the page);
* :func:`hamilton`, :func:`conj` -- the quaternion product and conjugate.

Pins (tests marked ``not gpu``): the Hamilton multiplication table and a
library rotation composition, closed forms for commuting single-axis inputs
against numpy's complex ``cumprod``, norm preservation, linearity in ``init``,
exact-rational brute force on tiny inputs, central finite differences and an
adjoint dot test for the backward, equality with the closed form for unit
quaternions, the closed form generalised to non-unit quaternions
(``G[t] = P_t (x) S[t] / |P_t|^2``, ``d_init = S[0]``), and the reverse-cumsum
special case for identity ``q``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "quat_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``quat_oracle.c`` into ``liboracle.so`` (gcc, fp64, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-pthread",
                   "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_hamilton.argtypes = [dp, dp, dp]
        lib.oracle_hamilton.restype = None
        lib.oracle_conj.argtypes = [dp, dp]
        lib.oracle_conj.restype = None
        lib.oracle_fwd.argtypes = [dp, dp, dp, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_fwd.restype = ctypes.c_int
        for name in ("oracle_bwd", "oracle_bwd_closed_form"):
            fn = getattr(lib, name)
            fn.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, ctypes.c_int]
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(q: np.ndarray, init: np.ndarray):
    if q.ndim != 5 or q.shape[-1] != 4:
        raise ValueError(f"q must be [B,S,H,J,4], got {q.shape}")
    B, S, H, J, _ = q.shape
    if init.shape != (B, H, J, 4):
        raise ValueError(f"init must be [B,H,J,4]={B, H, J, 4}, got {init.shape}")
    return B, S, H, J


def hamilton(a, b) -> np.ndarray:
    """a (x) b for single quaternions [w,x,y,z] (fp64)."""
    a, b = _f64(a), _f64(b)
    out = np.empty(4, np.float64)
    _load().oracle_hamilton(_ptr(a), _ptr(b), _ptr(out))
    return out


def conj(a) -> np.ndarray:
    a = _f64(a)
    out = np.empty(4, np.float64)
    _load().oracle_conj(_ptr(a), _ptr(out))
    return out


def fwd(q, init, nthreads: int = 0) -> np.ndarray:
    """cum [B,S,H,J,4] in fp64; inputs of any float dtype are widened to fp64."""
    q, init = _f64(q), _f64(init)
    B, S, H, J = _dims(q, init)
    cum = np.empty_like(q)
    rc = _load().oracle_fwd(_ptr(q), _ptr(init), _ptr(cum), B, S, H, J, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed ({rc})")
    return cum


def _bwd(name, q, init, d_cum, nthreads):
    q, init, d_cum = _f64(q), _f64(init), _f64(d_cum)
    B, S, H, J = _dims(q, init)
    if d_cum.shape != q.shape:
        raise ValueError("d_cum must have the shape of q")
    d_q = np.empty_like(q)
    d_init = np.empty_like(init)
    rc = getattr(_load(), name)(_ptr(q), _ptr(init), _ptr(d_cum), _ptr(d_q),
                                _ptr(d_init), B, S, H, J, nthreads)
    if rc != 0:
        raise RuntimeError(f"{name} failed ({rc})")
    return d_q, d_init


def bwd(q, init, d_cum, nthreads: int = 0):
    """(d_q, d_init) by the literal reverse recurrence, fp64."""
    return _bwd("oracle_bwd", q, init, d_cum, nthreads)


def bwd_closed_form(q, init, d_cum, nthreads: int = 0):
    """(d_q, d_init) by the page's unit-quaternion closed form, fp64."""
    return _bwd("oracle_bwd_closed_form", q, init, d_cum, nthreads)
