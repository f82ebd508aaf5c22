"""fp64 CPU oracle for topology-biased graph attention (ctypes driver for gt_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline leg may import this module; the library itself never does.  It
shares no code with the CUDA path.  The C source states the definitions it
follows (MegaGraph abstract: score matrix plus topology-aware bias; Fig. 4: the
bias column slice per KV block; Graphormer-style SPD buckets).

All floating-point work is done in fp64 on inputs upcast from whatever precision
they were generated in.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gt_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgt_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gt_oracle.c with gcc into oracle/_build/libgt_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_source(src_path: str, out_path: str) -> str:
    """Compile a copy of the oracle source (tests compile planted-mistake copies)."""
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", out_path, src_path, "-lm"])
    return out_path


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.gto_spd.argtypes = [i32, P, P, i32, P, i64, i32]
    lib.gto_spd.restype = ctypes.c_int
    lib.gto_attn_fwd_rows.argtypes = [i32, i32, i32, P, P, P, P, i64, P, i32, f64,
                                      P, i32, P, P, i32]
    lib.gto_attn_fwd_rows.restype = ctypes.c_int
    lib.gto_attn_bwd_delta.argtypes = [i32, i32, i32, P, P, P]
    lib.gto_attn_bwd_delta.restype = ctypes.c_int
    lib.gto_attn_bwd.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, i64, P, i32, f64,
                                 P, i32, P, P, P, i32, P, P, i32]
    lib.gto_attn_bwd.restype = ctypes.c_int
    return lib


def use_library(path: str | None) -> None:
    """Point this module at another compiled copy (None: the default build)."""
    global _lib
    with _lock:
        _lib = None if path is None else _bind(ctypes.CDLL(path))


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def spd(n: int, indptr, indices, D: int, nthreads: int | None = None) -> np.ndarray:
    """Clipped shortest-path buckets, int8 [n][n]: min(dist, D), D+1 if unreachable."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int64)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    out = np.empty((n, n), dtype=np.int8)
    rc = lib.gto_spd(n, _ptr(indptr), _ptr(indices), D, _ptr(out), n, nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"gto_spd rejected its arguments (rc={rc})")
    return out


def _rows(n, rows):
    if rows is None:
        return np.arange(n, dtype=np.int32)
    return np.ascontiguousarray(rows, dtype=np.int32)


def attn_fwd(q, k, v, spd_mat, T, scale: float | None = None, rows=None,
             nthreads: int | None = None):
    """Forward for `rows` (default: all).  Returns o [len(rows)][h][d], lse [h][len(rows)]."""
    lib = _load()
    q, k, v, T = _f64(q), _f64(k), _f64(v), _f64(T)
    n, h, d = q.shape
    spd_mat = np.ascontiguousarray(spd_mat, dtype=np.int8)
    nb = T.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r = _rows(n, rows)
    o = np.empty((r.shape[0], h, d), dtype=np.float64)
    lse = np.empty((h, r.shape[0]), dtype=np.float64)
    rc = lib.gto_attn_fwd_rows(n, h, d, _ptr(q), _ptr(k), _ptr(v), _ptr(spd_mat), spd_mat.shape[1],
                               _ptr(T), nb, float(scale), _ptr(r), r.shape[0], _ptr(o), _ptr(lse),
                               nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"gto_attn_fwd_rows rejected its arguments (rc={rc})")
    return o, lse


def bwd_delta(o, dO) -> np.ndarray:
    """D [h][n] with D_i = <dO_i, o_i> per head."""
    lib = _load()
    o, dO = _f64(o), _f64(dO)
    n, h, d = o.shape
    Dv = np.empty((h, n), dtype=np.float64)
    lib.gto_attn_bwd_delta(n, h, d, _ptr(o), _ptr(dO), _ptr(Dv))
    return Dv


def attn_bwd(q, k, v, dO, spd_mat, T, lse, Dv, scale: float | None = None,
             rows=None, cols=None, want_dq=True, want_dT=True, want_dkdv=True,
             nthreads: int | None = None):
    """Backward given the full-row lse [h][n] and D [h][n].

    dq is returned for `rows` (default all), dk/dv for `cols` (default all), and
    dT sums over `rows` (pass all rows for the full table gradient).
    """
    lib = _load()
    q, k, v, dO, T, lse, Dv = (_f64(a) for a in (q, k, v, dO, T, lse, Dv))
    n, h, d = q.shape
    nb = T.shape[1]
    spd_mat = np.ascontiguousarray(spd_mat, dtype=np.int8)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    r = _rows(n, rows)
    c = _rows(n, cols) if want_dkdv else np.zeros(0, dtype=np.int32)
    dq = np.empty((r.shape[0], h, d)) if want_dq else None
    dT = np.empty((h, nb)) if want_dT else None
    dk = np.empty((c.shape[0], h, d)) if want_dkdv else None
    dv = np.empty((c.shape[0], h, d)) if want_dkdv else None
    rc = lib.gto_attn_bwd(n, h, d, _ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(Dv),
                          _ptr(spd_mat), spd_mat.shape[1], _ptr(T), nb, float(scale),
                          _ptr(r), r.shape[0] if (want_dq or want_dT) else 0, _ptr(dq), _ptr(dT),
                          _ptr(c), c.shape[0], _ptr(dk), _ptr(dv), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"gto_attn_bwd failed (rc={rc})")
    return dict(dq=dq, dk=dk, dv=dv, dT=dT)


def attn_fwd_bwd(q, k, v, dO, spd_mat, T, scale: float | None = None, nthreads: int | None = None):
    """Full forward and backward over all rows and columns (small n)."""
    o, lse = attn_fwd(q, k, v, spd_mat, T, scale, nthreads=nthreads)
    Dv = bwd_delta(o, dO)
    g = attn_bwd(q, k, v, dO, spd_mat, T, lse, Dv, scale, nthreads=nthreads)
    return dict(o=o, lse=lse, D=Dv, **g)
