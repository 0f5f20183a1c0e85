"""CPU oracle for the tiled fp32 GEMM (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library's product path never does, and the CUDA
library shares no code with it.

* ``sgemm`` / ``sgemm_rows`` / ``sgemm_elements``: the plain definition of
  C = A*B (row-major, fp64 accumulation in increasing k, one rounding to
  fp32), from ``ref_gemm.c``; see that file's header for the passages it
  follows.  ``sgemm_general``: alpha*op(A)*op(B) + beta*C with leading
  dimensions and transposes, the same sum with one rounding.
* ``smem_rules``: the pages' padding rule, bank mapping, staged layout,
  stage selection and budget formula, plus a bank-conflict simulator.

The C source is compiled with gcc on first use (or by ``build()``) into
``oracle/_build/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import smem_rules  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_gemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmtoracle.so")
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
          "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle's C source into a shared library; returns its path."""
    if not force and os.path.exists(out) and \
            os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its calls."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        lib = ctypes.CDLL(path or build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_sgemm.argtypes = [p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_sgemm.restype = ctypes.c_int
        lib.oracle_sgemm_rows.argtypes = [p, p, p, p, i64, i64, i64, p, i64,
                                          ctypes.c_int]
        lib.oracle_sgemm_rows.restype = ctypes.c_int
        lib.oracle_sgemm_elements.argtypes = [p, p, p, p, i64, i64, i64, p, p,
                                              i64]
        lib.oracle_sgemm_elements.restype = ctypes.c_int
        lib.oracle_sgemm_general.argtypes = [p, i64, p, i64, p, i64, p, i64, i64, i64,
                                             ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int]
        lib.oracle_sgemm_general.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _f32(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle inputs must be float32")
    return np.ascontiguousarray(x)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dims(A, B):
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shape mismatch {A.shape} x {B.shape}")
    return A.shape[0], B.shape[1], A.shape[1]


def max_threads() -> int:
    return load().oracle_max_threads()


def sgemm(A, B, with_w: bool = False, threads: int = 0, lib=None):
    """C = A*B (float32) and, if asked, W = |A|*|B| (float64)."""
    A, B = _f32(A), _f32(B)
    M, N, K = _dims(A, B)
    C = np.empty((M, N), np.float32)
    W = np.empty((M, N), np.float64) if with_w else None
    rc = (lib or load()).oracle_sgemm(_ptr(A), _ptr(B), _ptr(C),
                                      _ptr(W) if with_w else None,
                                      M, N, K, threads)
    if rc:
        raise RuntimeError("oracle_sgemm failed")
    return (C, W) if with_w else C


def sgemm_rows(A, B, rows, with_w: bool = False, threads: int = 0, lib=None):
    """Rows `rows` of A*B: shape (len(rows), N)."""
    A, B = _f32(A), _f32(B)
    M, N, K = _dims(A, B)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    C = np.empty((rows.size, N), np.float32)
    W = np.empty((rows.size, N), np.float64) if with_w else None
    rc = (lib or load()).oracle_sgemm_rows(_ptr(A), _ptr(B), _ptr(C),
                                           _ptr(W) if with_w else None,
                                           M, N, K, _ptr(rows), rows.size,
                                           threads)
    if rc:
        raise RuntimeError("oracle_sgemm_rows failed")
    return (C, W) if with_w else C


def sgemm_elements(A, B, ii, jj, lib=None):
    """C[ii[t], jj[t]] and W[ii[t], jj[t]] for every t."""
    A, B = _f32(A), _f32(B)
    M, N, K = _dims(A, B)
    ii = np.ascontiguousarray(np.asarray(ii, dtype=np.int64))
    jj = np.ascontiguousarray(np.asarray(jj, dtype=np.int64))
    if ii.shape != jj.shape:
        raise ValueError("index arrays differ in shape")
    out = np.empty(ii.size, np.float32)
    w = np.empty(ii.size, np.float64)
    rc = (lib or load()).oracle_sgemm_elements(_ptr(A), _ptr(B), _ptr(out),
                                               _ptr(w), M, N, K, _ptr(ii),
                                               _ptr(jj), ii.size)
    if rc:
        raise RuntimeError("oracle_sgemm_elements failed")
    return out, w


def sgemm_general(A, B, C0, M, N, K, lda, ldb, ldc, alpha=1.0, beta=0.0,
                  trans_a=False, trans_b=False, with_w=False, threads: int = 0, lib=None):
    """alpha*op(A)*op(B) + beta*C on flat float32 buffers with leading
    dimensions (see oracle_sgemm_general); returns the new C buffer (and W,
    M x N, if asked).  C0 is copied, never modified."""
    A = np.ascontiguousarray(np.asarray(A, np.float32).reshape(-1))
    B = np.ascontiguousarray(np.asarray(B, np.float32).reshape(-1))
    C = np.array(np.asarray(C0, np.float32).reshape(-1), copy=True)
    W = np.empty((M, N), np.float64) if with_w else None
    rc = (lib or load()).oracle_sgemm_general(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc,
                                              _ptr(W) if with_w else None, M, N, K,
                                              float(alpha), float(beta), int(trans_a),
                                              int(trans_b), threads)
    if rc:
        raise RuntimeError("oracle_sgemm_general failed")
    return (C, W) if with_w else C
