"""CPU oracle for the tiled fp32 GEMM (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library's product path never does, and the CUDA
library shares no code with it.

* ``sgemm`` / ``sgemm_rows`` / ``sgemm_elements``: the plain definition of
  C = A*B (row-major, fp64 accumulation in increasing k, one rounding to
  fp32), from ``ref_gemm.c``; see that file's header for the passages it
  follows.  ``sgemm_general``: alpha*op(A)*op(B) + beta*C with leading
  dimensions and transposes, the same sum with one rounding.
* ``gemm_mixed_general``: the same general form on 16-bit inputs (fp16 or
  bf16 patterns, decoded from the formats' definitions), fp32 result.
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
        lib.oracle_sgemm_general_bias.argtypes = [p, i64, p, i64, p, p, i64, p, i64, i64,
                                                  i64, ctypes.c_double, ctypes.c_double,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_sgemm_general_bias.restype = ctypes.c_int
        lib.oracle_gemm_mixed_general.argtypes = [ctypes.c_int, p, i64, p, i64, p, i64, p, i64,
                                                  i64, i64, ctypes.c_double, ctypes.c_double,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_gemm_mixed_general.restype = ctypes.c_int
        lib.oracle_gemm_mixed_general_bias.argtypes = [ctypes.c_int, p, i64, p, i64, p, p, i64,
                                                       p, i64, i64, i64, ctypes.c_double,
                                                       ctypes.c_double, ctypes.c_int,
                                                       ctypes.c_int, ctypes.c_int]
        lib.oracle_gemm_mixed_general_bias.restype = ctypes.c_int
        lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = ctypes.c_double
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
                  trans_a=False, trans_b=False, with_w=False, threads: int = 0, lib=None,
                  bias=None):
    """alpha*op(A)*op(B) + beta*C (+ bias[j] on every row) on flat float32
    buffers with leading dimensions (see oracle_sgemm_general_bias); returns
    the new C buffer (and W, M x N, if asked).  C0 is copied, never
    modified."""
    A = np.ascontiguousarray(np.asarray(A, np.float32).reshape(-1))
    B = np.ascontiguousarray(np.asarray(B, np.float32).reshape(-1))
    C = np.array(np.asarray(C0, np.float32).reshape(-1), copy=True)
    W = np.empty((M, N), np.float64) if with_w else None
    if bias is not None:
        bias = np.ascontiguousarray(np.asarray(bias, np.float32).reshape(-1))
        if bias.size < N:
            raise ValueError("bias needs N values")
    rc = (lib or load()).oracle_sgemm_general_bias(
        _ptr(A), lda, _ptr(B), ldb, _ptr(bias) if bias is not None else None, _ptr(C), ldc,
        _ptr(W) if with_w else None, M, N, K, float(alpha), float(beta), int(trans_a),
        int(trans_b), threads)
    if rc:
        raise RuntimeError("oracle_sgemm_general_bias failed")
    return (C, W) if with_w else C


F16, BF16 = 1, 2  # dtype codes of oracle_gemm_mixed_general


def _u16(x) -> np.ndarray:
    """16-bit patterns as a flat uint16 array (accepts uint16/int16 numpy
    arrays or float16/bfloat16 torch tensors)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype).startswith("torch."):
        import torch
        x = x.detach().contiguous().view(torch.int16).numpy()
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype.kind in "iu" and x.dtype.itemsize > 2:
        if x.size and (x.min() < 0 or x.max() > 0xFFFF):
            raise ValueError("16-bit patterns lie in [0, 65535]")
        x = x.astype(np.uint16)
    if x.dtype not in (np.uint16, np.int16):
        raise TypeError("16-bit inputs must be 16-bit patterns")
    return np.ascontiguousarray(x.reshape(-1)).view(np.uint16)


def value16(dtype: int, patterns) -> np.ndarray:
    """The float64 value of each 16-bit pattern (oracle_f16_value /
    oracle_bf16_value, one call per element)."""
    lib = load()
    fn = lib.oracle_f16_value if dtype == F16 else lib.oracle_bf16_value
    pats = _u16(patterns)
    return np.array([fn(int(h)) for h in pats], dtype=np.float64)


def gemm_mixed_general(dtype, A, B, C0, M, N, K, lda, ldb, ldc, alpha=1.0, beta=0.0,
                       trans_a=False, trans_b=False, with_w=False, threads: int = 0,
                       lib=None, bias=None):
    """alpha*op(A)*op(B) + beta*C (+ bias[j] on every row) on flat 16-bit A
    and B (dtype F16 or BF16) and a flat float32 C; returns the new C buffer
    (and W, M x N, if asked).  C0 is copied, never modified."""
    A, B = _u16(A), _u16(B)
    C = np.array(np.asarray(C0, np.float32).reshape(-1), copy=True)
    W = np.empty((M, N), np.float64) if with_w else None
    if bias is not None:
        bias = np.ascontiguousarray(np.asarray(bias, np.float32).reshape(-1))
        if bias.size < N:
            raise ValueError("bias needs N values")
    rc = (lib or load()).oracle_gemm_mixed_general_bias(
        int(dtype), _ptr(A), lda, _ptr(B), ldb, _ptr(bias) if bias is not None else None,
        _ptr(C), ldc, _ptr(W) if with_w else None, M, N, K, float(alpha), float(beta),
        int(trans_a), int(trans_b), threads)
    if rc:
        raise RuntimeError("oracle_gemm_mixed_general_bias failed")
    return (C, W) if with_w else C
