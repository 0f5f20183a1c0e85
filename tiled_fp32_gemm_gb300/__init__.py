"""tiled_fp32_gemm_gb300 — fp32 GEMM for one GB300, C ABI plus a thin binding.

The compute lives in ``libmtsgemm.so`` (hand-written CUDA for sm_103a, built
by ``tiled_fp32_gemm_gb300.build``).  This module only marshals arguments:

* ``mt_sgemm``, ``mt_sgemm_ex``, ``mt_sgemm_general``, ``mt_sgemm_general_bias``,
  ``mt_sgemm_host``, ``mt_sgemm_host_async``,
  ``mt_sgemm_tf32x3_noalloc``,
  ``mt_sgemm_plan``, ``mt_sgemm_general_plan``, ``mt_gemm_mixed``,
  ``mt_gemm_mixed_general``, ``mt_gemm_mixed_general_bias``,
  ``mt_gemm_mixed_plan``,
  ``mt_smem_row_padding``, ``mt_smem_vector_row_padding``,
  ``mt_smem_layout_make``, ``mt_smem_layout_offset``, ``mt_check_device_status``
  (also under its earlier name ``mt_device_status``),
  ``mt_bounds_status``,
  ``mt_status_string``, ``mt_version`` — the C entry points under the same
  names, taking plain integers for pointers and streams;
* ``sgemm(a, b, out=None, **choices)`` — the same call on torch CUDA tensors
  (torch supplies device memory and the current stream; nothing else);
  ``gemm`` for the general form and ``gemm_mixed`` for 16-bit inputs.

There is no CPU fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading


MT_OK = 0
MT_ERR_INVALID_ARG = 1
MT_ERR_ALIAS = 2
MT_ERR_NO_DEVICE = 3
MT_ERR_UNSUPPORTED = 4
MT_ERR_SMEM_BUDGET = 5
MT_ERR_LAUNCH = 6
MT_ERR_TIMEOUT = 7
MT_ERR_CUDA = 8
MT_ERR_SCRATCH_LIMIT = 9
MT_NOALLOC_SCRATCH_BYTES = 32 << 20

MT_VARIANT_FFMA = 0
MT_VARIANT_TF32X3 = 1
MT_VARIANT_P18 = 2
MT_VARIANT_TC16 = 3
VARIANTS = {"ffma": MT_VARIANT_FFMA, "tf32x3": MT_VARIANT_TF32X3, "p18": MT_VARIANT_P18,
            "tc16": MT_VARIANT_TC16}
# mt_config.schedule: automatic, split tail, stream-K.
SCHEDULES = {"auto": 0, "split_tail": 1, "stream_k": 2}

MT_DTYPE_F16 = 1
MT_DTYPE_BF16 = 2

# mt_bounds_site: where the checked build found an access outside its buffer.
MT_SITE_A_LOAD, MT_SITE_B_LOAD, MT_SITE_A_SMEM, MT_SITE_B_SMEM = 1, 2, 3, 4
MT_SITE_FRAG, MT_SITE_C_STORE, MT_SITE_PARTIAL, MT_SITE_BIAS = 5, 6, 7, 8
MT_SITE_SLICE_SUM, MT_SITE_PREP_SRC, MT_SITE_PREP_DST, MT_SITE_P18 = 9, 10, 11, 12

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmtsgemm.so")
CHECKED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "checked",
                                "libmtsgemm_checked.so")


class mt_config(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("bm", ctypes.c_int), ("bn", ctypes.c_int),
                ("bk", ctypes.c_int), ("stages", ctypes.c_int), ("no_pad", ctypes.c_int),
                ("split_k", ctypes.c_int), ("fma", ctypes.c_int),
                ("fault_inject", ctypes.c_int), ("wm", ctypes.c_int), ("wn", ctypes.c_int),
                ("tm", ctypes.c_int), ("tn", ctypes.c_int), ("pack_a", ctypes.c_int),
                ("group_m", ctypes.c_int), ("schedule", ctypes.c_int)]


class mt_plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("bm", ctypes.c_int), ("bn", ctypes.c_int),
                ("bk", ctypes.c_int), ("stages", ctypes.c_int), ("pad_a", ctypes.c_int),
                ("pad_b", ctypes.c_int), ("threads", ctypes.c_int), ("vec_ab", ctypes.c_int),
                ("vec_c", ctypes.c_int), ("split_k", ctypes.c_int), ("fma", ctypes.c_int),
                ("wm", ctypes.c_int), ("wn", ctypes.c_int), ("tm", ctypes.c_int),
                ("tn", ctypes.c_int),
                ("grid", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("pack_a", ctypes.c_int),
                ("stream_k", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class mt_smem_layout(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int), ("columns", ctypes.c_int),
                ("row_padding", ctypes.c_int), ("stage_count", ctypes.c_int),
                ("row_stride", ctypes.c_int), ("stage_size", ctypes.c_int),
                ("size", ctypes.c_int), ("nbytes", ctypes.c_int64)]


class MtError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {mt_status_string(status)} (status {status})")


_P, _I64, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
# name -> (restype, argtypes): every function include/mt_sgemm.h declares.
SIGNATURES = {
    "mt_sgemm": (_I, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "mt_sgemm_ex": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, ctypes.POINTER(mt_config)]),
    "mt_sgemm_host": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, ctypes.POINTER(mt_config)]),
    "mt_sgemm_host_async": (_I, [_P, _P, _P, _I64, _I64, _I64, _P, ctypes.POINTER(mt_config)]),
    "mt_sgemm_tf32x3_noalloc": (_I, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "mt_sgemm_general": (_I, [_I, _I, _I64, _I64, _I64, ctypes.c_float, _P, _I64, _P, _I64,
                              ctypes.c_float, _P, _I64, _P, ctypes.POINTER(mt_config)]),
    "mt_sgemm_general_bias": (_I, [_I, _I, _I64, _I64, _I64, ctypes.c_float, _P, _I64, _P,
                                   _I64, ctypes.c_float, _P, _P, _I64, _P,
                                   ctypes.POINTER(mt_config)]),
    "mt_sgemm_plan": (_I, [_P, _P, _P, _I64, _I64, _I64, ctypes.POINTER(mt_config), _I64,
                           ctypes.POINTER(mt_plan)]),
    "mt_gemm_mixed": (_I, [_I, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mt_gemm_mixed_general": (_I, [_I, _I, _I, _I64, _I64, _I64, ctypes.c_float, _P, _I64,
                                   _P, _I64, ctypes.c_float, _P, _I64, _P,
                                   ctypes.POINTER(mt_config)]),
    "mt_gemm_mixed_general_bias": (_I, [_I, _I, _I, _I64, _I64, _I64, ctypes.c_float, _P,
                                        _I64, _P, _I64, ctypes.c_float, _P, _P, _I64, _P,
                                        ctypes.POINTER(mt_config)]),
    "mt_gemm_mixed_plan": (_I, [_I, _I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64,
                                ctypes.POINTER(mt_config), _I64, ctypes.POINTER(mt_plan)]),
    "mt_sgemm_general_plan": (_I, [_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64,
                                   ctypes.POINTER(mt_config), _I64, ctypes.POINTER(mt_plan)]),
    "mt_smem_row_padding": (_I, [_I, _I]),
    "mt_smem_vector_row_padding": (_I, [_I, _I]),
    "mt_smem_layout_make": (_I, [_I, _I, _I, _I, ctypes.POINTER(mt_smem_layout)]),
    "mt_smem_layout_offset": (_I64, [ctypes.POINTER(mt_smem_layout), _I, _I, _I]),
    "mt_check_device_status": (_I, [_P]),
    "mt_device_status": (_I, [_P]),
    "mt_bounds_status": (_I, [ctypes.POINTER(_I64), ctypes.POINTER(_I), ctypes.POINTER(_I64),
                              ctypes.POINTER(_I64)]),
    "mt_status_string": (ctypes.c_char_p, [_I]),
    "mt_version": (_I, []),
}

_lock = threading.Lock()
_lib = None
_checked = None


def _load(path: str, how: str):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           f"`python -m tiled_fp32_gemm_gb300.build{how}` (there is no CPU "
                           "fallback)")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                _lib = _load(LIB_PATH, "")
    return _lib


def checked_lib():
    """The bounds-checked build (libmtsgemm_checked.so, same entry points):
    its FFMA-path kernels skip and count any access outside their buffers;
    read the count with ``bounds_status(checked_lib())``."""
    global _checked
    if _checked is None:
        with _lock:
            if _checked is None:
                _checked = _load(CHECKED_LIB_PATH, " --checked")
    return _checked


def bounds_status(handle=None) -> dict:
    """mt_bounds_status of `handle` (default: the checked build) as a dict;
    raises MtError if the call fails (MT_ERR_UNSUPPORTED: a normal build)."""
    h = handle if handle is not None else checked_lib()
    count, site, offset, extent = ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64(), \
        ctypes.c_int64()
    st = h.mt_bounds_status(ctypes.byref(count), ctypes.byref(site), ctypes.byref(offset),
                            ctypes.byref(extent))
    if st != MT_OK:
        raise MtError(st, "mt_bounds_status")
    return {"count": count.value, "site": site.value, "offset": offset.value,
            "extent": extent.value}


def make_config(variant="ffma", bm=0, bn=0, bk=0, stages=0, no_pad=False, split_k=0,
                fma=0, fault_inject=0, wm=0, wn=0, tm=0, tn=0, pack_a=0,
                group_m=0, schedule=0) -> mt_config:
    c = mt_config()
    c.variant = VARIANTS[variant] if isinstance(variant, str) else int(variant)
    c.bm, c.bn, c.bk, c.stages = bm, bn, bk, stages
    c.no_pad = 1 if no_pad else 0
    c.split_k = split_k
    c.fma = fma
    c.fault_inject = fault_inject
    c.wm, c.wn = wm, wn
    c.tm, c.tn = tm, tn
    c.pack_a = pack_a
    c.group_m = group_m
    c.schedule = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    return c


# --- the C entry points, same names -----------------------------------------
def mt_sgemm(A: int, B: int, C: int, M: int, N: int, K: int, stream: int = 0) -> int:
    return lib().mt_sgemm(A, B, C, M, N, K, stream)


def mt_sgemm_ex(A: int, B: int, C: int, M: int, N: int, K: int, stream: int = 0,
                cfg: mt_config | None = None) -> int:
    return lib().mt_sgemm_ex(A, B, C, M, N, K, stream,
                             ctypes.byref(cfg) if cfg is not None else None)


def mt_sgemm_host(A: int, B: int, C: int, M: int, N: int, K: int, stream: int = 0,
                  cfg: mt_config | None = None) -> int:
    return lib().mt_sgemm_host(A, B, C, M, N, K, stream,
                               ctypes.byref(cfg) if cfg is not None else None)


def mt_sgemm_host_async(A: int, B: int, C: int, M: int, N: int, K: int, stream: int = 0,
                        cfg: mt_config | None = None) -> int:
    return lib().mt_sgemm_host_async(A, B, C, M, N, K, stream,
                                     ctypes.byref(cfg) if cfg is not None else None)


def mt_sgemm_general(trans_a: int, trans_b: int, M: int, N: int, K: int, alpha: float,
                     A: int, lda: int, B: int, ldb: int, beta: float, C: int, ldc: int,
                     stream: int = 0, cfg: mt_config | None = None) -> int:
    return lib().mt_sgemm_general(trans_a, trans_b, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                  ldc, stream, ctypes.byref(cfg) if cfg is not None else None)


def mt_sgemm_general_bias(trans_a: int, trans_b: int, M: int, N: int, K: int, alpha: float,
                          A: int, lda: int, B: int, ldb: int, beta: float, bias: int | None,
                          C: int, ldc: int, stream: int = 0,
                          cfg: mt_config | None = None) -> int:
    return lib().mt_sgemm_general_bias(trans_a, trans_b, M, N, K, alpha, A, lda, B, ldb, beta,
                                       bias, C, ldc, stream,
                                       ctypes.byref(cfg) if cfg is not None else None)


def mt_sgemm_tf32x3_noalloc(A: int, B: int, C: int, M: int, N: int, K: int,
                            stream: int = 0) -> int:
    """The 3xTF32 product with its scratch in the library's static device
    array: allocates nothing (see include/mt_sgemm.h for who needs that)."""
    return lib().mt_sgemm_tf32x3_noalloc(A, B, C, M, N, K, stream)


def mt_sgemm_plan(A: int, B: int, C: int, M: int, N: int, K: int,
                  cfg: mt_config | None = None, smem_limit_bytes: int = 0):
    out = mt_plan()
    st = lib().mt_sgemm_plan(A, B, C, M, N, K,
                             ctypes.byref(cfg) if cfg is not None else None,
                             smem_limit_bytes, ctypes.byref(out))
    return st, out


def mt_gemm_mixed(dtype: int, A: int, B: int, C: int, M: int, N: int, K: int,
                  stream: int = 0) -> int:
    return lib().mt_gemm_mixed(dtype, A, B, C, M, N, K, stream)


def mt_gemm_mixed_general(dtype: int, trans_a: int, trans_b: int, M: int, N: int, K: int,
                          alpha: float, A: int, lda: int, B: int, ldb: int, beta: float,
                          C: int, ldc: int, stream: int = 0,
                          cfg: mt_config | None = None) -> int:
    return lib().mt_gemm_mixed_general(dtype, trans_a, trans_b, M, N, K, alpha, A, lda, B,
                                       ldb, beta, C, ldc, stream,
                                       ctypes.byref(cfg) if cfg is not None else None)


def mt_gemm_mixed_general_bias(dtype: int, trans_a: int, trans_b: int, M: int, N: int, K: int,
                               alpha: float, A: int, lda: int, B: int, ldb: int, beta: float,
                               bias: int | None, C: int, ldc: int, stream: int = 0,
                               cfg: mt_config | None = None) -> int:
    return lib().mt_gemm_mixed_general_bias(dtype, trans_a, trans_b, M, N, K, alpha, A, lda,
                                            B, ldb, beta, bias, C, ldc, stream,
                                            ctypes.byref(cfg) if cfg is not None else None)


def mt_gemm_mixed_plan(dtype: int, trans_a: int, trans_b: int, M: int, N: int, K: int,
                       A: int | None, lda: int, B: int | None, ldb: int, C: int | None,
                       ldc: int, cfg: mt_config | None = None, smem_limit_bytes: int = 0):
    out = mt_plan()
    st = lib().mt_gemm_mixed_plan(dtype, trans_a, trans_b, M, N, K, A, lda, B, ldb, C, ldc,
                                  ctypes.byref(cfg) if cfg is not None else None,
                                  smem_limit_bytes, ctypes.byref(out))
    return st, out


def mt_sgemm_general_plan(trans_a: int, trans_b: int, M: int, N: int, K: int,
                          A: int | None, lda: int, B: int | None, ldb: int, C: int | None,
                          ldc: int, cfg: mt_config | None = None, smem_limit_bytes: int = 0):
    out = mt_plan()
    st = lib().mt_sgemm_general_plan(trans_a, trans_b, M, N, K, A, lda, B, ldb, C, ldc,
                                     ctypes.byref(cfg) if cfg is not None else None,
                                     smem_limit_bytes, ctypes.byref(out))
    return st, out


def mt_smem_row_padding(columns: int, simultaneous_rows: int) -> int:
    return lib().mt_smem_row_padding(columns, simultaneous_rows)


def mt_smem_vector_row_padding(columns: int, simultaneous_rows: int) -> int:
    return lib().mt_smem_vector_row_padding(columns, simultaneous_rows)


def mt_smem_layout_make(rows: int, columns: int, row_padding: int, stage_count: int):
    out = mt_smem_layout()
    st = lib().mt_smem_layout_make(rows, columns, row_padding, stage_count, ctypes.byref(out))
    return st, out


def mt_smem_layout_offset(layout: mt_smem_layout, stage: int, row: int, column: int) -> int:
    return lib().mt_smem_layout_offset(ctypes.byref(layout), stage, row, column)


def mt_check_device_status(stream: int = 0) -> int:
    return lib().mt_check_device_status(stream)


def mt_device_status(stream: int = 0) -> int:
    return lib().mt_device_status(stream)


def mt_status_string(status: int) -> str:
    return lib().mt_status_string(status).decode()


def mt_version() -> int:
    return lib().mt_version()


# --- torch convenience (marshalling only) ------------------------------------
def _check_device(t, name, device):
    """t must live on `device` (every operand of a call on one GPU): a host
    or other-GPU pointer handed to a kernel would read the wrong memory."""
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other operands on {device}")


def _check_tensor(t, name, device=None):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    _check_device(t, name, device)
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D (row-major) tensor")


def sgemm(a, b, out=None, stream=None, **choices):
    """out = a @ b through mt_sgemm_ex on torch tensors (float32, CUDA, row-major)."""
    import torch
    _check_tensor(a, "a")
    _check_tensor(b, "b", a.device)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    else:
        _check_tensor(out, "out", a.device)
        if tuple(out.shape) != (M, N):
            raise ValueError("out has the wrong shape")
    s = stream if stream is not None else torch.cuda.current_stream(a.device).cuda_stream
    with torch.cuda.device(a.device):
        st = mt_sgemm_ex(a.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K, s,
                         make_config(**choices) if choices else None)
    if st != MT_OK:
        raise MtError(st, "mt_sgemm_ex")
    return out


def plan(M: int, N: int, K: int, smem_limit_bytes: int = 0, a=None, b=None, c=None,
         **choices) -> dict:
    """mt_sgemm_plan as a dict (raises on a non-OK status)."""
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    st, p = mt_sgemm_plan(ptr(a), ptr(b), ptr(c), M, N, K,
                          make_config(**choices) if choices else None, smem_limit_bytes)
    if st != MT_OK:
        raise MtError(st, "mt_sgemm_plan")
    return p.as_dict()


def gemm(a, b, c=None, alpha=1.0, beta=0.0, trans_a=False, trans_b=False, stream=None,
         bias=None, **choices):
    """c = alpha * op(a) @ op(b) + beta * c (+ bias, a contiguous float32
    CUDA vector of N added to every row) on 2-D float32 CUDA tensors whose
    rows may be strided (unit column stride); op transposes the stored
    matrix when asked.  Returns c (allocated when not given; then beta must
    be 0)."""
    import torch
    for t, name in ((a, "a"), (b, "b")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
            raise TypeError(f"{name} must be a float32 CUDA tensor")
        _check_device(t, name, a.device)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be 2-D with unit column stride")
    M, K = (a.shape[1], a.shape[0]) if trans_a else (a.shape[0], a.shape[1])
    Kb, N = (b.shape[1], b.shape[0]) if trans_b else (b.shape[0], b.shape[1])
    if K != Kb:
        raise ValueError("inner dimensions differ")
    if c is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs c")
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if not isinstance(c, torch.Tensor) or c.dtype != torch.float32:
        raise TypeError("c must be a float32 CUDA tensor")
    _check_device(c, "c", a.device)
    if c.dim() != 2 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be M x N with unit column stride")
    def ld(t):  # row stride; any value >= the row length works for one row
        return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)

    if bias is not None:
        if (not isinstance(bias, torch.Tensor) or bias.dtype != torch.float32 or
                not bias.is_cuda or bias.dim() != 1 or bias.shape[0] != N or
                not bias.is_contiguous()):
            raise ValueError("bias must be a contiguous float32 CUDA vector of N")
        _check_device(bias, "bias", a.device)
    s = stream if stream is not None else torch.cuda.current_stream(a.device).cuda_stream
    cfg = make_config(**choices) if choices else None
    with torch.cuda.device(a.device):
        if bias is None:
            st = mt_sgemm_general(int(trans_a), int(trans_b), M, N, K, alpha, a.data_ptr(),
                                  ld(a), b.data_ptr(), ld(b), beta, c.data_ptr(), ld(c), s, cfg)
        else:
            st = mt_sgemm_general_bias(int(trans_a), int(trans_b), M, N, K, alpha, a.data_ptr(),
                                       ld(a), b.data_ptr(), ld(b), beta, bias.data_ptr(),
                                       c.data_ptr(), ld(c), s, cfg)
    if st != MT_OK:
        raise MtError(st, "mt_sgemm_general")
    return c


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return MT_DTYPE_F16
    if t.dtype == torch.bfloat16:
        return MT_DTYPE_BF16
    raise TypeError("16-bit inputs must be torch.float16 or torch.bfloat16")


def gemm_mixed(a, b, c=None, alpha=1.0, beta=0.0, trans_a=False, trans_b=False, stream=None,
               bias=None, **choices):
    """c (float32) = alpha * op(a) @ op(b) + beta * c (+ bias, N float32
    values on every row) with a and b 2-D CUDA tensors of the same 16-bit
    dtype (float16 or bfloat16) whose rows may be strided (unit column
    stride), through mt_gemm_mixed_general(_bias).  Returns c (allocated
    when not given; then beta must be 0)."""
    import torch
    for t, name in ((a, "a"), (b, "b")):
        _check_device(t, name, a.device if isinstance(a, torch.Tensor) else None)
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError(f"{name} must be 2-D with unit column stride")
    code = _dtype_code(a)
    if b.dtype != a.dtype:
        raise TypeError("a and b must have the same dtype")
    M, K = (a.shape[1], a.shape[0]) if trans_a else (a.shape[0], a.shape[1])
    Kb, N = (b.shape[1], b.shape[0]) if trans_b else (b.shape[0], b.shape[1])
    if K != Kb:
        raise ValueError("inner dimensions differ")
    if c is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs c")
        c = torch.empty((M, N), dtype=torch.float32, device=a.device)
    if not isinstance(c, torch.Tensor) or c.dtype != torch.float32:
        raise TypeError("c must be a float32 CUDA tensor")
    _check_device(c, "c", a.device)
    if c.dim() != 2 or c.stride(1) != 1 or tuple(c.shape) != (M, N):
        raise ValueError("c must be float32, M x N, with unit column stride")

    def ld(t):  # row stride; any value >= the row length works for one row
        return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)

    if bias is not None:
        if (not isinstance(bias, torch.Tensor) or bias.dtype != torch.float32 or
                not bias.is_cuda or bias.dim() != 1 or bias.shape[0] != N or
                not bias.is_contiguous()):
            raise ValueError("bias must be a contiguous float32 CUDA vector of N")
        _check_device(bias, "bias", a.device)
    s = stream if stream is not None else torch.cuda.current_stream(a.device).cuda_stream
    cfg = make_config(**choices) if choices else None
    with torch.cuda.device(a.device):
        if bias is None:
            st = mt_gemm_mixed_general(code, int(trans_a), int(trans_b), M, N, K, alpha,
                                       a.data_ptr(), ld(a), b.data_ptr(), ld(b), beta,
                                       c.data_ptr(), ld(c), s, cfg)
        else:
            st = mt_gemm_mixed_general_bias(code, int(trans_a), int(trans_b), M, N, K, alpha,
                                            a.data_ptr(), ld(a), b.data_ptr(), ld(b), beta,
                                            bias.data_ptr(), c.data_ptr(), ld(c), s, cfg)
    if st != MT_OK:
        raise MtError(st, "mt_gemm_mixed_general")
    return c


def plan_mixed(dtype: int, M: int, N: int, K: int, trans_a=False, trans_b=False, lda=0,
               ldb=0, ldc=0, a=None, b=None, c=None, smem_limit_bytes: int = 0,
               **choices) -> dict:
    """mt_gemm_mixed_plan as a dict (leading dimensions default to packed
    rows; raises on a non-OK status)."""
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    lda = lda or max(M if trans_a else K, 1)
    ldb = ldb or max(K if trans_b else N, 1)
    ldc = ldc or max(N, 1)
    st, p = mt_gemm_mixed_plan(dtype, int(trans_a), int(trans_b), M, N, K, ptr(a), lda, ptr(b),
                               ldb, ptr(c), ldc, make_config(**choices) if choices else None,
                               smem_limit_bytes)
    if st != MT_OK:
        raise MtError(st, "mt_gemm_mixed_plan")
    return p.as_dict()
