"""ctypes binding of libdgemm_gb300.so, one Python function per C entry point
(include/gemm.h), with the same names and arguments.  Pointers are plain ints
(device addresses), streams are ints (cudaStream_t); every function returns
the C status code.  No arithmetic happens here.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None
_debug_lib = None


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_ARG = 1
    ERR_UNSUPPORTED = 2
    ERR_WORKSPACE = 3
    ERR_CUDA = 4
    ERR_TIMEOUT = 5
    ERR_NO_DEVICE = 6
    ERR_DEVICE_CHECK = 7


class Layout(enum.IntEnum):
    ROW_MAJOR = 0
    COL_MAJOR = 1


class DType(enum.IntEnum):
    BF16 = 0
    F16 = 1
    F32 = 2


class Epi(enum.IntEnum):
    NONE = 0
    BIAS = 1
    GELU_TANH = 2
    BIAS_GELU_TANH = 3
    RELU = 4
    BIAS_RELU = 5
    GELU_ERF = 6
    BIAS_GELU_ERF = 7
    ROW_BIAS = 9
    ROW_BIAS_GELU_TANH = 11
    ROW_BIAS_RELU = 13
    ROW_BIAS_GELU_ERF = 15


class Option(enum.IntEnum):
    GROUP_M = 1
    MAX_CTAS = 2
    TIMEOUT_US = 3
    TEST_STALL = 4
    CTA_PAIR = 5
    SWAP_AB = 6
    L2_HINTS = 7
    STREAM_K = 8
    FAST_EPILOGUE = 9
    SGEMM_KERNEL = 10
    WIDE_TILE = 11
    SPLIT_REDUCE = 12
    BLOCK_N = 13
    DOUBLE_K = 14
    TEST_SIM_SMS = 15
    TEST_DEBUG_BOUND = 16
    OVERLAP_COPY = 17
    EPILOGUE_WARPS = 18


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("block_m", ctypes.c_int32),
                ("block_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("swap_ab", ctypes.c_int32), ("pack_a", ctypes.c_int32),
                ("pack_b", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("group_m", ctypes.c_int32), ("launches", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("cta_pair", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("fast_epilogue", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmError(RuntimeError):
    def __init__(self, status):
        self.status = Status(status)
        super().__init__(gemm_status_string(int(status)))


_i64, _i32, _f32, _vp, _sz = (ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                              ctypes.c_size_t)

_GEMM16 = [_i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _i32, _i32,
           _f32, _f32, _vp, _i32, _i32, _vp, _sz, _vp]
_SIGNATURES = {
    "gemm_bf16": (_GEMM16, _i32),
    "gemm_f16": (_GEMM16, _i32),
    "sgemm_f32": ([_i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _i32,
                   _f32, _f32, _vp, _i32, _vp], _i32),
    "gemm_batched": ([_i32, _i64, _i64, _i64, _i64, _vp, _i64, _i32, _i64, _vp, _i64, _i32, _i64,
                      _vp, _i64, _i32, _i64, _i32, _f32, _f32, _vp, _i32, _i32, _vp, _sz, _vp],
                     _i32),
    "gemm_workspace_size": ([_i32, _i64, _i64, _i64, _i64, _i32], _sz),
    "gemm_strided": ([_i32, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _i64,
                      _vp, _i64, _i64, _i64, _i32, _f32, _f32, _vp, _i32, _i32, _vp, _sz, _vp],
                     _i32),
    "gemm_strided_workspace_size": ([_i32, _i32, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _i64, _i64, _i64, _i32], _sz),
    "gemm_status_string": ([_i32], ctypes.c_char_p),
    "gemm_check_device_status": ([_vp], _i32),
    "gemm_plan_query": ([_i32, _i64, _i64, _i64, _i64, _vp, _i64, _i32, _i64, _vp, _i64, _i32,
                         _i64, _vp, _i64, _i32, _i64, _i32, _f32, _f32, _vp, _i32, _i32, _sz,
                         ctypes.POINTER(Plan)], _i32),
    "gemm_strided_plan_query": ([_i32, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _i64, _vp, _i64,
                                 _i64, _i64, _vp, _i64, _i64, _i64, _i32, _f32, _f32, _vp, _i32,
                                 _i32, _sz, ctypes.POINTER(Plan)], _i32),
    "gemm_set_option": ([_i32, _i64], _i32),
    "gemm_get_option": ([_i32], _i64),
    "gemm_tile_order": ([_i32, _i32, _i32, ctypes.POINTER(ctypes.c_int),
                         ctypes.POINTER(ctypes.c_int)], None),
    "gemm_bf16_static_workspace": ([_i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32, _vp,
                                    _i64, _i32, _i32, _f32, _f32, _vp, _i32, _i32, _vp], _i32),
    "gemm_build_flags": ([], _i32),
    "gemm_debug_count_writes": ([_vp, _i64], _i32),
}
# size of the library-owned scratch array used by gemm_bf16_static_workspace
STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024
EXPORTED = tuple(_SIGNATURES)


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (incremental)."""
    return _build.build(force=force)


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(dense_gemm_bf16_gb300.build() or __graft_entry__.build())")
    L = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    return L


def lib():
    """The loaded library.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(_build.LIB_PATH)
    return _lib


def debug_lib():
    """The debug build (libdgemm_gb300_debug.so: the same entry points, with
    device-side checks and the count-writes mode), as a ctypes library whose
    functions take the C arguments directly.  It keeps its own device state
    (status word, options) apart from lib()'s."""
    global _debug_lib
    with _lock:
        if _debug_lib is None:
            _debug_lib = _load(_build.DEBUG_LIB_PATH)
    return _debug_lib


def gemm_bf16(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta, bias, epi,
              split_k, workspace, workspace_bytes, stream) -> int:
    return lib().gemm_bf16(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta,
                           bias, epi, split_k, workspace, workspace_bytes, stream)


def gemm_f16(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta, bias, epi,
             split_k, workspace, workspace_bytes, stream) -> int:
    return lib().gemm_f16(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta,
                          bias, epi, split_k, workspace, workspace_bytes, stream)


def sgemm_f32(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, alpha, beta, bias, epi,
              stream) -> int:
    return lib().sgemm_f32(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, alpha, beta, bias, epi,
                           stream)


def gemm_batched(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb, stride_b, C, ldc,
                 lc, stride_c, c_dtype, alpha, beta, bias, epi, split_k, workspace,
                 workspace_bytes, stream) -> int:
    return lib().gemm_batched(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb,
                              stride_b, C, ldc, lc, stride_c, c_dtype, alpha, beta, bias, epi,
                              split_k, workspace, workspace_bytes, stream)


def gemm_bf16_static_workspace(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta,
                               bias, epi, split_k, stream) -> int:
    """gemm_bf16 with the library's own scratch array instead of a caller
    workspace (for callers that cannot allocate device memory)."""
    return lib().gemm_bf16_static_workspace(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype,
                                            alpha, beta, bias, epi, split_k, stream)


def gemm_workspace_size(ab_dtype, batch, M, N, K, split_k) -> int:
    return lib().gemm_workspace_size(ab_dtype, batch, M, N, K, split_k)


def gemm_strided(ab_dtype, batch, M, N, K, A, a_rs, a_cs, stride_a, B, b_rs, b_cs, stride_b, C,
                 c_rs, c_cs, stride_c, c_dtype, alpha, beta, bias, epi, split_k, workspace,
                 workspace_bytes, stream) -> int:
    return lib().gemm_strided(ab_dtype, batch, M, N, K, A, a_rs, a_cs, stride_a, B, b_rs, b_cs,
                              stride_b, C, c_rs, c_cs, stride_c, c_dtype, alpha, beta, bias, epi,
                              split_k, workspace, workspace_bytes, stream)


def gemm_strided_workspace_size(ab_dtype, c_dtype, batch, M, N, K, a_rs, a_cs, stride_a, b_rs,
                                b_cs, stride_b, c_rs, c_cs, stride_c, split_k) -> int:
    return lib().gemm_strided_workspace_size(ab_dtype, c_dtype, batch, M, N, K, a_rs, a_cs,
                                             stride_a, b_rs, b_cs, stride_b, c_rs, c_cs,
                                             stride_c, split_k)


def gemm_status_string(status) -> str:
    return lib().gemm_status_string(int(status)).decode()


def gemm_check_device_status(stream) -> int:
    return lib().gemm_check_device_status(stream)


def gemm_plan_query(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb, stride_b, C, ldc,
                    lc, stride_c, c_dtype, alpha, beta, bias, epi, split_k, workspace_bytes):
    """Returns (status, Plan)."""
    plan = Plan()
    st = lib().gemm_plan_query(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb,
                               stride_b, C, ldc, lc, stride_c, c_dtype, alpha, beta, bias, epi,
                               split_k, workspace_bytes, ctypes.byref(plan))
    return st, plan


def gemm_strided_plan_query(ab_dtype, batch, M, N, K, A, a_rs, a_cs, stride_a, B, b_rs, b_cs,
                            stride_b, C, c_rs, c_cs, stride_c, c_dtype, alpha, beta, bias, epi,
                            split_k, workspace_bytes):
    """Returns (status, Plan) of the gemm_strided call with these arguments."""
    plan = Plan()
    st = lib().gemm_strided_plan_query(ab_dtype, batch, M, N, K, A, a_rs, a_cs, stride_a, B, b_rs,
                                       b_cs, stride_b, C, c_rs, c_cs, stride_c, c_dtype, alpha,
                                       beta, bias, epi, split_k, workspace_bytes,
                                       ctypes.byref(plan))
    return st, plan


def gemm_build_flags() -> int:
    return lib().gemm_build_flags()


def gemm_debug_count_writes(counts, count_elems) -> int:
    return lib().gemm_debug_count_writes(counts, count_elems)


def gemm_set_option(option, value) -> int:
    return lib().gemm_set_option(int(option), int(value))


def gemm_get_option(option) -> int:
    return lib().gemm_get_option(int(option))


def gemm_tile_order(num_pid_m, num_pid_n, group_m):
    """Returns two lists: pid_m[t], pid_n[t] for t in [0, num_pid_m*num_pid_n)."""
    n = num_pid_m * num_pid_n
    pm = (ctypes.c_int * max(n, 1))()
    pn = (ctypes.c_int * max(n, 1))()
    lib().gemm_tile_order(num_pid_m, num_pid_n, group_m, pm, pn)
    return list(pm[:n]), list(pn[:n])
