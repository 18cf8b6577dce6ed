"""CPU oracle for the dense GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``oracle_gemm.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_gemm.so")
_lock = threading.Lock()
_lib = None

DT = {"bf16": 0, "f16": 1, "f32": 2, "f64": 3}
LAYOUT = {"row": 0, "col": 1}
ACT = {"none": 0, "gelu_tanh": 1, "relu": 2, "gelu_erf": 3}


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no -ffast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB lets the planted-mistake tests load a mutated build
            override = os.environ.get("ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            common = [i32, i32, i64, i64, i64, i64,
                      vp, i64, i32, i64,
                      vp, i64, i32, i64,
                      vp, i64, i32, i64,
                      dbl, dbl, vp, i32, i32]
            strided = [i32, i32, i64, i64, i64, i64,
                       vp, i64, i64, i64,
                       vp, i64, i64, i64,
                       vp, i64, i64, i64,
                       dbl, dbl, vp, i32, i32]
            lib.oracle_gemm.argtypes = common + [vp]
            lib.oracle_gemm.restype = i32
            lib.oracle_gemm_sampled.argtypes = common + [i64, vp, vp, vp, vp]
            lib.oracle_gemm_sampled.restype = i32
            lib.oracle_gemm_strided.argtypes = strided + [vp]
            lib.oracle_gemm_strided.restype = i32
            lib.oracle_gemm_strided_sampled.argtypes = strided + [i64, vp, vp, vp, vp]
            lib.oracle_gemm_strided_sampled.restype = i32
            for fn in ("oracle_gelu_tanh", "oracle_gelu_erf", "oracle_relu"):
                getattr(lib, fn).argtypes = [dbl]
                getattr(lib, fn).restype = dbl
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_bf16.restype = dbl
            lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
            lib.oracle_decode_f16.restype = dbl
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _storage(a, dt):
    if a is None:
        return None
    want = np.uint16 if dt in ("bf16", "f16") else (np.float32 if dt == "f32" else np.float64)
    a = np.asarray(a)
    if a.dtype != want:
        raise TypeError(f"operand stored as {a.dtype}, expected {np.dtype(want)} for {dt}")
    return np.ascontiguousarray(a)


class Problem:
    """One GEMM call described exactly as the C-ABI describes it.

    Buffers are flat numpy arrays holding the storage (uint16 bit patterns for
    bf16/f16, float32 for f32); ``ld``/``layout``/``stride`` give the indexing.
    With ``strides`` = ((rs, cs) of A, of B, of C) every element (r, c) is at
    r*rs + c*cs instead, and ld/layout are not used.
    """

    def __init__(self, *, ab_dtype, M, N, K, A, B, lda=0, la="row", ldb=0, lb="row",
                 c_dtype="f32", C0=None, ldc=None, lc="row", batch=1,
                 stride_a=0, stride_b=0, stride_c=0, alpha=1.0, beta=0.0,
                 bias=None, act="none", bias_rows=False, strides=None):
        self.ab_dtype, self.c_dtype = ab_dtype, c_dtype
        self.M, self.N, self.K, self.batch = int(M), int(N), int(K), int(batch)
        self.A, self.B = _storage(A, ab_dtype), _storage(B, ab_dtype)
        self.C0 = _storage(C0, c_dtype)
        self.lda, self.ldb = int(lda), int(ldb)
        self.ldc = int(ldc if ldc is not None else (N if lc == "row" else M))
        self.la, self.lb, self.lc = la, lb, lc
        self.stride_a, self.stride_b, self.stride_c = int(stride_a), int(stride_b), int(stride_c)
        self.alpha, self.beta = float(alpha), float(beta)
        self.bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        self.act = act
        self.bias_rows = 1 if bias_rows else 0
        self.strides = None if strides is None else [tuple(int(v) for v in st) for st in strides]

    def _args(self):
        if self.strides is not None:
            (ars, acs), (brs, bcs), (crs, ccs) = self.strides
            return [DT[self.ab_dtype], DT[self.c_dtype], self.batch, self.M, self.N, self.K,
                    _ptr(self.A), ars, acs, self.stride_a,
                    _ptr(self.B), brs, bcs, self.stride_b,
                    _ptr(self.C0), crs, ccs, self.stride_c,
                    self.alpha, self.beta, _ptr(self.bias), self.bias_rows, ACT[self.act]]
        return [DT[self.ab_dtype], DT[self.c_dtype], self.batch, self.M, self.N, self.K,
                _ptr(self.A), self.lda, LAYOUT[self.la], self.stride_a,
                _ptr(self.B), self.ldb, LAYOUT[self.lb], self.stride_b,
                _ptr(self.C0), self.ldc, LAYOUT[self.lc], self.stride_c,
                self.alpha, self.beta, _ptr(self.bias), self.bias_rows, ACT[self.act]]

    def _fns(self):
        lib = _load()
        if self.strides is not None:
            return lib.oracle_gemm_strided, lib.oracle_gemm_strided_sampled
        return lib.oracle_gemm, lib.oracle_gemm_sampled


def gemm(p: Problem) -> np.ndarray:
    """Full fp64 result, shape [batch, M, N]."""
    out = np.empty((p.batch, p.M, p.N), dtype=np.float64)
    rc = p._fns()[0](*p._args(), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected its arguments (rc={rc})")
    return out


def gemm_sampled(p: Problem, b_idx, i_idx, j_idx) -> np.ndarray:
    """fp64 values R[b, i, j] at the given index triples, computed one by one."""
    i_idx = np.ascontiguousarray(i_idx, dtype=np.int64)
    j_idx = np.ascontiguousarray(j_idx, dtype=np.int64)
    b_idx = (np.zeros_like(i_idx) if b_idx is None
             else np.ascontiguousarray(b_idx, dtype=np.int64))
    if not (len(b_idx) == len(i_idx) == len(j_idx)):
        raise ValueError("index arrays differ in length")
    out = np.empty(len(i_idx), dtype=np.float64)
    rc = p._fns()[1](*p._args(), len(i_idx), _ptr(b_idx), _ptr(i_idx), _ptr(j_idx), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_gemm_sampled rejected its arguments (rc={rc})")
    return out


def gelu_tanh(x: float) -> float:
    return _load().oracle_gelu_tanh(float(x))


def gelu_erf(x: float) -> float:
    return _load().oracle_gelu_erf(float(x))


def relu(x: float) -> float:
    return _load().oracle_relu(float(x))


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(int(bits))


def decode_f16(bits: int) -> float:
    return _load().oracle_decode_f16(int(bits))


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Vector decode of a storage array to fp64, through the oracle's decoders."""
    lib = _load()
    flat = np.asarray(bits).ravel()
    if dtype == "f32":
        return flat.astype(np.float64).reshape(np.shape(bits))
    fn = lib.oracle_decode_bf16 if dtype == "bf16" else lib.oracle_decode_f16
    # decode each distinct bit pattern once
    uniq, inv = np.unique(flat.astype(np.uint16), return_inverse=True)
    vals = np.array([fn(int(u)) for u in uniq], dtype=np.float64)
    return vals[inv].reshape(np.shape(bits))
