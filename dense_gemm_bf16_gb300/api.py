"""Tensor-level convenience over the C ABI: reads pointers, leading dimensions,
layouts and batch strides off torch tensors and calls ``gemm_batched``, or
``gemm_strided`` for views that are not row- or column-major matrices.
PyTorch only provides device memory and the current stream; every step of the
GEMM runs in the library's CUDA kernels.
"""
from __future__ import annotations

import torch

from . import _abi
from ._abi import DType, Epi, GemmError, Layout, Status

_DT = {torch.bfloat16: DType.BF16, torch.float16: DType.F16, torch.float32: DType.F32}
# "none", "bias", "gelu_tanh", "bias_gelu_tanh", ..., "row_bias_gelu_erf"
_EPI = {e.name.lower(): e for e in Epi}


def matrix_desc(t: torch.Tensor):
    """(ptr, ld, layout, batch, batch_stride) of a 2-D or 3-D tensor whose
    last two dims form a row- or column-major matrix with unit inner stride."""
    if t.dim() == 2:
        t3 = t.unsqueeze(0)
        batch, bstride = 1, 0
    elif t.dim() == 3:
        t3 = t
        batch, bstride = t.shape[0], (t.stride(0) if t.shape[0] > 1 else 0)
    else:
        raise ValueError("expected a 2-D or 3-D tensor")
    rows, cols = t3.shape[1], t3.shape[2]
    s_r, s_c = t3.stride(1), t3.stride(2)
    # a dimension of extent 1 may carry any stride; otherwise the rows (or the
    # columns) must not overlap, as an expanded dimension of stride 0 would
    if (s_c == 1 or cols == 1) and (rows == 1 or s_r >= cols):
        return t.data_ptr(), max(s_r if rows > 1 else cols, cols, 1), Layout.ROW_MAJOR, \
            batch, bstride
    if (s_r == 1 or rows == 1) and (cols == 1 or s_c >= rows):
        return t.data_ptr(), max(s_c if cols > 1 else rows, rows, 1), Layout.COL_MAJOR, \
            batch, bstride
    raise ValueError("expected a row- or column-major matrix with unit inner stride and "
                     f"non-overlapping lines (shape {tuple(t.shape)}, strides {tuple(t.stride())})")


def strided_desc(t: torch.Tensor):
    """(ptr, row stride, column stride, batch stride) in elements of a 2-D or
    3-D tensor, as ``gemm_strided`` takes them (batch stride 0 for one matrix)."""
    if t.dim() == 2:
        return t.data_ptr(), t.stride(0), t.stride(1), 0
    if t.dim() == 3:
        return t.data_ptr(), t.stride(1), t.stride(2), (t.stride(0) if t.shape[0] > 1 else 0)
    raise ValueError("expected a 2-D or 3-D tensor")


def check(status: int) -> None:
    if status != Status.OK:
        raise GemmError(status)


def _common(A, B, C, bias, epilogue):
    """Checks shared by both routes: (M, N, K, batch, epilogue, bias pointer)."""
    if A.dtype != B.dtype or A.dtype not in _DT:
        raise TypeError("A and B must share one dtype among bfloat16, float16, float32")
    for name, t in (("A", A), ("B", B), ("C", C)):
        if t.dim() not in (2, 3):
            raise ValueError(f"{name} must be a 2-D or 3-D tensor")
    if C.dtype not in _DT:
        raise TypeError("C must be bfloat16, float16 or float32")
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-1]
    if B.shape[-2] != K or C.shape[-2] != M or C.shape[-1] != N:
        raise ValueError(f"shape mismatch: A{tuple(A.shape)} B{tuple(B.shape)} C{tuple(C.shape)}")
    ba, bb, bc = (t.shape[0] if t.dim() == 3 else 1 for t in (A, B, C))
    batch = max(ba, bb, bc)
    if ba not in (1, batch) or bb not in (1, batch):
        raise ValueError(f"batch sizes {ba} (A) and {bb} (B) do not broadcast to {batch}")
    if bc != batch:
        raise ValueError("C must carry the full batch")
    epi = epilogue if isinstance(epilogue, Epi) else _EPI.get(str(epilogue).lower())
    if epi is None:
        raise ValueError(f"unknown epilogue {epilogue!r}; one of {sorted(_EPI)}")
    has_bias = bool(epi & Epi.BIAS)
    if has_bias != (bias is not None):
        raise ValueError(f"epilogue {epi.name.lower()} " +
                         ("needs a bias" if has_bias else "takes no bias"))
    bias_ptr = 0
    if bias is not None:
        n_bias = M if epi & 8 else N
        if bias.dtype != torch.float32 or bias.numel() != n_bias or \
                (bias.numel() > 1 and bias.stride(-1) != 1):
            raise ValueError(f"bias must be a contiguous fp32 vector of length {n_bias}")
        bias_ptr = bias.data_ptr()
    return M, N, K, batch, epi, bias_ptr


def _args(A, B, C, alpha, beta, bias, epilogue, split_k):
    """Arguments of gemm_batched / gemm_plan_query (without the workspace and
    stream); raises ValueError for a view that is not row- or column-major."""
    M, N, K, batch, epi, bias_ptr = _common(A, B, C, bias, epilogue)
    pa, lda, la, _, sa = matrix_desc(A)
    pb, ldb, lb, _, sb = matrix_desc(B)
    pc, ldc, lc, _, sc = matrix_desc(C)
    return [int(_DT[A.dtype]), batch, M, N, K, pa, lda, int(la), sa, pb, ldb, int(lb), sb,
            pc, ldc, int(lc), sc, int(_DT[C.dtype]), float(alpha), float(beta), bias_ptr,
            int(epi), int(split_k)]


def _strided_args(A, B, C, alpha, beta, bias, epilogue, split_k):
    """Arguments of gemm_strided (without the workspace and stream)."""
    M, N, K, batch, epi, bias_ptr = _common(A, B, C, bias, epilogue)
    pa, ars, acs, sa = strided_desc(A)
    pb, brs, bcs, sb = strided_desc(B)
    pc, crs, ccs, sc = strided_desc(C)
    return [int(_DT[A.dtype]), batch, M, N, K, pa, ars, acs, sa, pb, brs, bcs, sb,
            pc, crs, ccs, sc, int(_DT[C.dtype]), float(alpha), float(beta), bias_ptr,
            int(epi), int(split_k)]


def _require_cuda(**tensors):
    """The kernels read every buffer through device pointers: a host tensor,
    or one on another GPU than A, would be an illegal address there."""
    dev = tensors["A"].device
    for name, t in tensors.items():
        if t is not None and (not t.is_cuda or t.device != dev):
            where = dev if dev.type == "cuda" else "one CUDA device"
            raise ValueError(f"{name} must be a CUDA tensor on {where} (it is on {t.device})")


def _is_matrix(t):
    try:
        matrix_desc(t)
        return True
    except ValueError:
        return False


def plan(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, *, alpha=1.0, beta=0.0, bias=None,
         epilogue=None, split_k=0, workspace_bytes=None):
    """The kernel plan gemm() would use (a dict), without launching anything;
    for views that go through gemm_strided, the plan of that call (its copies
    counted in pack_a / pack_b, launches and workspace_bytes)."""
    if epilogue is None:
        epilogue = "bias" if bias is not None else "none"
    ws = (1 << 62) if workspace_bytes is None else int(workspace_bytes)
    if all(_is_matrix(t) for t in (A, B, C)):
        st, p = _abi.gemm_plan_query(*_args(A, B, C, alpha, beta, bias, epilogue, split_k), ws)
    else:
        st, p = _abi.gemm_strided_plan_query(
            *_strided_args(A, B, C, alpha, beta, bias, epilogue, split_k), ws)
    check(st)
    return p.as_dict()


def gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *, alpha=1.0,
         beta=0.0, bias=None, epilogue=None, out_dtype=None, split_k=0, workspace=None,
         stream=None) -> torch.Tensor:
    """C <- act(alpha * A @ B + beta * C + bias) on the current CUDA device.

    A: [M,K] or [batch,M,K]; B: [K,N] or [batch,K,N] (a batch stride of 0,
    e.g. from ``expand``, broadcasts); C: output (allocated when None, in
    ``out_dtype`` or A's dtype).  Row- and column-major views run in place
    through ``gemm_batched``; any other strides (a step along the inner
    dimension, repeated rows) go through ``gemm_strided``, which copies those
    matrices into the workspace.  ``epilogue`` is a ``gemm_epilogue_t`` name in
    lower case ("bias_gelu_tanh", "row_bias_relu", ...) or an ``Epi``; it
    defaults to "bias" when a bias is given.  A workspace is allocated with
    torch when the call needs one and none is given.
    """
    if epilogue is None:
        epilogue = "bias" if bias is not None else "none"
    _require_cuda(A=A, B=B, C=C, bias=bias, workspace=workspace)
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        batch = max(A.shape[0] if A.dim() == 3 else 1, B.shape[0] if B.dim() == 3 else 1)
        shape = (A.shape[-2], B.shape[-1]) if A.dim() == 2 and B.dim() == 2 else \
            (batch, A.shape[-2], B.shape[-1])
        C = torch.empty(shape, dtype=out_dtype or A.dtype, device=A.device)
    strided = not all(_is_matrix(t) for t in (A, B, C))
    if strided:
        args = _strided_args(A, B, C, alpha, beta, bias, epilogue, split_k)
    else:
        args = _args(A, B, C, alpha, beta, bias, epilogue, split_k)
    if workspace is None:
        if strided:
            ab, batch, M, N, K = args[:5]
            need = int(_abi.gemm_strided_workspace_size(ab, args[17], batch, M, N, K, *args[6:9],
                                                        *args[10:13], *args[14:17], args[22]))
        else:
            st, p = _abi.gemm_plan_query(*args, 1 << 62)
            check(st)
            need = int(p.workspace_bytes)
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device) if need > 0 else None
    ws_ptr = 0 if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    call = _abi.gemm_strided if strided else _abi.gemm_batched
    check(call(*args, ws_ptr, ws_bytes, stream))
    return C
