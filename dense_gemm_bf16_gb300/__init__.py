"""GB300-native (sm_103a) dense GEMM: C = act(alpha * A @ B + beta * C + bias).

The compute lives in the CUDA library libdgemm_gb300.so (C ABI:
include/gemm.h): a persistent tcgen05/TMA tensor-core kernel for bf16/fp16,
a CUDA-core SGEMM for fp32, their split-K / operand-copy helpers, and the
general-stride entry point.  This package is its binding: ``_abi`` mirrors the C entry points
one to one; ``api.gemm`` is the tensor-level convenience.
"""
from ._abi import (EXPORTED, STATIC_WORKSPACE_BYTES, DType, Epi, GemmError, Layout, Option, Plan,
                   Status, build, debug_lib, gemm_batched, gemm_bf16, gemm_bf16_static_workspace,
                   gemm_build_flags, gemm_check_device_status, gemm_debug_count_writes,
                   gemm_f16, gemm_get_option, gemm_plan_query,
                   gemm_set_option, gemm_status_string, gemm_strided, gemm_strided_plan_query,
                   gemm_strided_workspace_size, gemm_tile_order, gemm_workspace_size, lib,
                   library_path, sgemm_f32)

__all__ = [
    "EXPORTED", "STATIC_WORKSPACE_BYTES", "DType", "Epi", "GemmError", "Layout", "Option", "Plan",
    "Status", "build", "debug_lib", "gemm_batched", "gemm_bf16", "gemm_bf16_static_workspace",
    "gemm_build_flags", "gemm_check_device_status", "gemm_debug_count_writes", "gemm_f16", "gemm_get_option", "gemm_plan_query",
    "gemm_set_option", "gemm_status_string", "gemm_strided", "gemm_strided_plan_query",
    "gemm_strided_workspace_size", "gemm_tile_order", "gemm_workspace_size", "lib", "library_path", "sgemm_f32", "gemm", "plan",
]


def __getattr__(name):
    # the tensor-level API imports torch; load it on first use only
    if name in ("gemm", "plan", "api"):
        # import_module, not "from . import api": the latter looks the name up
        # on this package first, which would land here again
        import importlib
        api = importlib.import_module(".api", __name__)
        return api if name == "api" else getattr(api, name)
    raise AttributeError(name)
