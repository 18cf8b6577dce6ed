"""The C-ABI library without a GPU: it loads, exports every function the header
declares, rejects bad arguments before touching CUDA, and its host-side tile
order is a bijection ("Skill: Write a Triton GEMM Kernel", Correctness
requirements: every (pid_m, pid_n) exactly once)."""
import os
import re

import pytest

import dense_gemm_bf16_gb300 as dg
from dense_gemm_bf16_gb300 import DType, Epi, Layout, Option, Status

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dg.build()
    return dg.lib()


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M):
            if not m.group(0).lstrip().startswith(("typedef", "#")):
                names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_binding(lib):
    declared = header_functions()
    assert set(declared) == set(dg.EXPORTED), declared


@pytest.mark.parametrize("name", header_functions())
def test_symbol_exported(lib, name):
    assert hasattr(lib, name)


def test_status_strings(lib):
    for s in Status:
        assert dg.gemm_status_string(s) == "GEMM_" + s.name
    assert dg.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def _bf16(M, N, K, **kw):
    args = dict(M=M, N=N, K=K, A=16, lda=max(K, 1), la=Layout.ROW_MAJOR, B=16, ldb=max(N, 1),
                lb=Layout.ROW_MAJOR, C=16, ldc=max(N, 1), lc=Layout.ROW_MAJOR,
                c_dtype=DType.F32, alpha=1.0, beta=0.0, bias=None, epi=Epi.NONE, split_k=0,
                workspace=None, workspace_bytes=0, stream=None)
    args.update(kw)
    return dg.gemm_bf16(**args)


@pytest.mark.parametrize("kw", [
    dict(M=-1, N=4, K=4),
    dict(M=4, N=-1, K=4),
    dict(M=4, N=4, K=-1),
    dict(M=4, N=4, K=4, lda=3),                        # lda < K
    dict(M=4, N=4, K=4, ldb=3),                        # ldb < N
    dict(M=4, N=4, K=4, ldc=3),                        # ldc < N
    dict(M=4, N=4, K=4, la=7),                         # bad layout
    dict(M=4, N=4, K=4, epi=8),                        # row-bias flag without a bias
    dict(M=4, N=4, K=4, epi=16),                       # bad epilogue
    dict(M=4, N=4, K=4, epi=Epi.BIAS),                 # bias missing
    dict(M=4, N=4, K=4, A=None),                       # A missing
    dict(M=4, N=4, K=4, C=None),                       # C missing
    dict(M=4, N=4, K=4, A=17),                         # A not 2-byte aligned
    dict(M=4, N=4, K=4, split_k=-2),
    dict(M=1 << 31, N=4, K=4),
    dict(M=4, N=4, K=4, lda=1 << 60),                  # span beyond 2^48 elements
    dict(M=4, N=4, K=4, ldb=(1 << 47) + 1),            # 3 * ldb + 4 > 2^48
    dict(M=4, N=4, K=4, ldc=(1 << 62) + 5),            # (M - 1) * ldc overflows int64
])
def test_invalid_arguments_rejected_without_gpu(lib, kw):
    assert _bf16(**kw) == Status.ERR_INVALID_ARG


def test_unsupported_dtype_mix(lib):
    assert _bf16(4, 4, 4, c_dtype=DType.F16) == Status.ERR_UNSUPPORTED
    st = dg.gemm_batched(DType.F32, 1, 4, 4, 4, 16, 4, 0, 0, 16, 4, 0, 0, 16, 4, 0, 0,
                         DType.BF16, 1.0, 0.0, None, 0, 0, None, 0, None)
    assert st == Status.ERR_UNSUPPORTED


def test_empty_problems_are_noops(lib):
    assert _bf16(0, 5, 5, A=None, B=None, C=None) == Status.OK
    assert _bf16(5, 0, 5, A=None, B=None, C=None) == Status.OK
    st = dg.gemm_batched(DType.BF16, 0, 4, 4, 4, None, 4, 0, 0, None, 4, 0, 0, None, 4, 0, 0,
                         DType.F32, 1.0, 0.0, None, 0, 0, None, 0, None)
    assert st == Status.OK


def test_batched_overlapping_C_rejected(lib):
    st = dg.gemm_batched(DType.BF16, 2, 4, 4, 4, 16, 4, 0, 16, 16, 4, 0, 16, 16, 4, 0, 8,
                         DType.F32, 1.0, 0.0, None, 0, 0, None, 0, None)
    assert st == Status.ERR_INVALID_ARG


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host has a GPU")
def test_valid_call_without_gpu_reports_no_device(lib):
    assert _bf16(4, 4, 4) == Status.ERR_NO_DEVICE
    assert dg.gemm_workspace_size(DType.BF16, 1, 256, 256, 65536, 0) == 0


def test_options(lib):
    assert dg.gemm_get_option(Option.GROUP_M) == 8
    assert dg.gemm_set_option(Option.GROUP_M, 0) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.GROUP_M, 65) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.GROUP_M, 3) == Status.OK
    assert dg.gemm_get_option(Option.GROUP_M) == 3
    assert dg.gemm_set_option(Option.GROUP_M, 8) == Status.OK
    assert dg.gemm_set_option(Option.TIMEOUT_US, 0) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.TEST_STALL, 3) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(99, 1) == Status.ERR_INVALID_ARG
    assert dg.gemm_get_option(99) == -1
    assert dg.gemm_get_option(Option.OVERLAP_COPY) == 0
    assert dg.gemm_set_option(Option.OVERLAP_COPY, 2) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.OVERLAP_COPY, 1) == Status.OK
    assert dg.gemm_get_option(Option.OVERLAP_COPY) == 1
    assert dg.gemm_set_option(Option.OVERLAP_COPY, 0) == Status.OK
    assert dg.gemm_get_option(Option.EPILOGUE_WARPS) == 0
    assert dg.gemm_set_option(Option.EPILOGUE_WARPS, 8) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.EPILOGUE_WARPS, 4) == Status.OK
    assert dg.gemm_get_option(Option.EPILOGUE_WARPS) == 4
    assert dg.gemm_set_option(Option.EPILOGUE_WARPS, 0) == Status.OK


def test_split_reduce_and_block_n_options(lib):
    assert dg.gemm_get_option(Option.SPLIT_REDUCE) == 0
    assert dg.gemm_get_option(Option.BLOCK_N) == 0
    for v in (0, 1, 2, 3, 4):
        assert dg.gemm_set_option(Option.SPLIT_REDUCE, v) == Status.OK
        assert dg.gemm_get_option(Option.SPLIT_REDUCE) == v
    assert dg.gemm_set_option(Option.SPLIT_REDUCE, 5) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.SPLIT_REDUCE, -1) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.SPLIT_REDUCE, 0) == Status.OK
    for v in (16, 32, 64, 128, 256, 0):
        assert dg.gemm_set_option(Option.BLOCK_N, v) == Status.OK
        assert dg.gemm_get_option(Option.BLOCK_N) == v
    for v in (8, 48, 96, 512, -16):
        assert dg.gemm_set_option(Option.BLOCK_N, v) == Status.ERR_INVALID_ARG
    assert dg.gemm_get_option(Option.BLOCK_N) == 0
    assert dg.gemm_get_option(Option.DOUBLE_K) == 0
    assert dg.gemm_set_option(Option.DOUBLE_K, 1) == Status.OK
    assert dg.gemm_get_option(Option.DOUBLE_K) == 1
    assert dg.gemm_set_option(Option.DOUBLE_K, 2) == Status.ERR_INVALID_ARG
    assert dg.gemm_set_option(Option.DOUBLE_K, 0) == Status.OK


@pytest.mark.parametrize("group_m", [1, 2, 3, 5, 8, 64])
def test_tile_order_is_a_bijection(lib, group_m):
    for npm in (1, 2, 3, 7, 8, 9, 17, 33, 64):
        for npn in (1, 2, 5, 12, 32):
            pm, pn = dg.gemm_tile_order(npm, npn, group_m)
            pairs = set(zip(pm, pn))
            assert len(pairs) == npm * npn
            assert all(0 <= a < npm for a in pm) and all(0 <= b < npn for b in pn)


def test_tile_order_group_one_is_row_major(lib):
    pm, pn = dg.gemm_tile_order(5, 7, 1)
    assert pm == [t // 7 for t in range(35)]
    assert pn == [t % 7 for t in range(35)]


def test_tile_order_groups_walk_columns_of_tile_rows(lib):
    # 8 tile-rows per group: the first 8 work items cover column 0 of rows 0..7
    pm, pn = dg.gemm_tile_order(16, 4, 8)
    assert pm[:8] == list(range(8)) and pn[:8] == [0] * 8
    assert pm[8:16] == list(range(8)) and pn[8:16] == [1] * 8
    assert pm[32:40] == list(range(8, 16)) and pn[32:40] == [0] * 8


# ---------------------------------------------------------------- header <-> binding

def _header_source():
    src = open(os.path.join(ROOT, "include", "gemm.h")).read()
    return re.sub(r"/\*.*?\*/", "", src, flags=re.S)


def _header_enum(type_name):
    m = re.search(r"typedef enum\s*\{([^{}]*)\}\s*" + type_name + r"\s*;", _header_source())
    assert m, type_name
    values = {}
    for item in m.group(1).split(","):
        item = item.strip()
        if item:
            name, value = (x.strip() for x in item.split("="))
            values[name] = int(value)
    return values


@pytest.mark.parametrize("type_name,prefix,enum_cls", [
    ("gemm_status_t", "GEMM_", Status),
    ("gemm_layout_t", "GEMM_", Layout),
    ("gemm_dtype_t", "GEMM_DT_", DType),
    ("gemm_epilogue_t", "GEMM_EPI_", Epi),
    ("gemm_option_t", "GEMM_OPT_", Option),
])
def test_header_enums_match_the_binding(type_name, prefix, enum_cls):
    header = {name[len(prefix):]: value for name, value in _header_enum(type_name).items()}
    binding = {member.name: int(member) for member in enum_cls}
    assert header == binding


def test_plan_struct_matches_the_header():
    import ctypes
    m = re.search(r"typedef struct\s*\{([^{}]*)\}\s*gemm_plan_t\s*;", _header_source())
    assert m
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        ctype, names = decl.split(None, 1)
        for name in names.split(","):
            fields.append((name.strip(), {"int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64}[ctype]))
    assert [(n, t) for n, t in dg.Plan._fields_] == fields


def _batched(batch, M, N, K, sa, sb, sc, lda=None, ldb=None, ldc=None):
    return dg.gemm_batched(DType.BF16, batch, M, N, K, 16, lda or K, 0, sa, 16, ldb or N, 0, sb,
                           16, ldc or N, 0, sc, DType.F32, 1.0, 0.0, None, 0, 0, None, 0, None)


def test_oversized_spans_and_counts_rejected(lib):
    ok = Status.ERR_NO_DEVICE   # the same call with sane sizes gets as far as the device query
    assert _batched(2, 4, 4, 4, 16, 16, 16) == ok
    assert _batched(2, 4, 4, 4, 16, 16, 1 << 62) == Status.ERR_INVALID_ARG   # C batch stride
    assert _batched(3, 4, 4, 4, 1 << 62, 16, 16) == Status.ERR_INVALID_ARG   # A batch stride
    assert _batched(1 << 20, 4, 4, 4, 16, 16, 1 << 28) == ok     # C spans just under 2^48
    assert _batched(1 << 20, 4, 4, 4, 16, 16, 1 << 29) == Status.ERR_INVALID_ARG  # about 2^49
    # batches of A overlapping (stride 1) leave the span small but not the count:
    # 2^30 x 2^14 x 2^14 = 2^58 elements, which no dense copy could hold
    assert _batched(1 << 30, 1 << 14, 1, 1 << 14, 1, 0, 1 << 14) == Status.ERR_INVALID_ARG
    # whereas a broadcast B of the same product is fine
    assert _batched(1 << 10, 1 << 14, 1, 1 << 14, 1 << 28, 0, 1 << 14) == ok


def test_strided_oversized_spans_and_counts_rejected(lib):
    def strided(batch, M, N, K, a, b, c):
        return dg.gemm_strided(DType.BF16, batch, M, N, K, 16, *a, 16, *b, 16, *c, DType.F32,
                               1.0, 0.0, None, 0, 0, None, 0, None)
    ok = Status.ERR_NO_DEVICE
    assert strided(1, 4, 4, 4, (4, 1, 0), (4, 1, 0), (4, 1, 0)) == ok
    assert strided(1, 4, 4, 4, (1 << 60, 1, 0), (4, 1, 0), (4, 1, 0)) == Status.ERR_INVALID_ARG
    assert strided(2, 4, 4, 4, (4, 1, 0), (4, 1, 0), (4, 1, 1 << 62)) == Status.ERR_INVALID_ARG
    assert strided(1, 1 << 31, 4, 4, (4, 1, 0), (4, 1, 0), (4, 1, 0)) == Status.ERR_INVALID_ARG
    # an overlapping C (row and column stride 1) of 2^60 elements spans little memory
    big = (1 << 30)
    assert strided(1, big, big, 4, (4, 1, 0), (big, 1, 0), (1, 1, 0)) == Status.ERR_INVALID_ARG
    assert dg.gemm_strided_workspace_size(0, 2, 1, big, big, 4, 4, 1, 0, big, 1, 0, 1, 1, 0,
                                          0) == 0


def test_workspace_size_of_oversized_problems_is_zero(lib):
    big = (1 << 31) - 1
    assert dg.gemm_workspace_size(DType.BF16, big, big, big, big, 0) == 0
    assert dg.gemm_workspace_size(DType.BF16, 1 << 20, 1 << 20, 1 << 20, 8, 0) == 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host has a GPU")
def test_every_compute_entry_reports_no_device_without_a_gpu(lib):
    nd = Status.ERR_NO_DEVICE
    assert dg.gemm_f16(4, 4, 4, 16, 4, 0, 16, 4, 0, 16, 4, 0, DType.F32, 1.0, 0.0, None, 0, 0,
                       None, 0, None) == nd
    assert dg.sgemm_f32(4, 4, 4, 16, 4, 0, 16, 4, 0, 16, 4, 0, 1.0, 0.0, None, 0, None) == nd
    assert dg.gemm_batched(DType.BF16, 2, 4, 4, 4, 16, 4, 0, 16, 16, 4, 0, 16, 16, 4, 0, 16,
                           DType.F32, 1.0, 0.0, None, 0, 0, None, 0, None) == nd
    assert dg.gemm_strided(DType.BF16, 1, 4, 4, 4, 16, 4, 1, 0, 16, 4, 1, 0, 16, 4, 1, 0,
                           DType.F32, 1.0, 0.0, None, 0, 0, None, 0, None) == nd
    assert dg.gemm_bf16_static_workspace(4, 4, 4, 16, 4, 0, 16, 4, 0, 16, 4, 0, DType.F32, 1.0,
                                         0.0, None, 0, 0, None) == nd
    assert dg.gemm_check_device_status(None) == nd
    st, _ = dg.gemm_plan_query(DType.BF16, 1, 4, 4, 4, 16, 4, 0, 0, 16, 4, 0, 0, 16, 4, 0, 0,
                               DType.F32, 1.0, 0.0, None, 0, 0, 0)
    assert st == nd


def test_debug_build_exports_the_same_entry_points_and_reports_itself():
    """libdgemm_gb300_debug.so (device-side checks, count-writes mode) has the
    same C interface; only it takes the debug-only option and count mode."""
    import dense_gemm_bf16_gb300 as dg
    D = dg.debug_lib()
    for name in dg.EXPORTED:
        assert hasattr(D, name), name
    assert dg.gemm_build_flags() == 0 and D.gemm_build_flags() == 1
    assert dg.gemm_set_option(dg.Option.TEST_DEBUG_BOUND, 1) == dg.Status.ERR_UNSUPPORTED
    assert dg.gemm_debug_count_writes(None, 0) == dg.Status.ERR_UNSUPPORTED
    assert D.gemm_set_option(int(dg.Option.TEST_DEBUG_BOUND), 3) == dg.Status.ERR_INVALID_ARG
    assert D.gemm_set_option(int(dg.Option.TEST_DEBUG_BOUND), 0) == dg.Status.OK
    assert D.gemm_debug_count_writes(1 << 24, 0) == dg.Status.ERR_INVALID_ARG
    assert D.gemm_debug_count_writes(None, 0) == dg.Status.OK
    assert D.gemm_status_string(7) == b"GEMM_ERR_DEVICE_CHECK"
