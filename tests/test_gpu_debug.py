"""The debug build (libdgemm_gb300_debug.so: the same sources with device-side
checks and the count-writes mode).

- Clean runs: every kernel family through the debug build gives the oracle's
  result, trips no check, and writes every output element exactly once (the
  count-writes mode), including the 8192^3 headline call and the ragged
  4097 x 3001 x 1000 workload in the bench's plans.
- Planted mistakes: a test-only option hands the next launch one bound that
  is too small (the buffers themselves are fine), so a check must fail; the
  accesses it guards are skipped (their outputs keep their poison), the rest
  of the result is right, the status word reports GEMM_ERR_DEVICE_CHECK, and
  the next call is clean.
"""
import numpy as np
import pytest

from gemm_case import Case, check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def D():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_bf16_gb300 as dg
    dg.build()
    L = dg.debug_lib()
    assert L.gemm_build_flags() == 1
    return L


def _opts(D, opts):
    import dense_gemm_bf16_gb300 as dg
    for k, v in opts.items():
        assert D.gemm_set_option(int(dg.Option[k]), v) == 0


def _reset(D, opts):
    import dense_gemm_bf16_gb300 as dg
    for k in opts:
        D.gemm_set_option(int(dg.Option[k]), 0)


def _counted_run(D, case):
    """Runs the case through the debug build with the count-writes mode on;
    returns (status, C storage, counts [batch, M, N])."""
    n = max(case.batch * case.M * case.N, 1)
    counts = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert D.gemm_debug_count_writes(counts.data_ptr(), n) == 0
    try:
        st, out = case.run_gpu(L=D)
    finally:
        D.gemm_debug_count_writes(None, 0)
    torch.cuda.synchronize()
    return st, out, counts.cpu().numpy().reshape(case.batch, case.M, case.N)


# name: (Case arguments, library options, exact)
CLEAN = {
    "pair_two_k_blocks": (dict(M=700, N=600, K=640, lb="col"), {"CTA_PAIR": 3}, True),
    "pair_two_k_blocks_mn_major": (dict(M=700, N=600, K=640), {"CTA_PAIR": 3}, True),
    "single_cta_bn64": (dict(M=300, N=100, K=200), {}, True),
    "pairs_copied_b_overlapped": (dict(M=700, N=601, K=1000, lb="row"),
                                  {"CTA_PAIR": 3, "BLOCK_N": 256}, True),
    "eight_epilogue_warps_col_major": (dict(M=600, N=520, K=256, lc="col"),
                                       {"CTA_PAIR": 3, "BLOCK_N": 256}, True),
    "eight_epilogue_warps_beta_tma": (dict(M=520, N=700, K=300, c_dtype="bf16", beta=1.0,
                                           values="uniform", split_k=1),
                                      {"CTA_PAIR": 3, "BLOCK_N": 256}, False),
    "stream_k_split_pairs": (dict(M=700, N=600, K=1088, lb="col"),
                             {"STREAM_K": 3, "CTA_PAIR": 3, "MAX_CTAS": 8, "BLOCK_N": 256}, True),
    "stream_k_contiguous": (dict(M=700, N=600, K=1000),
                            {"STREAM_K": 2, "MAX_CTAS": 8, "CTA_PAIR": 1}, True),
    "spread_split_k": (dict(M=128, N=256, K=8192), {"SPLIT_REDUCE": 2}, True),
    "atomic_split_k": (dict(M=128, N=256, K=8192, beta=2.0, c_values="ints"), {}, True),
    "atomic_swapped": (dict(M=16, N=900, K=8192, beta=2.0, c_values="ints"),
                       {"SPLIT_REDUCE": 4}, True),
    "explicit_split_k": (dict(M=130, N=200, K=2048, split_k=4), {}, True),
    "swap_ab": (dict(M=16, N=900, K=256), {}, True),
    "batched_broadcast": (dict(M=300, N=400, K=150, batch=3, broadcast_b=True), {}, True),
    "unaligned_c_st_global": (dict(M=300, N=301, K=200, pads=(0, 0, 1)), {}, True),
    "col_major_c": (dict(M=200, N=300, K=128, lc="col"), {}, True),
    "wide_tile": (dict(M=600, N=700, K=1000), {"WIDE_TILE": 2, "CTA_PAIR": 3}, True),
    "packed_operands": (dict(M=257, N=333, K=100, pads=(1, 1, 0), offsets=(1, 1, 0)), {}, True),
    "beta_bf16_tma_loads": (dict(M=520, N=700, K=300, c_dtype="bf16", beta=1.0, bias=True,
                                 act="gelu_tanh", values="uniform"), {}, False),
    "general_epilogue_beta": (dict(M=333, N=520, K=300, c_dtype="f32", beta=0.5, bias=True,
                                   row_bias=True, act="relu", values="uniform"),
                              {"FAST_EPILOGUE": 1}, False),
    "sgemm": (dict(ab="f32", M=130, N=70, K=50, alpha=1.5), {}, True),
    "k_zero": (dict(M=50, N=60, K=0, beta=0.5, bias=True, values="uniform"), {}, False),
}


@pytest.mark.parametrize("name", sorted(CLEAN))
def test_clean_run_matches_and_writes_every_element_once(D, name):
    kw, opts, exact = CLEAN[name]
    kw = dict(kw)
    ab = kw.pop("ab", "bf16")
    kw.setdefault("values", "ints")
    case = Case(ab, seed=1201, **kw)
    _opts(D, opts)
    try:
        st, out, counts = _counted_run(D, case)
    finally:
        _reset(D, opts)
    assert st == 0, (st, case.plan)
    assert D.gemm_check_device_status(None) == 0, case.plan
    got, ref = case.result(out), case.oracle_full()
    if exact:
        assert np.array_equal(got, ref), case.plan
    else:
        check_close(case, got, ref)
    assert case.untouched_padding(out)
    assert (counts == 1).all(), (np.unique(counts, return_counts=True), case.plan)


def _count_full_size(D, M, N, K, args_fn, ws_bytes):
    n = M * N
    counts = torch.zeros(n, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    assert D.gemm_debug_count_writes(counts.data_ptr(), n) == 0
    try:
        st = D.gemm_batched(*args_fn(), ws.data_ptr() if ws_bytes else None, ws_bytes, stream)
        torch.cuda.synchronize()
    finally:
        D.gemm_debug_count_writes(None, 0)
    assert st == 0
    assert D.gemm_check_device_status(None) == 0
    assert bool((counts == 1).all()), int((counts != 1).sum())


def test_headline_writes_every_element_once(D):
    """bf16 8192^3, A row-major, B column-major, bias + GELU: the bench's call
    and plan (CTA pairs, two K blocks per load, no workspace)."""
    import ctypes

    import dense_gemm_bf16_gb300 as dg
    M = N = K = 8192
    A = torch.zeros(M * K, dtype=torch.int16, device="cuda")
    B = torch.zeros(K * N, dtype=torch.int16, device="cuda")
    bias = torch.zeros(N, dtype=torch.float32, device="cuda")
    C = torch.empty(M * N, dtype=torch.int16, device="cuda")

    def args():
        return [0, 1, M, N, K, A.data_ptr(), K, 0, 0, B.data_ptr(), K, 1, 0, C.data_ptr(), N, 0,
                0, 0, 1.0, 0.0, bias.data_ptr(), 3, 0]
    plan = dg.Plan()
    assert D.gemm_plan_query(*args(), 0, ctypes.byref(plan)) == 0
    assert plan.cta_pair == 2 and plan.block_k == 128 and plan.fast_epilogue == 1
    _count_full_size(D, M, N, K, args, 0)


def test_ragged_workload_writes_every_element_once(D):
    """4097 x 3001 x 1000 with an fp32 output whose rows are not 16-byte
    aligned (st.global epilogue on eight warps) and a B copied for alignment
    (the GEMM launched as the copy's programmatic dependent)."""
    import ctypes

    import dense_gemm_bf16_gb300 as dg
    M, N, K = 4097, 3001, 1000
    A = torch.zeros(M * K, dtype=torch.int16, device="cuda")
    B = torch.zeros(K * N, dtype=torch.int16, device="cuda")
    C = torch.empty(M * N, dtype=torch.float32, device="cuda")

    def args():
        return [0, 1, M, N, K, A.data_ptr(), K, 0, 0, B.data_ptr(), N, 0, 0, C.data_ptr(), N, 0,
                0, 2, 1.0, 0.0, None, 0, 0]
    plan = dg.Plan()
    assert D.gemm_plan_query(*args(), 1 << 40, ctypes.byref(plan)) == 0
    assert plan.pack_b == 1 and plan.fast_epilogue == 3
    _count_full_size(D, M, N, K, args, int(plan.workspace_bytes))


def test_planted_c_span_skips_the_stores_beyond_it(D):
    """C's span handed to the kernel halved: the st.global stores past it are
    skipped (those elements keep their NaN poison), every other element is
    right, and the status word reports a failed check."""
    case = Case("bf16", 300, 301, 200, pads=(0, 0, 1), values="ints", seed=1202)
    _opts(D, {"TEST_DEBUG_BOUND": 1})
    try:
        st, out = case.run_gpu(L=D)
    finally:
        _reset(D, {"TEST_DEBUG_BOUND": 1})
    assert st == 0 and case.plan["fast_epilogue"] == 0, case.plan
    assert D.gemm_check_device_status(None) == 7            # GEMM_ERR_DEVICE_CHECK
    got, ref = case.result(out)[0], case.oracle_full()[0]
    span = (case.M - 1) * case.ldc + case.N
    off = np.arange(case.M)[:, None] * case.ldc + np.arange(case.N)[None, :]
    kept = off < span // 2
    assert np.array_equal(got[kept], ref[kept])
    assert np.isnan(got[~kept]).all() and (~kept).sum() > 0
    # the next call is clean
    st, out = Case("bf16", 300, 301, 200, pads=(0, 0, 1), values="ints", seed=1203).run_gpu(L=D)
    assert st == 0 and D.gemm_check_device_status(None) == 0


def test_planted_tile_column_bound_skips_those_units(D):
    """The last tile column counted as outside the problem: every role of the
    kernel skips those work units together (no wait is left hanging), their
    outputs keep their poison, the rest is right, and the status word reports
    a failed check."""
    case = Case("bf16", 300, 600, 256, values="ints", split_k=1, seed=1204)
    _opts(D, {"TEST_DEBUG_BOUND": 2})
    try:
        st, out = case.run_gpu(L=D)
    finally:
        _reset(D, {"TEST_DEBUG_BOUND": 2})
    assert st == 0 and case.plan["stream_k"] == 0 and case.plan["swap_ab"] == 0, case.plan
    assert D.gemm_check_device_status(None) == 7
    got, ref = case.result(out)[0], case.oracle_full()[0]
    bn = case.plan["block_n"]
    last = (-(-case.N // bn) - 1) * bn                       # first column of the last tile column
    assert np.array_equal(got[:, :last], ref[:, :last])
    assert np.isnan(got[:, last:]).all()
    st, out = Case("bf16", 300, 600, 256, values="ints", split_k=1, seed=1205).run_gpu(L=D)
    assert st == 0 and D.gemm_check_device_status(None) == 0
