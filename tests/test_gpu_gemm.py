"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Sizes span several tiles and ragged tails; every layout combination, the
split-K and swap-AB plans, batched/broadcast strides, unaligned operands,
fused epilogues and the degenerate cases are covered.  Small-integer inputs
make every fp32 partial sum exact, so those cases must match the oracle
bit for bit whatever the tile order, split or batch.
"""
import numpy as np
import pytest

from gemm_case import Case, check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_bf16_gb300 as dg
    dg.build()
    dg.lib()
    yield
    dg.gemm_set_option(dg.Option.MAX_CTAS, 0)
    dg.gemm_set_option(dg.Option.GROUP_M, 8)


def run_exact(case):
    st, out = case.run_gpu()
    assert st == 0, f"status {st}"
    got = case.result(out)
    ref = case.oracle_full()
    assert np.array_equal(got, ref), (
        f"max |diff| {np.abs(got - ref).max()} plan={getattr(case, 'plan', None)}")
    assert case.untouched_padding(out)
    return case


def run_close(case):
    st, out = case.run_gpu()
    assert st == 0, f"status {st}"
    got = case.result(out)
    ref = case.oracle_full()
    check_close(case, got, ref)
    assert case.untouched_padding(out)
    return case


# ---------------------------------------------------------------- exact integer cases

@pytest.mark.parametrize("la", ["row", "col"])
@pytest.mark.parametrize("lb", ["row", "col"])
@pytest.mark.parametrize("ab", ["bf16", "f16"])
def test_exact_layouts(la, lb, ab):
    run_exact(Case(ab, 300, 520, 200, la=la, lb=lb, values="ints", pads=(3, 5, 7), seed=11))


@pytest.mark.parametrize("lc", ["row", "col"])
def test_exact_output_layout(lc):
    run_exact(Case("bf16", 257, 130, 190, lc=lc, values="ints", pads=(0, 0, 3), seed=12))


@pytest.mark.parametrize("N", [16, 24, 32, 48, 64, 100, 128, 200, 600])
def test_exact_block_n_variants(N):
    import dense_gemm_bf16_gb300 as dg
    # few CTAs: every CTA walks several tiles, so the stage ring and both TMEM
    # accumulators wrap many times
    dg.gemm_set_option(dg.Option.MAX_CTAS, 6)
    try:
        c = run_exact(Case("bf16", 700, N, 333, values="ints", seed=13))
    finally:
        dg.gemm_set_option(dg.Option.MAX_CTAS, 0)
    assert c.plan["kernel"] == 1


@pytest.mark.parametrize("lb", ["row", "col"])
@pytest.mark.parametrize("split", [2, 3, 7])
def test_exact_split_k(lb, split):
    c = run_exact(Case("bf16", 256, 384, 1000, lb=lb, values="ints", split_k=split, seed=14))
    assert c.plan["split_k"] == split


@pytest.mark.parametrize("la", ["row", "col"])
@pytest.mark.parametrize("M", [1, 5, 16, 33, 64])
def test_exact_swap_ab(la, M):
    c = run_exact(Case("bf16", M, 1000, 300, la=la, values="ints", seed=15))
    assert c.plan["swap_ab"] == 1


def test_exact_batched_broadcast():
    run_exact(Case("bf16", 130, 200, 150, batch=3, values="ints", broadcast_b=True, seed=16))
    run_exact(Case("bf16", 130, 200, 150, batch=3, la="col", lb="col", values="ints", seed=17))


def test_exact_persistent_many_tiles_group_orders():
    import dense_gemm_bf16_gb300 as dg
    for g in (1, 3, 8):
        dg.gemm_set_option(dg.Option.GROUP_M, g)
        dg.gemm_set_option(dg.Option.MAX_CTAS, 7)
        try:
            run_exact(Case("bf16", 1100, 900, 128, values="ints", seed=18))
        finally:
            dg.gemm_set_option(dg.Option.GROUP_M, 8)
            dg.gemm_set_option(dg.Option.MAX_CTAS, 0)


# ---------------------------------------------------------------- tolerance cases

@pytest.mark.parametrize("act", ["none", "gelu_tanh"])
@pytest.mark.parametrize("c_dtype", ["bf16", "f32"])
def test_epilogue_bias_alpha_beta(act, c_dtype):
    run_close(Case("bf16", 333, 444, 555, c_dtype=c_dtype, alpha=0.75, beta=-0.5, bias=True,
                   act=act, pads=(2, 2, 2), seed=21))


@pytest.mark.parametrize("c_dtype", ["f16", "f32"])
def test_f16_inputs(c_dtype):
    run_close(Case("f16", 300, 260, 520, lb="col", c_dtype=c_dtype, alpha=1.5, beta=0.5,
                   bias=True, seed=22))


def test_long_k_fp32_accumulation():
    # K = 8192: an fp16/bf16 accumulator would be far outside the fp32 bound
    run_close(Case("bf16", 128, 256, 8192, c_dtype="f32", seed=23))


def test_split_k_with_epilogue():
    run_close(Case("bf16", 200, 300, 4096, c_dtype="bf16", alpha=2.0, beta=1.0, bias=True,
                   act="gelu_tanh", split_k=5, seed=24))


def test_swap_with_bias_col_major_c():
    run_close(Case("bf16", 12, 700, 640, lc="col", c_dtype="f32", bias=True, beta=0.25, seed=25))


def test_batched_in_place_beta_one():
    run_close(Case("bf16", 256, 256, 256, batch=4, c_dtype="bf16", alpha=0.5, beta=1.0,
                   broadcast_b=True, seed=26))


# ---------------------------------------------------------------- unaligned operands

@pytest.mark.parametrize("pads,offsets", [((1, 0, 0), (0, 0, 0)), ((0, 1, 0), (0, 0, 0)),
                                          ((0, 0, 0), (1, 0, 0)), ((0, 0, 0), (0, 3, 0)),
                                          ((0, 0, 1), (0, 0, 1)), ((1, 1, 1), (1, 1, 1))])
def test_unaligned_operands(pads, offsets):
    c = run_exact(Case("bf16", 190, 301, 157, values="ints", pads=pads, offsets=offsets, seed=31))
    assert c.plan["pack_a"] or c.plan["pack_b"] or pads[:2] == (0, 0) and offsets[:2] == (0, 0)


def test_unaligned_batched_and_broadcast():
    run_exact(Case("bf16", 70, 90, 33, batch=3, values="ints", pads=(1, 3, 1), seed=32))
    run_exact(Case("bf16", 70, 90, 33, batch=3, values="ints", pads=(1, 3, 1),
                   broadcast_b=True, seed=33))


# ---------------------------------------------------------------- degenerate cases

def test_k_zero_and_alpha_zero():
    run_close(Case("bf16", 50, 60, 0, c_dtype="f32", beta=0.5, bias=True, act="gelu_tanh",
                   seed=41))
    run_close(Case("bf16", 50, 60, 40, c_dtype="bf16", alpha=0.0, beta=2.0, seed=42))


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 7, 3), (3, 1, 5), (2, 3, 1), (129, 257, 17),
                                   (128, 256, 64), (127, 255, 63)])
def test_tiny_and_boundary_shapes(shape):
    M, N, K = shape
    run_exact(Case("bf16", M, N, K, values="ints", seed=43 + M))


def test_beta_zero_ignores_nan_in_c():
    c = Case("bf16", 100, 100, 100, c_dtype="f32", beta=0.0, seed=44)
    st, out = c.run_gpu()
    assert st == 0
    assert np.all(np.isfinite(c.result(out)))


# ---------------------------------------------------------------- fp32 CUDA-core SGEMM

@pytest.mark.parametrize("la", ["row", "col"])
@pytest.mark.parametrize("lb", ["row", "col"])
def test_sgemm_exact_layouts(la, lb):
    run_exact(Case("f32", 300, 260, 270, la=la, lb=lb, values="ints", pads=(1, 3, 2), seed=51))


def test_sgemm_alpha_beta_bias_gelu():
    run_close(Case("f32", 257, 129, 333, alpha=1.5, beta=0.5, bias=True, act="gelu_tanh",
                   seed=52))


def test_sgemm_batched_unaligned():
    run_exact(Case("f32", 70, 90, 33, batch=3, values="ints", pads=(1, 1, 1),
                   offsets=(1, 2, 3), seed=53))


# Row-major A and B with 16-byte aligned rows take the cp.async kernel; the
# padding keeps lda = 272 and ldb = 260 multiples of 4 while K = 270 and N = 258
# end inside a 16-byte copy, so the zero-filled tails are exercised.
def test_sgemm_async_exact_ragged():
    c = run_exact(Case("f32", 300, 258, 270, values="ints", pads=(2, 2, 0), seed=55))
    assert c.lda % 4 == 0 and c.ldb % 4 == 0


def test_sgemm_async_batched():
    run_exact(Case("f32", 70, 92, 36, batch=3, values="ints", seed=56))


@pytest.mark.parametrize("shape", [(300, 258, 270), (129, 260, 1000)])
def test_sgemm_async_matches_register_staged(shape):
    # both kernels add the products of each output in ascending k with fmaf
    import dense_gemm_bf16_gb300 as dg
    M, N, K = shape
    kw = dict(alpha=1.5, beta=0.5, bias=True, act="gelu_tanh", pads=(2, 2, 0), seed=57)
    fast = Case("f32", M, N, K, **kw)
    st, out_a = fast.run_gpu()
    assert st == 0
    check_close(fast, fast.result(out_a), fast.oracle_full())
    dg.gemm_set_option(dg.Option.SGEMM_KERNEL, 1)
    try:
        st, out_b = Case("f32", M, N, K, **kw).run_gpu()
    finally:
        dg.gemm_set_option(dg.Option.SGEMM_KERNEL, 0)
    assert st == 0
    assert np.array_equal(out_a.view(np.uint8), out_b.view(np.uint8))


def test_sgemm_is_true_fp32():
    # TF32 would keep 10 mantissa bits (rms error ~3e-4); fp32 FFMA gives ~1e-6.
    c = Case("f32", 256, 256, 1024, seed=54)
    st, out = c.run_gpu()
    assert st == 0
    got, ref = c.result(out), c.oracle_full()
    assert np.sqrt(np.mean((got - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)) <= 1e-5


# ---------------------------------------------------------------- bounded waits

def test_stalled_pipeline_reports_timeout_and_recovers():
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.TIMEOUT_US, 20000)
    try:
        dg.gemm_set_option(dg.Option.TEST_STALL, 1)
        c = Case("bf16", 256, 256, 256, values="ints", seed=61)
        st, _ = c.run_gpu()
        assert st == 0
        stream = torch.cuda.current_stream().cuda_stream
        assert dg.gemm_check_device_status(stream) == dg.Status.ERR_TIMEOUT
        assert dg.gemm_check_device_status(stream) == dg.Status.OK
    finally:
        dg.gemm_set_option(dg.Option.TEST_STALL, 0)
        dg.gemm_set_option(dg.Option.TIMEOUT_US, 1000000)
    # the context is still usable and the next GEMM is right
    run_exact(Case("bf16", 256, 256, 256, values="ints", seed=62))
    assert dg.gemm_check_device_status(torch.cuda.current_stream().cuda_stream) == 0


# ---------------------------------------------------------------- two-CTA clusters

@pytest.fixture(params=[3], ids=["pair_mma"])
def pairs(request):
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.CTA_PAIR, request.param)
    dg.gemm_set_option(dg.Option.MAX_CTAS, 8)  # four clusters walk many tile pairs
    yield request.param - 1
    dg.gemm_set_option(dg.Option.CTA_PAIR, 0)
    dg.gemm_set_option(dg.Option.MAX_CTAS, 0)


@pytest.mark.parametrize("la", ["row", "col"])
@pytest.mark.parametrize("lb", ["row", "col"])
@pytest.mark.parametrize("N", [200, 600])
def test_exact_cluster_pairs(pairs, la, lb, N):
    # 700 rows = 5.5 tiles: the second CTA of the last pair has no valid rows
    c = run_exact(Case("bf16", 700, N, 333, la=la, lb=lb, values="ints", seed=71))
    assert c.plan["cta_pair"] == pairs


def test_exact_cluster_pairs_batched(pairs):
    c = run_exact(Case("bf16", 300, 400, 150, batch=3, values="ints", broadcast_b=True, seed=72))
    assert c.plan["cta_pair"] in (pairs, 0)
    run_exact(Case("bf16", 300, 400, 150, batch=3, lb="col", values="ints", seed=73))


def test_cluster_pairs_epilogue(pairs):
    c = run_close(Case("bf16", 520, 700, 300, c_dtype="bf16", alpha=0.5, beta=1.0, bias=True,
                       act="gelu_tanh", seed=74))
    assert c.plan["cta_pair"] in (pairs, 0)


# ---------------------------------------------------------------- stream-K

# GEMM_OPT_STREAM_K 2 forces the contiguous form (plan stream_k 1), 3 the split
# form (plan stream_k 2); each with one CTA per tile and with pair MMA
@pytest.fixture(params=[(2, 1), (2, 3), (3, 1), (3, 3)],
                ids=["contiguous-single_cta", "contiguous-pair_mma", "split-single_cta",
                     "split-pair_mma"])
def streamk(request):
    import dense_gemm_bf16_gb300 as dg
    form, pair = request.param
    dg.gemm_set_option(dg.Option.STREAM_K, form)
    dg.gemm_set_option(dg.Option.CTA_PAIR, pair)
    dg.gemm_set_option(dg.Option.MAX_CTAS, 8)  # few clusters: several whole units, then a cut tail
    yield form - 1
    dg.gemm_set_option(dg.Option.STREAM_K, 0)
    dg.gemm_set_option(dg.Option.CTA_PAIR, 0)
    dg.gemm_set_option(dg.Option.MAX_CTAS, 0)


# On 8 CTAs and on 4 CTA pairs each shape leaves a last wave of 1 to 3 units
# after whole ones, cut into 2 or 4 pieces by the split form (pieces of 4, 5 or
# 5 and 6 K blocks).
@pytest.mark.parametrize("shape", [(700, 600, 1000), (700, 600, 600), (700, 600, 700)])
def test_exact_stream_k(streamk, shape):
    M, N, K = shape
    c = run_exact(Case("bf16", M, N, K, values="ints", seed=81 + K))
    assert c.plan["stream_k"] == streamk


# contiguous form only: partial last waves the split form leaves alone
@pytest.mark.parametrize("shape", [(700, 600, 333), (1100, 700, 1000), (300, 1200, 130),
                                   (1300, 1100, 257)])
def test_exact_stream_k_contiguous(streamk, shape):
    M, N, K = shape
    c = run_exact(Case("bf16", M, N, K, values="ints", seed=91 + M))
    if streamk == 1:
        assert c.plan["stream_k"] == 1


def test_exact_stream_k_batched(streamk):
    c = run_exact(Case("bf16", 300, 520, 600, batch=3, values="ints", seed=85))
    assert c.plan["stream_k"] == streamk


def test_stream_k_epilogue(streamk):
    c = run_close(Case("bf16", 700, 600, 600, c_dtype="bf16", alpha=0.5, beta=1.0, bias=True,
                       act="gelu_tanh", seed=86))
    assert c.plan["stream_k"] == streamk


def test_stream_k_fp32_out(streamk):
    c = run_close(Case("bf16", 700, 600, 1000, c_dtype="f32", beta=-1.0, seed=88))
    assert c.plan["stream_k"] == streamk


def test_stream_k_unaligned_c(streamk):
    # st.global epilogue path (ldc not a multiple of 16 bytes)
    c = run_exact(Case("bf16", 700, 601, 1000, values="ints", pads=(0, 0, 1), seed=87))
    assert c.plan["stream_k"] == streamk


# ---------------------------------------------------------------- epilogue forms

@pytest.fixture
def general_epilogue():
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.FAST_EPILOGUE, 1)
    yield
    dg.gemm_set_option(dg.Option.FAST_EPILOGUE, 0)


# The TMA-store-only epilogue (beta == 0 or split-K partials) and the general
# one do the same fp32 arithmetic in the same order, so they agree bit for bit;
# each case also meets the oracle.  Shapes leave a ragged last 64-column step
# (N % 64 != 0, with C rows still 16-byte aligned for TMA) and a ragged last
# row block.
FORM_CASES = {
    "bf16_bias_gelu": dict(ab="bf16", M=333, N=712, K=300, c_dtype="bf16", alpha=0.5, bias=True,
                           act="gelu_tanh"),
    "f16_out": dict(ab="f16", M=300, N=520, K=200, c_dtype="f16", alpha=2.0),
    "f32_out_bias": dict(ab="bf16", M=260, N=332, K=450, c_dtype="f32", bias=True),
    "batched_bf16": dict(ab="bf16", M=200, N=264, K=130, batch=3, c_dtype="bf16", bias=True),
    "splitk_partials": dict(ab="bf16", M=130, N=200, K=2048, c_dtype="bf16", split_k=4,
                            bias=True, act="gelu_tanh"),
    # swap-AB computes C^T: a column-major C makes it row-major, and the bias
    # runs along its rows
    "swap_row_bias": dict(ab="bf16", M=40, N=900, K=256, lc="col", c_dtype="f32", bias=True),
    "pair_mma": dict(ab="bf16", M=1100, N=1304, K=320, c_dtype="bf16", alpha=0.25, bias=True,
                     opts={"CTA_PAIR": 3}),
}


def _form_run(name, seed):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(FORM_CASES[name])
    opts = kw.pop("opts", {})
    for k, v in opts.items():
        dg.gemm_set_option(dg.Option[k], v)
    try:
        c = Case(seed=seed, **kw)
        st, out = c.run_gpu()
    finally:
        for k in opts:
            dg.gemm_set_option(dg.Option[k], 0)
    assert st == 0, f"status {st}"
    return c, out


@pytest.mark.parametrize("name", sorted(FORM_CASES))
def test_fast_epilogue_matches_general(name):
    import dense_gemm_bf16_gb300 as dg
    fast, out_fast = _form_run(name, 301)
    assert fast.plan["fast_epilogue"] == 1, fast.plan
    if "opts" in FORM_CASES[name]:
        assert fast.plan["cta_pair"] == FORM_CASES[name]["opts"]["CTA_PAIR"] - 1, fast.plan
    check_close(fast, fast.result(out_fast), fast.oracle_full())
    assert fast.untouched_padding(out_fast)
    dg.gemm_set_option(dg.Option.FAST_EPILOGUE, 1)
    try:
        gen, out_gen = _form_run(name, 301)
    finally:
        dg.gemm_set_option(dg.Option.FAST_EPILOGUE, 0)
    assert gen.plan["fast_epilogue"] == 0
    assert np.array_equal(out_fast.view(np.uint8), out_gen.view(np.uint8))


def test_beta_epilogue_forms():
    # a 16-bit C that takes TMA stores reads beta * C by TMA loads (form 2); an
    # fp32 C keeps the general form
    c = run_close(Case("bf16", 300, 520, 200, c_dtype="bf16", beta=0.5, seed=311))
    assert c.plan["fast_epilogue"] == 2
    c = run_close(Case("bf16", 300, 520, 200, c_dtype="f32", beta=0.5, seed=312))
    assert c.plan["fast_epilogue"] == 0


# beta * C by TMA loads: tile widths, pair tiles, ragged edges (N = 712 ends 8
# columns into a 64-column step; M = 333 inside a 32-row box), a row bias, a
# batch (3-D maps) and the finishing piece of an in-kernel split
BETA_FORM_CASES = {
    "bn64": dict(ab="bf16", M=333, N=712, K=300, opts={"BLOCK_N": 64}),
    "bn128": dict(ab="bf16", M=333, N=712, K=300, bias=True, act="gelu_tanh"),
    "bn256": dict(ab="bf16", M=333, N=712, K=300, opts={"BLOCK_N": 256}),
    "pair128": dict(ab="bf16", M=1100, N=1304, K=320, opts={"CTA_PAIR": 3, "BLOCK_N": 128}),
    "pair256": dict(ab="bf16", M=1100, N=1304, K=320, bias=True,
                    opts={"CTA_PAIR": 3, "BLOCK_N": 256}),
    "f16_row_bias_relu": dict(ab="f16", M=300, N=520, K=200, bias=True, row_bias=True,
                              act="relu"),
    "batched": dict(ab="bf16", M=200, N=264, K=130, batch=3, bias=True, act="gelu_erf"),
    "inkernel_split_head": dict(ab="bf16", M=1024, N=640, K=4096, bias=True,
                                opts={"SPLIT_REDUCE": 3}),
    "balanced_contiguous_head": dict(ab="bf16", M=1024, N=640, K=4096, bias=True),
}


@pytest.mark.parametrize("name", sorted(BETA_FORM_CASES))
def test_beta_epilogue_matches_general(name):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(BETA_FORM_CASES[name])
    opts = kw.pop("opts", {})

    def run(extra):
        for k, v in {**opts, **extra}.items():
            dg.gemm_set_option(dg.Option[k], v)
        try:
            c = Case(c_dtype=kw["ab"], alpha=0.5, beta=-0.75, seed=331, **kw)
            st, out = c.run_gpu()
        finally:
            for k in {**opts, **extra}:
                dg.gemm_set_option(dg.Option[k], 0)
        assert st == 0, f"status {st}"
        return c, out
    c, out = run({})
    # 4: the same form on eight epilogue warps (whole 256-wide pair tiles of at
    # most 32 K blocks)
    assert c.plan["fast_epilogue"] in (2, 4), c.plan
    if name == "pair256":
        assert c.plan["fast_epilogue"] == 4, c.plan
    if "CTA_PAIR" in opts:
        assert c.plan["cta_pair"] == 2, c.plan
    if "BLOCK_N" in opts:
        assert c.plan["block_n"] == opts["BLOCK_N"], c.plan
    if name == "inkernel_split_head":
        assert c.plan["stream_k"] == 2, c.plan
    if name == "balanced_contiguous_head":
        assert c.plan["stream_k"] == 1, c.plan
    check_close(c, c.result(out), c.oracle_full())
    assert c.untouched_padding(out)
    g, out_g = run({"FAST_EPILOGUE": 1})
    assert g.plan["fast_epilogue"] == 0
    assert np.array_equal(out.view(np.uint8), out_g.view(np.uint8))
    if c.plan["fast_epilogue"] == 4:
        f, out_f = run({"EPILOGUE_WARPS": 4})
        assert f.plan["fast_epilogue"] == 2, f.plan
        assert np.array_equal(out.view(np.uint8), out_f.view(np.uint8))


@pytest.mark.parametrize("shape", [(700, 600, 333), (4097, 700, 64)])
def test_exact_general_epilogue_forced(general_epilogue, shape):
    M, N, K = shape
    c = run_exact(Case("bf16", M, N, K, values="ints", seed=321 + M))
    assert c.plan["fast_epilogue"] == 0


# ---------------------------------------------------------------- activations and bias orientation

# Every route the epilogue can take, with each activation and the bias along
# columns or rows.  Each entry: Case keyword arguments, options to set, and the
# plan fields the route must show.
EPI_ROUTES = {
    "tc_fast": (dict(ab="bf16", M=333, N=712, K=300, c_dtype="bf16", alpha=0.5), {},
                {"fast_epilogue": 1}),
    "tc_general_beta": (dict(ab="bf16", M=333, N=712, K=300, c_dtype="bf16", beta=0.75),
                        {"FAST_EPILOGUE": 1}, {"fast_epilogue": 0}),
    "tc_beta_tma": (dict(ab="bf16", M=333, N=712, K=300, c_dtype="bf16", beta=0.75), {},
                    {"fast_epilogue": 2}),
    "tc_unaligned_ldc": (dict(ab="bf16", M=260, N=701, K=200, c_dtype="f32"), {},
                         {"fast_epilogue": 0}),
    "tc_col_major_c": (dict(ab="f16", M=200, N=300, K=160, lc="col", c_dtype="f32",
                            beta=-0.5), {}, {"swap_ab": 0}),
    "swap_ab": (dict(ab="bf16", M=40, N=900, K=256, c_dtype="f32"), {}, {"swap_ab": 1}),
    "split_k": (dict(ab="bf16", M=130, N=200, K=2048, c_dtype="bf16", split_k=4), {},
                {"split_k": 4}),
    "pair_mma": (dict(ab="bf16", M=1100, N=1304, K=320, c_dtype="bf16", alpha=0.25),
                 {"CTA_PAIR": 3}, {"cta_pair": 2}),
    "sgemm_cp_async": (dict(ab="f32", M=300, N=260, K=272, alpha=1.5, beta=0.5), {}, {}),
    "sgemm_staged": (dict(ab="f32", M=300, N=260, K=270, la="col", beta=0.5), {}, {}),
    "k_zero": (dict(ab="bf16", M=70, N=90, K=0, c_dtype="f32", beta=0.5), {}, {}),
}


@pytest.mark.parametrize("row_bias", [False, True], ids=["col_bias", "row_bias"])
@pytest.mark.parametrize("act", ["relu", "gelu_erf", "gelu_tanh"])
@pytest.mark.parametrize("route", sorted(EPI_ROUTES))
def test_epilogue_activation_routes(route, act, row_bias):
    import dense_gemm_bf16_gb300 as dg
    kw, opts, want = EPI_ROUTES[route]
    for k, v in opts.items():
        dg.gemm_set_option(dg.Option[k], v)
    try:
        c = run_close(Case(bias=True, act=act, row_bias=row_bias, seed=401, **kw))
    finally:
        for k in opts:
            dg.gemm_set_option(dg.Option[k], 0)
    for k, v in want.items():
        assert c.plan[k] == v, (k, c.plan)


@pytest.mark.parametrize("shape", [(333, 712, 300), (40, 900, 256), (300, 260, 272)])
@pytest.mark.parametrize("row_bias", [False, True], ids=["col_bias", "row_bias"])
def test_exact_relu(shape, row_bias):
    # small integers: the accumulator is exact, so is ReLU of it plus an
    # integer-valued bias
    M, N, K = shape
    ab = "f32" if shape == (300, 260, 272) else "bf16"
    c = Case(ab, M, N, K, values="ints", bias=True, act="relu", row_bias=row_bias, seed=411)
    c.bias = np.round(c.bias * 4).astype(np.float32)
    run_exact(c)



@pytest.mark.parametrize("shape", [(16, 8192, 8192), (256, 256, 65536), (128, 256, 8192)])
def test_auto_split_keeps_its_splits_in_the_reported_workspace(shape):
    # a call given exactly the workspace its plan reported must make the same plan
    import dense_gemm_bf16_gb300 as dg
    M, N, K = shape
    args = [0, 1, M, N, K, 1 << 20, K, 0, 0, 1 << 20, N, 0, 0, 1 << 20, N, 0, 0, 2, 1.0, 0.0,
            None, 0, 0]
    st, big = dg.gemm_plan_query(*args, 1 << 40)
    assert st == 0 and (big.split_k > 1 or big.stream_k in (1, 2, 3, 4))
    st, exact = dg.gemm_plan_query(*args, int(big.workspace_bytes))
    assert st == 0
    assert (exact.split_k, exact.stream_k, exact.grid) == (big.split_k, big.stream_k, big.grid)
    assert exact.workspace_bytes == big.workspace_bytes


# ---------------------------------------------------------------- automatic split-K in one kernel

# An automatic split of 2-4 pieces per unit runs in one kernel (plan split_k 1,
# no reduction launch): by default balanced over every CTA as the contiguous
# form of stream-K (plan stream_k 1), or with GEMM_OPT_SPLIT_REDUCE = 3 as equal
# pieces, one CTA each (the split form, stream_k 2); GEMM_OPT_STREAM_K = 1
# falls back to the two-pass split-K.
INKERNEL_CASES = {
    # C rows 4 bytes past a 16-byte multiple: no TMA reduce-adds, so the
    # swapped product keeps a one-kernel form with partials
    "skinny_swap": dict(M=16, N=8192, K=4096, pads=(0, 0, 1)),
    "three_pieces": dict(M=1024, N=640, K=4096),
}
INKERNEL_FORMS = {"balanced": ({}, 1), "equal_pieces": ({"SPLIT_REDUCE": 3}, 2)}


@pytest.fixture(params=sorted(INKERNEL_FORMS))
def inkernel_form(request):
    import dense_gemm_bf16_gb300 as dg
    opts, form = INKERNEL_FORMS[request.param]
    for k, v in opts.items():
        dg.gemm_set_option(dg.Option[k], v)
    yield form
    for k in opts:
        dg.gemm_set_option(dg.Option[k], 0)


@pytest.mark.parametrize("name", sorted(INKERNEL_CASES))
def test_exact_inkernel_split(name, inkernel_form):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(INKERNEL_CASES[name])
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    c = run_exact(Case("bf16", M, N, K, values="ints", seed=501, **kw))
    assert c.plan["stream_k"] == inkernel_form and c.plan["split_k"] == 1, c.plan
    assert c.plan["launches"] == 1, c.plan
    dg.gemm_set_option(dg.Option.STREAM_K, 1)
    try:
        c2 = run_exact(Case("bf16", M, N, K, values="ints", seed=501, **kw))
    finally:
        dg.gemm_set_option(dg.Option.STREAM_K, 0)
    assert c2.plan["stream_k"] == 0 and c2.plan["split_k"] > 1


def test_inkernel_split_epilogue_and_beta(inkernel_form):
    c = run_close(Case("bf16", 1024, 640, 4096, c_dtype="bf16", alpha=0.5, beta=0.75, bias=True,
                       act="gelu_tanh", seed=502))
    assert c.plan["stream_k"] == inkernel_form


def test_inkernel_split_unaligned_c(inkernel_form):
    # fp32 C with ldc = 641: the head's output goes through the st.global path
    c = run_close(Case("bf16", 1024, 641, 4096, c_dtype="f32", bias=True, act="relu",
                       row_bias=True, seed=503))
    assert c.plan["stream_k"] == inkernel_form


# ---------------------------------------------------------------- atomic split-K (option)

# GEMM_OPT_SPLIT_REDUCE = 4: every K piece adds alpha * its partial into an fp32
# C by TMA reduce-add, after the CTAs set C to beta * C + bias (the pages'
# atomic accumulation; the sum order varies between runs, so only small-integer
# data is bit-exact).  An activation or a 16-bit C keeps the default forms.
ATOMIC_CASES = {
    "square_long_k": dict(M=256, N=256, K=16384),
    "pieces_per_tile_38": dict(M=256, N=256, K=65536),
    "one_tile_152_pieces": dict(M=128, N=128, K=32768),
    "alpha_beta_bias": dict(M=256, N=384, K=8192, alpha=0.5, beta=2.0, bias=True,
                            c_values="ints"),
    "row_bias_batched": dict(M=128, N=256, K=8192, batch=2, bias=True, row_bias=True),
    "ragged_k": dict(M=200, N=264, K=6000),
    "ragged_m": dict(M=384, N=256, K=8192),
    "batched_pairs": dict(M=256, N=256, K=4096, batch=2),
    "wide_n": dict(M=256, N=768, K=16384),
    # swapped skinny products (C^T = B^T A^T, column-major computed C): 16-,
    # 32- and 64-wide tiles reduce-added through column boxes
    "swapped_bn16": dict(M=16, N=900, K=8192),
    "swapped_bn32": dict(M=32, N=520, K=8192, alpha=0.5, beta=2.0, bias=True, c_values="ints"),
    "swapped_bn64_row_bias": dict(M=48, N=640, K=16384, bias=True, row_bias=True),
    "swapped_ragged_k": dict(M=16, N=1000, K=6000),
}


# each case with the plan's own pairing (CTA pairs wherever there are two tile
# rows) and with single CTAs forced
@pytest.mark.parametrize("pairs", [True, False], ids=["auto", "single"])
@pytest.mark.parametrize("name", sorted(ATOMIC_CASES))
def test_exact_atomic_split_k(name, pairs):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(ATOMIC_CASES[name])
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 4)
    dg.gemm_set_option(dg.Option.CTA_PAIR, 0 if pairs else 1)
    try:
        c = Case("bf16", values="ints", seed=509, **kw)
        if c.bias is not None:
            c.bias = np.round(c.bias * 4).astype(np.float32)
        st, out = c.run_gpu()
    finally:
        dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)
        dg.gemm_set_option(dg.Option.CTA_PAIR, 0)
    assert st == 0, c.plan
    assert c.plan["stream_k"] == 4 and c.plan["split_k"] == 1 and c.plan["launches"] == 1 + \
        c.plan["pack_a"] + c.plan["pack_b"], c.plan
    assert c.plan["cta_pair"] == (2 if pairs and kw["M"] > 128 else 0), c.plan
    assert np.array_equal(c.result(out), c.oracle_full()), c.plan
    assert c.untouched_padding(out)
    assert dg.gemm_check_device_status(None) == 0


def test_atomic_split_k_uniform_values_within_tolerance():
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 4)
    try:
        c = run_close(Case("bf16", 256, 256, 65536, alpha=1.5, beta=0.5, bias=True, seed=510))
    finally:
        dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)
    assert c.plan["stream_k"] == 4, c.plan


@pytest.mark.parametrize("kw", [dict(c_dtype="bf16"), dict(act="relu")], ids=["bf16_out", "relu"])
def test_atomic_split_k_needs_fp32_out_and_no_activation(kw):
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 4)
    try:
        c = run_close(Case("bf16", 256, 256, 16384, seed=511, **kw))
    finally:
        dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)
    assert c.plan["stream_k"] in (1, 3), c.plan     # the default one-kernel forms


# ---------------------------------------------------------------- spread split-K in one kernel

# More than 4 automatic pieces per tile: every piece publishes its fp32 partial
# and then reduces one equal share of the tile (plan stream_k 3, one launch).
# Shares end at arbitrary positions of a tile (S does not divide it), tiles run
# past the matrix edges, and the swapped skinny case has 16-wide tiles.
SPREAD_CASES = {
    "square_long_k": dict(M=256, N=256, K=16384),
    "ragged": dict(M=200, N=312, K=20000),
    "skinny_swap": dict(M=16, N=1008, K=32768),
    "batched": dict(M=130, N=200, K=8192, batch=3),
}


def _spread_case(name, **extra):
    kw = dict(SPREAD_CASES[name])
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    return Case("bf16", M, N, K, **kw, **extra)


@pytest.fixture
def fixed_order():
    # GEMM_OPT_SPLIT_REDUCE = 2: the spread reduction (fixed order of addition)
    # also where the default would add the pieces atomically (an fp32 C that
    # takes TMA stores, no activation)
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 2)
    yield
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)


@pytest.mark.parametrize("name", sorted(SPREAD_CASES))
def test_exact_spread_split(name, fixed_order):
    c = run_exact(_spread_case(name, values="ints", seed=701))
    assert c.plan["stream_k"] == 3 and c.plan["split_k"] == 1 and c.plan["launches"] == 1, c.plan


@pytest.mark.parametrize("name", sorted(SPREAD_CASES))
def test_exact_default_many_pieces(name):
    # by default an fp32 C that takes TMA stores (without an activation) gets
    # the atomic form, the swapped skinny case (column-major C^T) included
    c = run_exact(_spread_case(name, values="ints", seed=710))
    assert c.plan["stream_k"] == 4, c.plan
    assert c.plan["split_k"] == 1 and c.plan["launches"] == 1, c.plan


@pytest.mark.parametrize("name", ["square_long_k", "ragged"])
def test_spread_matches_two_pass(name):
    # GEMM_OPT_SPLIT_REDUCE = 1 keeps the two-pass form; exact inputs, so both
    # forms give the oracle's result bit for bit
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 1)
    try:
        c = run_exact(_spread_case(name, values="ints", seed=702))
    finally:
        dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)
    assert c.plan["stream_k"] == 0 and c.plan["split_k"] > 1 and c.plan["launches"] == 2, c.plan


@pytest.mark.parametrize("name", sorted(INKERNEL_CASES))
def test_exact_spread_forced_for_few_pieces(name):
    import dense_gemm_bf16_gb300 as dg
    kw = INKERNEL_CASES[name]
    dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 2)
    try:
        c = run_exact(Case("bf16", kw["M"], kw["N"], kw["K"], values="ints", seed=703))
    finally:
        dg.gemm_set_option(dg.Option.SPLIT_REDUCE, 0)
    assert c.plan["stream_k"] == 3 and c.plan["launches"] == 1, c.plan


@pytest.mark.parametrize("lc", ["row", "col"])
def test_spread_epilogue_and_beta(lc):
    c = run_close(Case("bf16", 256, 256, 16384, lc=lc, c_dtype="bf16", alpha=0.5, beta=0.75,
                       bias=True, act="gelu_tanh", seed=704))
    assert c.plan["stream_k"] == 3


def test_spread_fp32_unaligned_c_row_bias():
    c = run_close(Case("bf16", 200, 301, 20000, c_dtype="f32", bias=True, row_bias=True,
                       act="relu", seed=705))
    assert c.plan["stream_k"] == 3


def test_spread_f16_swap_with_bias():
    c = run_close(Case("f16", 16, 1000, 32768, c_dtype="f16", bias=True, act="gelu_erf",
                       seed=706))
    assert c.plan["stream_k"] == 3 and c.plan["swap_ab"] == 1


@pytest.mark.parametrize("bn", [64, 256])
def test_exact_spread_other_tile_widths(bn, fixed_order):
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.BLOCK_N, bn)
    try:
        c = run_exact(Case("bf16", 256, 512, 16384, values="ints", seed=707))
    finally:
        dg.gemm_set_option(dg.Option.BLOCK_N, 0)
    assert c.plan["block_n"] == bn and c.plan["stream_k"] == 3, c.plan


def test_spread_unpublished_partial_reports_timeout_and_recovers(fixed_order):
    # the first CTA leaves its partial unpublished: the pieces of its tile give
    # up after the wait bound, the call reports a timeout, and the context stays
    # usable
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.TIMEOUT_US, 20000)
    try:
        dg.gemm_set_option(dg.Option.TEST_STALL, 2)
        c = Case("bf16", 256, 256, 16384, values="ints", seed=708)
        st, _ = c.run_gpu()
        assert st == 0 and c.plan["stream_k"] == 3
        stream = torch.cuda.current_stream().cuda_stream
        assert dg.gemm_check_device_status(stream) == dg.Status.ERR_TIMEOUT
        assert dg.gemm_check_device_status(stream) == dg.Status.OK
    finally:
        dg.gemm_set_option(dg.Option.TEST_STALL, 0)
        dg.gemm_set_option(dg.Option.TIMEOUT_US, 1000000)
    run_exact(_spread_case("square_long_k", values="ints", seed=709))
    assert dg.gemm_check_device_status(torch.cuda.current_stream().cuda_stream) == 0


# ---------------------------------------------------------------- two K blocks per TMA load

# CTA-pair plans bring two 64-deep K blocks per load (plan block_k 128): a
# K-major operand through a (64 K, rows, K blocks) view, where an odd count of
# K blocks reads its last block's partner past the end of K (zeros); an
# MN-major operand in atom columns of 128 K rows, where rows past K read
# zeros.  The K order is the same, so the bits match the one-block form
# exactly.
DOUBLE_K_CASES = {
    "even_bn128": dict(M=600, N=700, K=640, opts={"CTA_PAIR": 3, "BLOCK_N": 128}),
    "odd_bn256": dict(M=600, N=700, K=320, opts={"CTA_PAIR": 3, "BLOCK_N": 256}),
    "odd_many_tiles": dict(M=1100, N=1304, K=1088, opts={"CTA_PAIR": 3}),
    "packed_a": dict(M=520, N=600, K=704, pads=(8, 0, 0), offsets=(1, 0, 0),
                     opts={"CTA_PAIR": 3}),
}


def _double_k_run(kw, extra, **case_kw):
    import dense_gemm_bf16_gb300 as dg
    kw = {"la": "row", "lb": "col", **kw}
    opts = {**kw.pop("opts"), **extra}
    for k, v in opts.items():
        dg.gemm_set_option(dg.Option[k], v)
    try:
        c = Case("bf16", **kw, **case_kw)
        st, out = c.run_gpu()
    finally:
        for k in opts:
            dg.gemm_set_option(dg.Option[k], 0)
    assert st == 0, f"status {st}"
    return c, out


@pytest.mark.parametrize("name", sorted(DOUBLE_K_CASES))
def test_exact_double_k(name):
    c, out = _double_k_run(DOUBLE_K_CASES[name], {}, values="ints", seed=901)
    assert c.plan["block_k"] == 128 and c.plan["cta_pair"] == 2, c.plan
    assert np.array_equal(c.result(out), c.oracle_full())
    assert c.untouched_padding(out)
    one, out1 = _double_k_run(DOUBLE_K_CASES[name], {"DOUBLE_K": 1}, values="ints", seed=901)
    assert one.plan["block_k"] == 64
    assert np.array_equal(out.view(np.uint8), out1.view(np.uint8))


def test_double_k_bias_gelu_matches_one_block():
    kw = dict(M=1100, N=1304, K=1024, opts={"CTA_PAIR": 3})
    c, out = _double_k_run(kw, {}, c_dtype="bf16", bias=True, act="gelu_tanh", seed=902)
    assert c.plan["block_k"] == 128, c.plan
    check_close(c, c.result(out), c.oracle_full())
    _, out1 = _double_k_run(kw, {"DOUBLE_K": 1}, c_dtype="bf16", bias=True, act="gelu_tanh",
                            seed=902)
    assert np.array_equal(out.view(np.uint8), out1.view(np.uint8))


# MN-major operands (row-major B, column-major A): every layout pair, even and
# odd K-block counts, K ragged inside its last block (MN-major only), batches
# with per-entry operands, an operand copied for alignment, 128-wide tiles
MN_DOUBLE_K_CASES = {
    "rr_even": dict(M=600, N=700, K=640, la="row", lb="row"),
    "rr_odd_bn128": dict(M=600, N=700, K=320, la="row", lb="row", opts={"BLOCK_N": 128}),
    "cc_odd": dict(M=600, N=700, K=1088, la="col", lb="col"),
    "cr_ragged_k": dict(M=600, N=700, K=1000, la="col", lb="row"),
    "cr_ragged_k_bn128": dict(M=520, N=332, K=777, la="col", lb="row", opts={"BLOCK_N": 128}),
    "rr_many_tiles": dict(M=1100, N=1304, K=1088, la="row", lb="row"),
    "cr_batched": dict(M=300, N=400, K=520, batch=3, la="col", lb="row"),
    "cc_broadcast_b": dict(M=300, N=400, K=512, batch=2, la="col", lb="col", broadcast_b=True),
    "rr_packed_b": dict(M=520, N=600, K=704, la="row", lb="row", pads=(0, 1, 0)),
    "rr_bn256": dict(M=600, N=704, K=640, la="row", lb="row", opts={"BLOCK_N": 256}),
    "cr_bn256_ragged_k": dict(M=520, N=768, K=1000, la="col", lb="row", opts={"BLOCK_N": 256}),
}


@pytest.mark.parametrize("name", sorted(MN_DOUBLE_K_CASES))
def test_exact_double_k_mn_major(name):
    # CTA pairs forced, and split_k = 1 so that no split or stream-K pieces
    # take the plan off whole units
    kw = dict(MN_DOUBLE_K_CASES[name], split_k=1)
    kw["opts"] = {"CTA_PAIR": 3, **kw.get("opts", {})}
    c, out = _double_k_run(kw, {}, values="ints", seed=903)
    a_mn, b_mn = kw["la"] == "col", kw["lb"] == "row"
    k_major_ok = kw["K"] % 64 == 0 and (kw.get("batch", 1) == 1)
    expect = 128 if (a_mn or k_major_ok) and (b_mn or k_major_ok or kw.get("broadcast_b")) \
        else 64
    assert c.plan["block_k"] == expect and c.plan["cta_pair"] == 2, c.plan
    assert np.array_equal(c.result(out), c.oracle_full())
    assert c.untouched_padding(out)
    one, out1 = _double_k_run(kw, {"DOUBLE_K": 1}, values="ints", seed=903)
    assert one.plan["block_k"] == 64
    assert np.array_equal(out.view(np.uint8), out1.view(np.uint8))


def test_double_k_mn_major_bias_gelu_bf16_matches_one_block():
    kw = dict(M=1100, N=1304, K=1000, la="row", lb="row", opts={"CTA_PAIR": 3})
    c, out = _double_k_run(kw, {}, c_dtype="bf16", bias=True, act="gelu_tanh", seed=904)
    assert c.plan["block_k"] == 64, c.plan        # K-major A with a ragged K: one block
    kw = dict(kw, K=1024)
    c, out = _double_k_run(kw, {}, c_dtype="bf16", bias=True, act="gelu_tanh", seed=904)
    assert c.plan["block_k"] == 128, c.plan
    check_close(c, c.result(out), c.oracle_full())
    _, out1 = _double_k_run(kw, {"DOUBLE_K": 1}, c_dtype="bf16", bias=True, act="gelu_tanh",
                            seed=904)
    assert np.array_equal(out.view(np.uint8), out1.view(np.uint8))


# The split form on CTA pairs with two K blocks per load: pieces start and end
# on whole two-block steps (an odd count of K blocks ends with a step whose
# partner block lies past K).  4 CTA pairs, 9 units of 256 x 256: a last wave of
# one unit cut into 4 pieces.
SK_TWO_BLOCK_CASES = {
    "k_major_odd_blocks": dict(la="row", lb="col", K=1088),      # 17 blocks
    "mn_major_ragged_k": dict(la="col", lb="row", K=1000),       # 16 blocks, last one 40 deep
    "rr_odd_blocks": dict(la="row", lb="row", K=704),            # 11 blocks
}


@pytest.mark.parametrize("name", sorted(SK_TWO_BLOCK_CASES))
def test_exact_stream_k_split_pieces_two_k_blocks(name):
    kw = dict(SK_TWO_BLOCK_CASES[name])
    K = kw.pop("K")
    opts = {"STREAM_K": 3, "CTA_PAIR": 3, "MAX_CTAS": 8, "BLOCK_N": 256}
    c, out = _double_k_run(dict(M=700, N=600, K=K, opts=opts, **kw), {}, values="ints",
                           seed=905)
    assert c.plan["stream_k"] == 2 and c.plan["block_k"] == 128, c.plan
    assert np.array_equal(c.result(out), c.oracle_full())
    assert c.untouched_padding(out)
    one, out1 = _double_k_run(dict(M=700, N=600, K=K, opts=opts, **kw), {"DOUBLE_K": 1},
                              values="ints", seed=905)
    assert one.plan["stream_k"] == 2 and one.plan["block_k"] == 64, one.plan
    assert np.array_equal(out.view(np.uint8), out1.view(np.uint8))


# The operand copy (2-byte loads, 16-byte stores) at every base offset of 0-7
# elements, rows of one 8-element group or less and of many, pitches that put
# later rows at other offsets.
@pytest.mark.parametrize("off", range(8))
@pytest.mark.parametrize("shape", [(37, 70, 45), (130, 300, 1000), (64, 9, 7)])
def test_exact_operand_copy_offsets(off, shape):
    M, N, K = shape
    c = run_exact(Case("bf16", M, N, K, la="row", lb="row", values="ints", pads=(1, 3, 0),
                       offsets=(off, 7 - off, 0), seed=1601 + off))
    assert c.plan["pack_a"] + c.plan["pack_b"] >= 1, c.plan


# Operands copied for alignment before the GEMM (A, B, both, batched per
# entry, a broadcast B), each GEMM launched as its copy's programmatic
# dependent: exact against the oracle, and byte-identical to plain stream
# order (GEMM_OPT_OVERLAP_COPY = 1).
OVERLAP_CASES = {
    "copied_a": dict(M=300, N=520, K=200, pads=(3, 0, 0)),
    "copied_b_row_major": dict(M=700, N=600, K=1000, lb="row", pads=(0, 1, 0)),
    "copied_both_col_major": dict(M=520, N=300, K=330, la="col", lb="col", pads=(5, 3, 0)),
    "batched_copied": dict(M=130, N=200, K=90, batch=3, pads=(1, 3, 0)),
    "broadcast_b_copied": dict(M=260, N=200, K=150, batch=2, broadcast_b=True, pads=(0, 1, 0)),
}


@pytest.mark.parametrize("name", sorted(OVERLAP_CASES))
def test_exact_overlapped_operand_copy(name):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(OVERLAP_CASES[name])
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    outs = []
    for overlap in (0, 1):
        dg.gemm_set_option(dg.Option.OVERLAP_COPY, overlap)
        try:
            c = Case("bf16", M, N, K, values="ints", seed=1401, **kw)
            st, out = c.run_gpu()
        finally:
            dg.gemm_set_option(dg.Option.OVERLAP_COPY, 0)
        assert st == 0 and c.plan["pack_a"] + c.plan["pack_b"] >= 1, c.plan
        assert np.array_equal(c.result(out), c.oracle_full()), (c.plan, overlap)
        assert c.untouched_padding(out)
        outs.append(out)
    assert np.array_equal(outs[0].view(np.uint8), outs[1].view(np.uint8))


# Epilogue form 3: whole 256-wide pair tiles whose output takes plain stores
# run the epilogue on eight warps, two per tensor-memory lane quarter, each
# writing half of the columns.  fp32 rows 4, 8 and 12 bytes past a 16-byte
# multiple, 16-bit outputs, a column-major C, beta * C, ragged M and N, a
# batch with an unaligned C stride, a copied operand: bit-exact against the
# oracle and byte-identical to four warps (GEMM_OPT_EPILOGUE_WARPS = 4).
EPI8_CASES = {
    "f32_ldc_1_mod_4": dict(M=700, N=601, K=1000),
    "f32_ldc_2_mod_4": dict(M=520, N=770, K=512),
    "f32_ldc_3_mod_4": dict(M=600, N=515, K=384),
    "bf16_odd_ldc": dict(M=520, N=601, K=512, c_dtype="bf16", values="uniform"),
    "col_major_c": dict(M=600, N=520, K=256, lc="col"),
    "beta_f32": dict(M=520, N=601, K=512, beta=2.0, c_values="ints"),
    "ragged_m_n": dict(M=257, N=259, K=200),
    "batched": dict(M=300, N=257, K=128, batch=2),
    "copied_b": dict(M=700, N=601, K=1000, lb="row"),
}


def _epi8_run(name, warps, **case_kw):
    import dense_gemm_bf16_gb300 as dg
    kw = dict(EPI8_CASES[name])
    kw.setdefault("values", "ints")
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    opts = {"CTA_PAIR": 3, "BLOCK_N": 256, "EPILOGUE_WARPS": warps}
    for k, v in opts.items():
        dg.gemm_set_option(dg.Option[k], v)
    try:
        # split_k = 1: whole tiles (no automatic split or stream-K pieces)
        c = Case("bf16", M, N, K, seed=1501, split_k=1, **kw, **case_kw)
        st, out = c.run_gpu()
    finally:
        for k in opts:
            dg.gemm_set_option(dg.Option[k], 0)
    assert st == 0, f"status {st}"
    return c, out


@pytest.mark.parametrize("name", sorted(EPI8_CASES))
def test_exact_eight_epilogue_warps(name):
    c, out = _epi8_run(name, 0)
    assert c.plan["fast_epilogue"] == 3 and c.plan["cta_pair"] == 2, c.plan
    ref = c.oracle_full()
    if c.c_dtype == "f32":
        assert np.array_equal(c.result(out), ref), c.plan
    else:
        check_close(c, c.result(out), ref)
    assert c.untouched_padding(out)
    four, out4 = _epi8_run(name, 4)
    assert four.plan["fast_epilogue"] == 0, four.plan
    assert np.array_equal(out.view(np.uint8), out4.view(np.uint8))


def test_eight_epilogue_warps_epilogue_terms():
    c, out = _epi8_run("f32_ldc_1_mod_4", 0, alpha=0.75, bias=True, act="gelu_tanh")
    assert c.plan["fast_epilogue"] == 3, c.plan
    check_close(c, c.result(out), c.oracle_full())
    c, out = _epi8_run("col_major_c", 0, bias=True, row_bias=True, act="relu", alpha=1.5)
    assert c.plan["fast_epilogue"] == 3, c.plan
    check_close(c, c.result(out), c.oracle_full())


def test_copied_operand_calls_back_to_back():
    # B with 601-element rows is copied into the workspace before each GEMM,
    # which is launched as the copy's programmatic dependent.  Three calls on
    # one stream with no host sync between them, each with new B values in the
    # same workspace: each result must be its own inputs' (a GEMM that read the
    # copy before it completed would see the previous call's B).  Then the same
    # with the overlap off, byte for byte.
    import dense_gemm_bf16_gb300 as dg
    import datagen
    import oracle
    dev = torch.device("cuda:0")
    M, N, K = 700, 601, 1000
    args0 = [0, 1, M, N, K, None, K, 0, 0, None, N, 0, 0, None, N, 0, 0, 2, 1.0, 0.0, None, 0, 0]
    st, plan = dg.gemm_plan_query(*args0[:5], 1 << 20, K, 0, 0, 1 << 20, N, 0, 0, 1 << 20, N, 0, 0,
                                  2, 1.0, 0.0, None, 0, 0, 1 << 40)
    assert st == 0 and plan.pack_b == 1 and plan.launches == 2, plan.as_dict()
    ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev)
    outs = {}
    for overlap in (0, 1):
        assert dg.gemm_set_option(dg.Option.OVERLAP_COPY, overlap) == 0
        try:
            jobs = []
            for seed in (98001, 98011, 98021):
                a = datagen.to_bf16_bits(datagen.small_ints(seed, (M, K), -4, 4))
                b = datagen.to_bf16_bits(datagen.small_ints(seed + 1, (K, N), -4, 4))
                dA = torch.from_numpy(a.view(np.int16)).to(dev)
                dB = torch.from_numpy(b.view(np.int16)).to(dev)
                dC = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
                jobs.append((a, b, dA, dB, dC))
            torch.cuda.synchronize()
            s = torch.cuda.current_stream().cuda_stream
            for a, b, dA, dB, dC in jobs:
                args = list(args0)
                args[5], args[9], args[13] = dA.data_ptr(), dB.data_ptr(), dC.data_ptr()
                assert dg.gemm_batched(*args, ws.data_ptr(), ws.numel(), s) == 0
            torch.cuda.synchronize()
        finally:
            dg.gemm_set_option(dg.Option.OVERLAP_COPY, 0)
        assert dg.gemm_check_device_status(None) == 0
        outs[overlap] = [dC.cpu().numpy() for *_, dC in jobs]
        for a, b, *_, dC in jobs:
            ref = oracle.gemm(oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K,
                                             A=a.reshape(-1), B=b.reshape(-1), lda=K, ldb=N))[0]
            assert np.array_equal(dC.cpu().numpy().astype(np.float64), ref), overlap
    for x, y in zip(outs[0], outs[1]):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_stream_k_split_two_k_blocks_bias_gelu():
    opts = {"STREAM_K": 3, "CTA_PAIR": 3, "MAX_CTAS": 8, "BLOCK_N": 256}
    c, out = _double_k_run(dict(M=700, N=600, K=1024, opts=opts), {}, c_dtype="bf16",
                           bias=True, act="gelu_tanh", seed=906)
    assert c.plan["stream_k"] == 2 and c.plan["block_k"] == 128, c.plan
    check_close(c, c.result(out), c.oracle_full())


# The automatic split-K balanced over every CTA (the contiguous form with no
# whole units first): on 8 CTAs a few tiles' K steps are dealt in equal ranges,
# so one tile spans up to four CTAs and its first piece adds the partials of
# every later one, in order.  Forced contiguous form on CTA pairs likewise.
BALANCED_CASES = {
    "3_tiles_8_ctas": dict(M=384, N=128, K=4096, opts={"MAX_CTAS": 8}),
    "mn_major_ragged_k": dict(M=384, N=100, K=3000, la="col", lb="row", opts={"MAX_CTAS": 8}),
    "swap_ab_8_tiles_16_ctas": dict(M=16, N=1000, K=4096, pads=(0, 0, 1), opts={"MAX_CTAS": 16}),
    "pairs_contiguous_long_spans": dict(M=700, N=600, K=2048, lb="col",
                                        opts={"STREAM_K": 2, "CTA_PAIR": 3, "MAX_CTAS": 8,
                                              "BLOCK_N": 256}),
}


@pytest.mark.parametrize("name", sorted(BALANCED_CASES))
def test_exact_contiguous_form_spans_several_ctas(name):
    kw = dict(BALANCED_CASES[name])
    for dk in (0, 1):   # two K blocks per load where the plan takes them, then one
        c, out = _double_k_run(kw, {"DOUBLE_K": dk}, values="ints", seed=907)
        assert c.plan["stream_k"] == 1, c.plan
        if dk == 1:
            assert c.plan["block_k"] == 64
        assert np.array_equal(c.result(out), c.oracle_full()), (c.plan, dk)
        assert c.untouched_padding(out)
        if dk == 0:
            first, out0 = c, out
    assert np.array_equal(out0.view(np.uint8), out.view(np.uint8))


def test_contiguous_form_epilogue():
    kw = dict(M=384, N=100, K=3000, la="col", lb="row", opts={"MAX_CTAS": 8})
    c, out = _double_k_run(kw, {}, c_dtype="bf16", beta=0.5, bias=True, act="gelu_tanh",
                           seed=908)
    assert c.plan["stream_k"] == 1, c.plan
    check_close(c, c.result(out), c.oracle_full())


# ---------------------------------------------------------------- 256 x 512 pair tiles

@pytest.fixture
def wide_tile():
    import dense_gemm_bf16_gb300 as dg
    dg.gemm_set_option(dg.Option.WIDE_TILE, 2)
    dg.gemm_set_option(dg.Option.CTA_PAIR, 3)
    yield
    dg.gemm_set_option(dg.Option.WIDE_TILE, 0)
    dg.gemm_set_option(dg.Option.CTA_PAIR, 0)


# N = 700 leaves the second 512-wide tile mostly past the edge; M = 600 a
# partial 256-row block; K = 1000 a ragged last K block
@pytest.mark.parametrize("la", ["row", "col"])
@pytest.mark.parametrize("lb", ["row", "col"])
def test_exact_wide_tile_layouts(wide_tile, la, lb):
    c = run_exact(Case("bf16", 600, 700, 1000, la=la, lb=lb, values="ints", seed=601))
    assert c.plan["block_n"] == 512 and c.plan["cta_pair"] == 2, c.plan


def test_exact_wide_tile_batched_broadcast(wide_tile):
    c = run_exact(Case("bf16", 300, 1100, 320, batch=3, broadcast_b=True, values="ints",
                       seed=602))
    assert c.plan["block_n"] == 512


@pytest.mark.parametrize("beta", [0.0, 0.5])
def test_wide_tile_epilogue(wide_tile, beta):
    c = run_close(Case("bf16", 520, 1536, 640, c_dtype="bf16", alpha=0.5, beta=beta, bias=True,
                       act="gelu_tanh", seed=603))
    assert c.plan["block_n"] == 512 and c.plan["fast_epilogue"] == (1 if beta == 0.0 else 0)


def test_wide_tile_f16_fp32_out_unaligned_c(wide_tile):
    c = run_close(Case("f16", 512, 1030, 512, c_dtype="f32", bias=True, row_bias=True,
                       act="relu", seed=604))
    assert c.plan["block_n"] == 512
