"""The planner without a GPU: with the test-only GEMM_OPT_TEST_SIM_SMS the plan
queries plan for a simulated sm_103 device of 152 SMs (76 co-resident CTA
pairs), and these tests pin the plan of every workload the bench times, the
options that change it, and the workspace rules.  Pointers are stand-in
addresses that planning only checks for alignment."""
import pytest

import dense_gemm_bf16_gb300 as dg
from dense_gemm_bf16_gb300 import Option, Status

BASE = 1 << 24      # 256-byte aligned stand-in address (never dereferenced)
UNLIMITED = 1 << 40


@pytest.fixture(scope="module", autouse=True)
def simulated_device():
    dg.build()
    dg.lib()
    assert dg.gemm_set_option(Option.TEST_SIM_SMS, 152) == Status.OK
    yield
    dg.gemm_set_option(Option.TEST_SIM_SMS, 0)


@pytest.fixture
def options():
    """Sets options for one test and restores their previous values afterwards."""
    saved = []

    def set_(**kw):
        for k, v in kw.items():
            saved.append((Option[k], dg.gemm_get_option(Option[k])))
            assert dg.gemm_set_option(Option[k], v) == Status.OK
    yield set_
    for opt, v in reversed(saved):
        assert dg.gemm_set_option(opt, v) == Status.OK


def plan(M, N, K, *, ab=0, batch=1, la=0, lb=0, lc=0, lda=None, ldb=None, ldc=None, cdt=None,
         alpha=1.0, beta=0.0, epi=0, split_k=0, ws=0, sa=0, sb=0, sc=0, a=BASE, b=BASE, c=BASE):
    lda = lda or (K if la == 0 else M)
    ldb = ldb or (N if lb == 0 else K)
    ldc = ldc or (N if lc == 0 else M)
    cdt = ab if cdt is None else cdt
    bias = BASE if epi & 1 else None
    st, p = dg.gemm_plan_query(ab, batch, M, N, K, a, lda, la, sa, b, ldb, lb, sb, c, ldc, lc, sc,
                               cdt, alpha, beta, bias, epi, split_k, ws)
    assert st == Status.OK, Status(st)
    return p.as_dict()


def headline(**kw):
    # bf16 8192^3, A row-major, B column-major, bias + GELU(tanh), bf16 out, no workspace
    return plan(8192, 8192, 8192, lb=1, epi=3, **kw)


def test_headline_plan():
    p = headline()
    assert p["kernel"] == 1 and p["cta_pair"] == 2 and p["block_n"] == 256
    assert p["block_k"] == 128 and p["stages"] == 3          # two K blocks per load
    assert p["grid"] == 152 and p["group_m"] == 8 and p["launches"] == 1
    assert p["fast_epilogue"] == 1 and p["stream_k"] == 0 and p["workspace_bytes"] == 0
    assert p["swap_ab"] == 0 and p["pack_a"] == 0 and p["pack_b"] == 0


def test_two_k_blocks_per_load_for_mn_major_operands_too(options):
    assert plan(8192, 8192, 8192, epi=3)["block_k"] == 128           # row-major B
    assert plan(8192, 8192, 8192, la=1, lb=1, epi=3)["block_k"] == 128  # column-major A
    assert plan(8192, 8192, 8192, la=1, epi=3)["block_k"] == 128     # both MN-major
    # an MN-major operand needs no whole number of K blocks (rows past K read zeros)
    assert plan(8192, 8192, 8120, la=1, epi=3)["block_k"] == 128
    # a K-major one does: the two-block view is (64 K, rows, K blocks)
    assert plan(8192, 8192, 8120, epi=3)["block_k"] == 64            # A row-major
    assert plan(4097, 3001, 1000, cdt=2, ws=1 << 40)["block_k"] == 64   # the ragged workload
    # batched: MN-major operands keep their batch dimension; a K-major A must be
    # broadcast (one matrix) to take the two-block view
    n = 2048
    assert plan(n, n, n, la=1, batch=4, sa=n * n, sb=n * n, sc=n * n)["block_k"] == 128
    assert plan(n, n, n, batch=4, sa=n * n, sb=n * n, sc=n * n)["block_k"] == 64
    assert plan(n, n, n, batch=4, sa=0, sb=n * n, sc=n * n)["block_k"] == 128
    options(DOUBLE_K=1)
    p = headline()
    assert p["block_k"] == 64 and p["stages"] == 6


def test_headline_options_change_the_plan(options):
    options(CTA_PAIR=1, GROUP_M=4)
    p = headline()
    assert p["cta_pair"] == 0 and p["group_m"] == 4 and p["block_k"] == 128


def test_split_k_row_adds_its_pieces_atomically(options):
    # fp32 C, no activation, 38 pieces per tile: the atomic form, whose scratch
    # is one flag per CTA; CTA pairs (each operand element loaded once per piece)
    p = plan(256, 256, 65536, cdt=2, ws=UNLIMITED)
    assert p["stream_k"] == 4 and p["split_k"] == 1 and p["launches"] == 1
    assert p["grid"] == 152 and p["block_n"] == 128 and p["cta_pair"] == 2
    assert p["workspace_bytes"] == 256 * ((152 * 8 + 255) // 256)
    assert plan(128, 256, 65536, cdt=2, ws=UNLIMITED)["cta_pair"] == 0   # one tile row
    options(CTA_PAIR=1)
    p1 = plan(256, 256, 65536, cdt=2, ws=UNLIMITED)
    assert p1["stream_k"] == 4 and p1["cta_pair"] == 0 and p1["grid"] == 152
    options(CTA_PAIR=0)
    # an activation, or a 16-bit C: the spread reduction
    assert plan(256, 256, 65536, cdt=2, epi=4, ws=UNLIMITED)["stream_k"] == 3
    assert plan(256, 256, 65536, cdt=0, ws=UNLIMITED)["stream_k"] == 3
    options(SPLIT_REDUCE=2)       # fixed order of addition: the spread reduction
    assert plan(256, 256, 65536, cdt=2, ws=UNLIMITED)["stream_k"] == 3
    options(SPLIT_REDUCE=1)
    p2 = plan(256, 256, 65536, cdt=2, ws=UNLIMITED)
    assert p2["stream_k"] == 0 and p2["split_k"] > 4 and p2["launches"] == 2


def test_atomic_split_k_on_request_for_few_pieces(options):
    # 3 tiles' worth of pieces per CTA stay in the balanced form by default;
    # GEMM_OPT_SPLIT_REDUCE = 4 adds them atomically instead
    assert plan(1024, 640, 4096, cdt=2, ws=UNLIMITED)["stream_k"] == 1
    options(SPLIT_REDUCE=4)
    assert plan(1024, 640, 4096, cdt=2, ws=UNLIMITED)["stream_k"] == 4
    assert plan(1024, 640, 4096, cdt=2, epi=4, ws=UNLIMITED)["stream_k"] == 1


def test_split_k_without_workspace_runs_whole_tiles():
    p = plan(256, 256, 65536, cdt=2)
    assert p["split_k"] == 1 and p["stream_k"] == 0 and p["workspace_bytes"] == 0


def test_skinny_row_swaps_and_spreads_k_over_every_cta(options):
    # 64 tiles of 128 x 16 on 152 CTAs, each CTA an equal range of two-block K
    # steps, no whole units first: every piece adds its partial into the fp32
    # C^T (column-major) by TMA reduce-add, whose scratch is one flag per CTA
    p = plan(16, 8192, 8192, cdt=2, ws=UNLIMITED)
    assert p["swap_ab"] == 1 and p["block_n"] == 16 and p["block_k"] == 128
    assert p["stream_k"] == 4 and p["split_k"] == 1 and p["grid"] == 152 and p["launches"] == 1
    assert p["workspace_bytes"] == 256 * ((152 * 8 + 255) // 256)
    # a 16-bit C, or C rows that are not 16-byte aligned: the partials of the
    # pieces go to the piece holding each tile's first step (contiguous form)
    assert plan(16, 8192, 8192, cdt=0, ws=UNLIMITED)["stream_k"] == 1
    assert plan(16, 8190, 8192, cdt=2, ws=UNLIMITED)["stream_k"] == 1
    options(SPLIT_REDUCE=3)   # equal pieces instead: 2 per tile, on 128 CTAs
    q = plan(16, 8192, 8192, cdt=2, ws=UNLIMITED)
    assert q["stream_k"] == 2 and q["grid"] == 128 and q["block_k"] == 128


def test_batched_beta_rows_read_c_by_tma_loads():
    s = 1024
    for sb in (s * s, 0):
        p = plan(s, s, s, batch=64, alpha=0.5, beta=1.0, sa=s * s, sb=sb, sc=s * s)
        # the TMA-store epilogue reading beta * C, on eight warps (16 K blocks)
        assert p["fast_epilogue"] == 4 and p["cta_pair"] == 2 and p["block_k"] == 64
        assert p["stages"] == 4


def test_ragged_row_copies_b_and_stores_with_st_global(options):
    p = plan(4097, 3001, 1000, cdt=2, ws=UNLIMITED)
    assert p["pack_b"] == 1 and p["pack_a"] == 0 and p["launches"] == 2
    # plain stores (3001-float rows) on eight epilogue warps: 64 KB of staging,
    # one pipeline stage fewer
    assert p["fast_epilogue"] == 3 and p["workspace_bytes"] > 0
    assert p["cta_pair"] == 2 and p["block_n"] == 256 and p["stages"] == 5
    options(EPILOGUE_WARPS=4)
    q = plan(4097, 3001, 1000, cdt=2, ws=UNLIMITED)
    assert q["fast_epilogue"] == 0 and q["stages"] == 6
    options(EPILOGUE_WARPS=0)
    # not for C that TMA can store, nor for stream-K pieces or split-K slices
    assert plan(4096, 3008, 1000, cdt=2, ws=UNLIMITED)["fast_epilogue"] == 1
    assert plan(4097, 3001, 1000, cdt=2, ws=UNLIMITED, split_k=2)["fast_epilogue"] != 3
    # B's rows of 3001 bf16 are not 16-byte aligned: TMA cannot read it in place
    st, _ = dg.gemm_plan_query(0, 1, 4097, 3001, 1000, BASE, 1000, 0, 0, BASE, 3001, 0, 0,
                               BASE, 3001, 0, 0, 2, 1.0, 0.0, None, 0, 0, 0)
    assert st == Status.ERR_WORKSPACE


def test_flat_row_keeps_single_cta_tiles():
    p = plan(4096, 4096, 16)
    assert p["cta_pair"] == 0 and p["block_n"] == 256 and p["fast_epilogue"] == 1


def test_stream_k_needs_a_workspace_and_keeps_two_k_blocks(options):
    p = plan(2560, 2560, 16384, lb=1, ws=UNLIMITED)
    assert p["stream_k"] == 2 and p["block_k"] == 128
    # the headline with a workspace: split-form pieces on whole two-block steps
    assert headline(ws=UNLIMITED)["block_k"] == 128
    options(STREAM_K=2)           # the contiguous form's ranges, in two-block steps too
    p = plan(2560, 2560, 16384, lb=1, ws=UNLIMITED)
    assert p["stream_k"] == 1 and p["block_k"] == 128
    p0 = plan(2560, 2560, 16384, lb=1)
    assert p0["stream_k"] == 0 and p0["block_k"] == 128


def test_sgemm_and_epilogue_only_plans():
    assert plan(4096, 4096, 4096, ab=2, cdt=2, alpha=1.5, beta=0.5)["kernel"] == 2
    assert plan(70, 90, 0, cdt=2, beta=0.5)["kernel"] == 3
    assert plan(70, 90, 64, cdt=2, alpha=0.0, beta=0.5)["kernel"] == 3


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (256, 256, 65536), (128, 256, 8192),
                                   (2560, 2560, 16384), (4097, 3001, 1000)])
def test_exact_reported_workspace_gives_the_same_plan(shape):
    M, N, K = shape
    big = plan(M, N, K, cdt=2, ws=UNLIMITED)
    exact = plan(M, N, K, cdt=2, ws=big["workspace_bytes"])
    assert exact == big


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (256, 256, 65536), (2560, 2560, 16384),
                                   (4097, 3001, 1000), (333, 712, 300)])
@pytest.mark.parametrize("layouts", [(0, 0, 0), (1, 1, 1), (0, 1, 0)])
def test_workspace_size_covers_every_plan(shape, layouts):
    M, N, K = shape
    la, lb, lc = layouts
    need = plan(M, N, K, la=la, lb=lb, lc=lc, cdt=2, ws=UNLIMITED)["workspace_bytes"]
    assert dg.gemm_workspace_size(0, 1, M, N, K, 0) >= need


def test_simulated_device_changes_with_the_sm_count(options):
    options(TEST_SIM_SMS=64)
    p = plan(256, 256, 65536, cdt=2, ws=UNLIMITED)
    assert p["grid"] <= 64 and p["stream_k"] == 4


@pytest.mark.parametrize("ab,cdt", [(0, 0), (1, 1), (1, 2)])
@pytest.mark.parametrize("shape", [(4, 16, 4096, 4096), (64, 1024, 1024, 1024),
                                   (3, 4097, 3001, 1000), (8, 256, 256, 65536)])
def test_workspace_size_covers_batched_plans(ab, cdt, shape):
    bt, M, N, K = shape
    for sb in (K * N, 0):
        need = plan(M, N, K, ab=ab, cdt=cdt, batch=bt, sa=M * K, sb=sb, sc=M * N,
                    ws=UNLIMITED)["workspace_bytes"]
        assert dg.gemm_workspace_size(ab, bt, M, N, K, 0) >= need


# kernel instantiations compiled into the library: (tile width, CTA mode) per epilogue form,
# and the two-K-blocks-per-load form (pairs, TMA-store-only epilogue)
INSTANTIATED = {
    0: {(16, 0), (32, 0), (64, 0), (128, 0), (256, 0), (128, 2), (256, 2), (512, 2)},
    1: {(64, 0), (128, 0), (256, 0), (128, 2), (256, 2), (512, 2)},
    2: {(64, 0), (128, 0), (256, 0), (128, 2), (256, 2)},
    3: {(256, 2)},
    4: {(256, 2)},
}
# (tile width, mode, epilogue form) compiled with two K blocks per load
TWO_K_BLOCKS = {(128, 2, 1), (256, 2, 1), (16, 0, 0), (32, 0, 0), (64, 0, 0), (64, 0, 1),
                (128, 0, 1), (256, 0, 1)}


def _random_calls(n, seed=20261202):
    import random
    rng = random.Random(seed)
    dims_m = [1, 15, 16, 64, 65, 128, 200, 257, 1000, 2560, 4097, 8192]
    dims_n = [1, 8, 16, 100, 128, 256, 384, 1000, 3001, 8192]
    dims_k = [0, 1, 16, 64, 100, 256, 768, 1000, 4096, 8192, 65536]
    dts = [(0, 0), (0, 2), (1, 1), (1, 2), (2, 2)]
    for _ in range(n):
        M, N, K = rng.choice(dims_m), rng.choice(dims_n), rng.choice(dims_k)
        ab, cdt = rng.choice(dts)
        la, lb, lc = rng.randrange(2), rng.randrange(2), rng.randrange(2)
        batch = rng.choice([1, 1, 1, 3, 64])
        sb_bcast = rng.random() < 0.3
        beta = rng.choice([0.0, 0.0, 1.0])
        alpha = rng.choice([1.0, 1.0, 0.5, 0.0])
        epi = rng.choice([0, 1, 3, 5, 7, 9, 11])
        ws = rng.choice([0, UNLIMITED])
        split_k = rng.choice([0, 0, 0, 1, 2, 7])
        yield dict(M=M, N=N, K=K, ab=ab, cdt=cdt, la=la, lb=lb, lc=lc, batch=batch,
                   sa=M * K, sb=0 if sb_bcast else K * N, sc=M * N, alpha=alpha, beta=beta,
                   epi=epi, ws=ws, split_k=split_k)


OPTION_SETS = [
    {}, {"CTA_PAIR": 1}, {"CTA_PAIR": 3}, {"WIDE_TILE": 2},
    {"CTA_PAIR": 3, "WIDE_TILE": 2}, {"SWAP_AB": 1}, {"SWAP_AB": 2}, {"STREAM_K": 1},
    {"STREAM_K": 2}, {"STREAM_K": 3}, {"FAST_EPILOGUE": 1}, {"SPLIT_REDUCE": 1},
    {"SPLIT_REDUCE": 2}, {"BLOCK_N": 16}, {"BLOCK_N": 64}, {"BLOCK_N": 128}, {"DOUBLE_K": 1},
    {"MAX_CTAS": 37}, {"GROUP_M": 1}, {"CTA_PAIR": 3, "EPILOGUE_WARPS": 4},
]


def _opts_id(o):
    return ",".join(f"{k}={v}" for k, v in o.items()) or "defaults"


@pytest.mark.parametrize("opts", OPTION_SETS, ids=_opts_id)
def test_every_plan_names_a_compiled_kernel_and_keeps_its_invariants(options, opts):
    options(**opts)
    n_ctas = opts.get("MAX_CTAS", 152)
    checked = 0
    for kw in _random_calls(1500):
        ws = kw.pop("ws")
        M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
        lda = K if kw["la"] == 0 else M
        ldb = N if kw["lb"] == 0 else K
        ldc = N if kw["lc"] == 0 else M
        bias = BASE if kw["epi"] & 1 else None
        st, p = dg.gemm_plan_query(kw["ab"], kw["batch"], M, N, K, BASE, max(lda, 1), kw["la"],
                                   kw["sa"], BASE, max(ldb, 1), kw["lb"], kw["sb"], BASE,
                                   max(ldc, 1), kw["lc"], kw["sc"], kw["cdt"], kw["alpha"],
                                   kw["beta"], bias, kw["epi"], kw["split_k"], ws)
        ctx = (M, N, K, kw, ws)
        if st == Status.ERR_WORKSPACE:
            assert ws == 0, ctx      # only an operand copy or split-K needs one
            continue
        assert st == Status.OK, (Status(st), ctx)
        p = p.as_dict()
        assert 0 <= p["workspace_bytes"] <= ws, ctx
        # gemm_workspace_size bounds the scratch of any call with these sizes
        assert dg.gemm_workspace_size(kw["ab"], kw["batch"], M, N, K, kw["split_k"]) >= \
            p["workspace_bytes"], (p, ctx)
        if kw["split_k"] == 1:
            assert p["split_k"] == 1 and p["stream_k"] == 0, (p, ctx)
        if kw["ab"] == 2:
            assert p["kernel"] in (2, 3), ctx
        if K == 0 or kw["alpha"] == 0.0:
            assert p["kernel"] == 3, ctx
        if p["kernel"] != 1:
            continue
        checked += 1
        bn, mode, form = p["block_n"], p["cta_pair"], p["fast_epilogue"]
        assert (bn, mode) in INSTANTIATED[form], (p, ctx)
        if opts.get("WIDE_TILE", 0) != 2:     # 256 x 512 tiles measured slower: only on request
            assert bn != 512, (p, ctx)
        assert 1 <= p["grid"] <= n_ctas and p["stages"] >= 2, (p, ctx)
        if mode:
            assert p["grid"] % 2 == 0, (p, ctx)
        if p["block_k"] == 128:
            assert (bn, mode, form) in TWO_K_BLOCKS, (p, ctx)
            # each operand MN-major, or K-major with whole K blocks and one matrix
            for mn, stride in ((kw["la"] == 1, kw["sa"]), (kw["lb"] == 0, kw["sb"])):
                assert mn or (K % 64 == 0 and (kw["batch"] == 1 or stride == 0)), (p, ctx)
            assert p["split_k"] == 1, (p, ctx)
            assert mode == 2 or K > 7 * 64, (p, ctx)    # single CTAs: 8 K blocks at least
        else:
            assert p["block_k"] == 64, (p, ctx)
        if form in (2, 4):
            assert kw["beta"] != 0.0 and kw["cdt"] in (0, 1), (p, ctx)
        if form in (3, 4):           # eight epilogue warps: whole tiles
            assert p["stream_k"] == 0 and p["split_k"] == 1 and p["block_k"] == 64, (p, ctx)
            assert opts.get("EPILOGUE_WARPS", 0) == 0, (p, ctx)
        if form == 4:
            assert K <= 32 * 64, (p, ctx)
        if p["stream_k"] == 3:       # the spread reduction runs on single CTAs only
            assert mode == 0 and p["workspace_bytes"] > 0, (p, ctx)
            assert p["launches"] == 1 + p["pack_a"] + p["pack_b"], (p, ctx)   # no reduction pass
        if p["stream_k"]:
            assert p["split_k"] == 1 and p["workspace_bytes"] > 0, (p, ctx)
        if p["split_k"] > 1:
            assert p["launches"] >= 2 and p["workspace_bytes"] > 0, (p, ctx)
        assert p["launches"] >= 1 + p["pack_a"] + p["pack_b"], (p, ctx)
    assert checked > 500


def test_more_work_units_than_32_bits_count_is_unsupported():
    # 2^30 batch entries of 256 x 16: two tiles each, 2^31 units in all
    bt = 1 << 30
    st, _ = dg.gemm_plan_query(0, bt, 256, 16, 16, BASE, 16, 0, 256 * 16, BASE, 16, 0, 0,
                               BASE, 16, 0, 256 * 16, 2, 1.0, 0.0, None, 0, 0, 0)
    assert st == Status.ERR_UNSUPPORTED
    st, p = dg.gemm_plan_query(0, bt // 2, 256, 16, 16, BASE, 16, 0, 256 * 16, BASE, 16, 0, 0,
                               BASE, 16, 0, 256 * 16, 2, 1.0, 0.0, None, 0, 0, 0)
    assert st == Status.OK and p.kernel == 1


# The automatic stream-K choice against the shapes it was measured on (bf16,
# A row-major, B column-major, a workspace given): the split form where it ran
# faster than whole tiles, whole tiles where it ran slower.
STREAM_K_MEASURED = [
    ((2560, 2560, 16384), 2),   # +25 %
    ((4096, 4096, 8192), 2),    # +6 %
    ((4096, 4096, 4096), 2),    # +3 %
    ((5120, 5120, 4096), 2),    # +2 %
    ((4096, 4096, 2048), 0),    # -3 % when forced
    ((6144, 4096, 4096), 0),    # -18 % when forced
]


@pytest.mark.parametrize("shape,form", STREAM_K_MEASURED)
def test_auto_stream_k_follows_the_measurements(shape, form):
    M, N, K = shape
    p = plan(M, N, K, lb=1, ws=UNLIMITED)
    assert p["stream_k"] == form and p["cta_pair"] == 2, p
    if form == 0:
        assert plan(M, N, K, lb=1)["stream_k"] == 0


@pytest.mark.parametrize("K,pair", [(128, 0), (256, 0), (512, 0), (704, 0), (768, 2), (1024, 2),
                                    (2048, 2)])
def test_cta_pairs_start_at_twelve_k_blocks(K, pair):
    # measured on 4096 x 4096 x K: paired tiles ran 10-25 % slower for K <= 256,
    # even at 512 and 5-20 % faster from 1024; the threshold is 12 K blocks
    p = plan(4096, 4096, K, lb=1)
    assert p["cta_pair"] == pair and p["block_n"] == 256, p


def splan(M, N, K, a, b, c, *, ab=0, cdt=2, batch=1, alpha=1.0, beta=0.0, ws=UNLIMITED,
          split_k=0):
    """gemm_strided_plan_query with (row stride, column stride, batch stride) per matrix."""
    st, p = dg.gemm_strided_plan_query(ab, batch, M, N, K, BASE, *a, BASE, *b, BASE, *c, cdt,
                                       alpha, beta, None, 0, split_k, ws)
    return st, p.as_dict()


def test_strided_plan_of_dense_strides_is_the_batched_plan():
    M, N, K = 2560, 2560, 16384
    st, sp = splan(M, N, K, (K, 1, 0), (1, K, 0), (N, 1, 0))     # B column-major
    assert st == Status.OK
    assert sp == plan(M, N, K, lb=1, ws=UNLIMITED)


def test_strided_plan_counts_the_copies():
    M, N, K = 300, 256, 200     # dense rows of 400 and 512 bytes: TMA reads them in place
    st, dense = splan(M, N, K, (K, 1, 0), (N, 1, 0), (N, 1, 0))
    assert st == Status.OK and dense["pack_a"] == 0 and dense["pack_b"] == 0
    # A with a step of 2 along K: gathered into a copy, one more launch
    st, p = splan(M, N, K, (2 * K, 2, 0), (N, 1, 0), (N, 1, 0))
    assert st == Status.OK and p["pack_a"] == 1 and p["pack_b"] == 0
    assert p["launches"] == dense["launches"] + 1
    assert p["workspace_bytes"] > dense["workspace_bytes"]
    # C interleaved (column stride 2): computed densely, then scattered; with
    # beta != 0 also gathered first
    st, pc = splan(M, N, K, (K, 1, 0), (N, 1, 0), (2 * N, 2, 0))
    assert st == Status.OK and pc["launches"] == dense["launches"] + 1
    st, pcb = splan(M, N, K, (K, 1, 0), (N, 1, 0), (2 * N, 2, 0), beta=1.0)
    assert st == Status.OK and pcb["launches"] >= dense["launches"] + 2
    # with alpha == 0 A and B are never read, so they are not gathered either
    st, p0 = splan(M, N, K, (2 * K, 2, 0), (N, 1, 0), (N, 1, 0), alpha=0.0, beta=1.0)
    assert st == Status.OK and p0["kernel"] == 3


def test_strided_plan_workspace_rules():
    M, N, K = 300, 260, 200
    a, b, c = (2 * K, 2, 0), (N, 1, 0), (N, 1, 0)
    st, p = splan(M, N, K, a, b, c)
    assert st == Status.OK
    need = p["workspace_bytes"]
    assert dg.gemm_strided_workspace_size(0, 2, 1, M, N, K, *a, *b, *c, 0) >= need
    st, exact = splan(M, N, K, a, b, c, ws=need)
    assert st == Status.OK and exact == p
    st, _ = splan(M, N, K, a, b, c, ws=need - 256)
    assert st == Status.ERR_WORKSPACE
    st, _ = splan(M, N, K, a, b, c, ws=0)
    assert st == Status.ERR_WORKSPACE


def test_strided_plan_rejects_what_gemm_strided_rejects():
    M, N, K = 64, 64, 64
    st, _ = splan(M, N, K, (K, 1, 0), (N, 1, 0), (0, 1, 0))          # rows of C repeated
    assert st == Status.ERR_INVALID_ARG
    st, _ = splan(M, N, K, (-K, 1, 0), (N, 1, 0), (N, 1, 0))         # negative stride
    assert st == Status.ERR_INVALID_ARG
    st, _ = splan(M, N, K, (1 << 60, 1, 0), (N, 1, 0), (N, 1, 0))    # span too large
    assert st == Status.ERR_INVALID_ARG


def test_wide_tiles_on_request(options):
    options(WIDE_TILE=2)
    p = headline()
    assert p["block_n"] == 512 and p["cta_pair"] == 2 and p["block_k"] == 64   # one K block
    q = plan(4096, 256, 4096, lb=1)                # N < 512: the 256-wide pair tile stays
    assert q["block_n"] != 512


def test_the_multicast_pair_value_is_refused():
    """GEMM_OPT_CTA_PAIR = 2 named CTA pairs that shared B through multicast TMA
    loads; the library has no such load any more, and the value is refused
    without changing the option."""
    before = dg.gemm_get_option(Option.CTA_PAIR)
    assert dg.gemm_set_option(Option.CTA_PAIR, 2) == Status.ERR_INVALID_ARG
    assert dg.gemm_get_option(Option.CTA_PAIR) == before
    for v in (0, 1, 3):
        assert dg.gemm_set_option(Option.CTA_PAIR, v) == Status.OK
    assert dg.gemm_set_option(Option.CTA_PAIR, before) == Status.OK


def test_no_source_names_a_multicast_load():
    """No TMA load in the library's sources is multicast (the commit arrive
    that signals both CTAs of a pair is an mbarrier signal, not a load)."""
    import pathlib
    csrc = pathlib.Path(dg.__file__).parent / "csrc"
    for f in sorted(csrc.iterdir()):
        if f.suffix not in (".cu", ".cuh", ".h"):
            continue
        for n, line in enumerate(f.read_text().splitlines(), 1):
            if "multicast::cluster" in line:
                assert "cp.async" not in line and "tcgen05.commit" in line, (f.name, n, line)
