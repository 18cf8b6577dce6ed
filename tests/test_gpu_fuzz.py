"""Seeded random sweep of small problems against the oracle, through the C ABI:
ragged shapes, every layout, bf16 and fp16, fp32 or 16-bit outputs, padded
leading dimensions, pointer offsets that defeat TMA alignment, batches with
and without a broadcast B, explicit and automatic split-K, alpha, beta, a bias
along columns or rows, and every activation.  Half the draws run under the
default plan, half under forced options (CTA pairs, wide tiles, stream-K on a
few CTAs) so that the less common kernels meet the same mix.  Cases whose
arithmetic is exact (small-integer inputs, fp32 output, no beta, bias or
smooth activation) must match bit for bit; the rest within the stated
tolerance.  Every byte of C outside the matrix must keep its poison."""
import random

import numpy as np
import pytest

from gemm_case import Case, check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_DRAWS = 64
FORCED = [{"CTA_PAIR": 3}, {"CTA_PAIR": 3, "WIDE_TILE": 2}, {"STREAM_K": 3, "MAX_CTAS": 8},
          {"STREAM_K": 2, "MAX_CTAS": 8}, {"FAST_EPILOGUE": 1}, {"SWAP_AB": 2}]


def draw(i):
    r = random.Random(7000 + i)
    forced = i % 2 == 1
    ab = r.choice(["bf16", "f16"])
    if forced:   # shapes with several tile pairs and partial last waves
        M = r.choice([257, 300, 513, 700])
        N = r.choice([200, 256, 600, 700])
        K = r.choice([333, 600, 1000])
    else:
        M = r.choice([1, 2, 15, 64, 65, 127, 129, 200, 300])
        N = r.choice([1, 8, 17, 64, 100, 256, 257, 600])
        K = r.choice([1, 7, 16, 64, 100, 333, 600, 1000])
    batch = r.choice([1, 1, 2, 3])
    exact = r.random() < 0.5
    if exact:    # every fp32 partial sum and the output are integers
        c_dtype, beta, bias, act = "f32", 0.0, False, r.choice(["none", "relu"])
    else:
        c_dtype = r.choice([ab, "f32"])
        beta = r.choice([0.0, 0.5, 1.0])
        bias = r.random() < 0.5
        act = r.choice(["none", "relu", "gelu_tanh", "gelu_erf"])
    kw = dict(batch=batch, la=r.choice(["row", "col"]), lb=r.choice(["row", "col"]),
              lc=r.choice(["row", "col"]), c_dtype=c_dtype,
              pads=tuple(r.choice([0, 0, 1, 8]) for _ in range(3)),
              offsets=tuple(r.choice([0, 0, 0, 1]) for _ in range(3)),
              alpha=r.choice([1.0, 0.5, 2.0]), beta=beta, bias=bias,
              row_bias=bias and r.random() < 0.5, act=act,
              broadcast_b=batch > 1 and r.random() < 0.5, values="ints", seed=500 + i,
              split_k=r.choice([0, 0, 0, 1, 3]))
    opts = FORCED[(i // 2) % len(FORCED)] if forced else {}
    return Case(ab, M, N, K, **kw), exact, opts


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_bf16_gb300 as dg
    dg.build()
    dg.lib()


@pytest.mark.parametrize("i", range(N_DRAWS))
def test_random_problem_matches_the_oracle(i):
    import dense_gemm_bf16_gb300 as dg
    from dense_gemm_bf16_gb300 import Option
    case, exact, opts = draw(i)
    saved = {k: dg.gemm_get_option(Option[k]) for k in opts}
    try:
        for k, v in opts.items():
            assert dg.gemm_set_option(Option[k], v) == 0
        st, out = case.run_gpu()
    finally:
        for k, v in saved.items():
            dg.gemm_set_option(Option[k], v)
    assert st == 0, (st, getattr(case, "plan", None))
    got, ref = case.result(out), case.oracle_full()
    if exact:
        assert np.array_equal(got, ref), (np.abs(got - ref).max(), case.plan, opts)
    else:
        check_close(case, got, ref)
    assert case.untouched_padding(out), (case.plan, opts)
