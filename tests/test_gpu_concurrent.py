"""Two GEMMs whose plans cut tiles into K pieces, running at the same time on
two streams.  In those plans the piece that finishes a tile waits for the
partials of the others; each launch is cooperative, so all its CTAs are
resident together and a waiting CTA never holds an SM its publishers need,
whatever the other kernel occupies.  Both results must equal the oracle
exactly on sampled outputs (small-integer inputs, fp32 output), and no wait
may have expired."""
import numpy as np
import pytest

import datagen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# name: (M, N, K), options, expected plan stream_k.  Each grid fills the GPU.
CASES = {
    "split_pairs": ((2560, 2560, 16384), {}, 2),
    "contiguous_pairs": ((2560, 2560, 16384), {"STREAM_K": 2}, 1),
    "contiguous_single": ((2560, 2560, 8192), {"STREAM_K": 2, "CTA_PAIR": 1}, 1),
    "spread_split_k": ((256, 256, 65536), {"SPLIT_REDUCE": 2}, 3),
    "atomic_split_k": ((256, 256, 65536), {}, 4),
}


def _problem(seed, M, N, K, dev):
    a = datagen.to_bf16_bits(datagen.small_ints(seed, (M, K), -2, 2))
    b = datagen.to_bf16_bits(datagen.small_ints(seed + 1, (K, N), -2, 2))
    p = oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K, A=a.reshape(-1),
                       B=b.reshape(-1), lda=K, ldb=N)
    return (p, torch.from_numpy(a.view(np.int16)).to(dev),
            torch.from_numpy(b.view(np.int16)).to(dev))


@pytest.mark.parametrize("name", list(CASES))
def test_two_streams_at_once(name):
    import dense_gemm_bf16_gb300 as dg
    from dense_gemm_bf16_gb300 import Option
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dg.build()
    dg.lib()
    (M, N, K), opts, form = CASES[name]
    dev = torch.device("cuda:0")
    saved = {k: dg.gemm_get_option(Option[k]) for k in opts}
    try:
        for k, v in opts.items():
            assert dg.gemm_set_option(Option[k], v) == 0
        jobs = []
        for seed in (97001, 97011):
            p, dA, dB = _problem(seed, M, N, K, dev)
            dC = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
            args = [0, 1, M, N, K, dA.data_ptr(), K, 0, 0, dB.data_ptr(), N, 0, 0,
                    dC.data_ptr(), N, 0, 0, 2, 1.0, 0.0, None, 0, 0]
            st, plan = dg.gemm_plan_query(*args, 1 << 40)
            assert st == 0 and plan.stream_k == form, plan.as_dict()
            ws = torch.empty(max(int(plan.workspace_bytes), 256), dtype=torch.uint8, device=dev)
            jobs.append((p, dA, dB, dC, args, ws, torch.cuda.Stream(dev)))
        torch.cuda.synchronize()
        # both streams queued back to back, several rounds, no host sync between
        for _ in range(4):
            for p, dA, dB, dC, args, ws, s in jobs:
                assert dg.gemm_batched(*args, ws.data_ptr(), ws.numel(), s.cuda_stream) == 0
        torch.cuda.synchronize()
    finally:
        for k, v in saved.items():
            dg.gemm_set_option(Option[k], v)
    assert dg.gemm_check_device_status(None) == 0
    for n, (p, dA, dB, dC, args, ws, s) in enumerate(jobs):
        got = dC.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        rows = np.array(sorted({0, 1, 127, 128, 255, M // 2, M - 1}))
        cols = np.array(sorted({0, 1, 127, 128, 255, N // 2, N - 1}))
        ii, jj = np.meshgrid(rows, cols, indexing="ij")
        r = datagen.raw64(97100 + n, 2 * 512)
        i = np.concatenate([ii.ravel(), (r[0::2] % np.uint64(M)).astype(np.int64)])
        j = np.concatenate([jj.ravel(), (r[1::2] % np.uint64(N)).astype(np.int64)])
        ref = oracle.gemm_sampled(p, None, i, j)
        assert np.array_equal(got[i, j], ref), (name, n)
