"""CUDA-graph capture of calls whose plans cut tiles into K pieces (stream-K in
its contiguous and split forms, on single CTAs and CTA pairs, the spread and
the atomic split-K), and of a call that copies an operand first.  Those pieces
hand partials over through flags that hold the launch's epoch; a graph replays
the epoch it captured, so the library clears the flags inside the graph before
each kernel.  Each case captures one call, then replays
it with two input sets in turn, and every replay must equal the oracle exactly
(small-integer inputs, fp32 output)."""
import numpy as np
import pytest
import torch

import datagen
import dense_gemm_bf16_gb300 as dg
import oracle
from dense_gemm_bf16_gb300 import Option

pytestmark = pytest.mark.gpu

# name: (M, N, K), options during planning and capture, expected plan stream_k
CASES = {
    "contiguous": ((700, 600, 1000), {"STREAM_K": 2, "MAX_CTAS": 8, "CTA_PAIR": 1}, 1),
    "split": ((700, 600, 1000), {"STREAM_K": 3, "MAX_CTAS": 8, "CTA_PAIR": 1}, 2),
    "split_pair_mma": ((700, 600, 1000), {"STREAM_K": 3, "MAX_CTAS": 8, "CTA_PAIR": 3}, 2),
    "spread": ((128, 256, 8192), {"SPLIT_REDUCE": 2}, 3),
    "atomic": ((128, 256, 8192), {}, 4),
    # B's 601-element rows are not 16-byte aligned: the call copies B, and the
    # GEMM is the copy's programmatic dependent (a graph edge of that kind)
    "copied_operand": ((700, 601, 1000), {}, 0),
}


def _input_set(seed, M, N, K, dev):
    a = datagen.to_bf16_bits(datagen.small_ints(seed, (M, K), -4, 4))
    b = datagen.to_bf16_bits(datagen.small_ints(seed + 1, (K, N), -4, 4))
    ref = oracle.gemm(oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K,
                                     A=a.reshape(-1), B=b.reshape(-1), lda=K, ldb=N))[0]
    return (torch.from_numpy(a.view(np.int16)).to(dev),
            torch.from_numpy(b.view(np.int16)).to(dev), ref)


@pytest.mark.parametrize("name", list(CASES))
def test_captured_call_replays_with_fresh_flags(name):
    (M, N, K), opts, form = CASES[name]
    dev = torch.device("cuda:0")
    sets = [_input_set(seed, M, N, K, dev) for seed in (96001, 96011)]
    A = torch.empty(M, K, dtype=torch.int16, device=dev)
    B = torch.empty(K, N, dtype=torch.int16, device=dev)
    C = torch.empty(M, N, dtype=torch.float32, device=dev)
    args = [0, 1, M, N, K, A.data_ptr(), K, 0, 0, B.data_ptr(), N, 0, 0, C.data_ptr(), N, 0, 0,
            2, 1.0, 0.0, None, 0, 0]
    saved = {k: dg.gemm_get_option(Option[k]) for k in opts}
    graph = torch.cuda.CUDAGraph()
    try:
        for k, v in opts.items():
            assert dg.gemm_set_option(Option[k], v) == 0
        st, plan = dg.gemm_plan_query(*args, 1 << 40)
        assert st == 0 and plan.stream_k == form, plan.as_dict()
        assert plan.pack_b == (1 if name == "copied_operand" else 0), plan.as_dict()
        ws = torch.empty(int(plan.workspace_bytes), dtype=torch.uint8, device=dev)
        A.copy_(sets[0][0])
        B.copy_(sets[0][1])
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):   # one uncaptured call first: one-time setup
            assert dg.gemm_batched(*args, ws.data_ptr(), ws.numel(), side.cuda_stream) == 0
        side.synchronize()
        status = []
        with torch.cuda.graph(graph, stream=side):
            status.append(dg.gemm_batched(*args, ws.data_ptr(), ws.numel(), side.cuda_stream))
        assert status == [0]
    finally:
        for k, v in saved.items():
            dg.gemm_set_option(Option[k], v)
    for i in (0, 1, 0, 1):
        A.copy_(sets[i][0])
        B.copy_(sets[i][1])
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(C.cpu().numpy().astype(np.float64), sets[i][2]), (name, i)
    assert dg.gemm_check_device_status(None) == 0
