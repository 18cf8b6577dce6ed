"""gemm_bf16_static_workspace: the bf16 GEMM for callers that cannot allocate
device memory (a host framework that has reserved the device's memory for its
own allocator, a plugin hook whose contract forbids allocation, a loop that
must not enter the allocator).  Its scratch is a library-owned device array,
so the caller passes only inputs and outputs.

Checked through the C ABI on two calls in a row (the array keeps the previous
call's contents) against the oracle on sampled outputs and against gemm_bf16
with a caller workspace, with plans that really use the scratch: an explicit
split-K, an automatic split that has to shrink to fit the array, and an
unaligned operand copied into the array.  A plan too large for the array is
refused before anything is enqueued.  This file is collected last on purpose.
"""
import math

import numpy as np
import pytest

import datagen
import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

UNLIMITED = 1 << 40


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_bf16_gb300 as dg
    dg.build()
    dg.lib()
    return dg


def _inputs(seed, M, N, K, ldb):
    """bf16 A (M x K, row-major), B (K x N, row-major with leading dimension
    ldb), fp32 bias; host bits and device copies."""
    a = datagen.to_bf16_bits(datagen.uniform(seed, (M, K)))
    b = np.zeros((K, ldb), dtype=np.uint16)
    b[:, :N] = datagen.to_bf16_bits(datagen.uniform(seed + 1, (K, N)))
    bias = datagen.to_f32(datagen.normal(seed + 2, (N,)))
    dev = [torch.from_numpy(x.view(np.int16)).cuda() for x in (a, b)]
    return a, b, bias, dev[0], dev[1], torch.from_numpy(bias).cuda()


# bias + ReLU: an activation keeps the automatic split-K off the atomic form,
# whose scratch is only a few flags, so that the plans below need real scratch
def _args(dg, M, N, K, dA, ldb, dB, dC, dbias, split_k):
    return (M, N, K, dA.data_ptr(), K, 0, dB.data_ptr(), ldb, 0, dC.data_ptr(), N, 0,
            int(dg.DType.F32), 1.0, 0.0, dbias.data_ptr(), int(dg.Epi.BIAS_RELU), split_k)


def _plan(dg, M, N, K, ldb, split_k, ws_bytes):
    # planning only inspects the pointers' alignment: 256-aligned stand-ins
    base = 1 << 24
    st, p = dg.gemm_plan_query(0, 1, M, N, K, base, K, 0, 0, base, ldb, 0, 0, base, N, 0, 0, 2,
                               1.0, 0.0, base, int(dg.Epi.BIAS_RELU), split_k, ws_bytes)
    return st, p.as_dict()


def _run_both(dg, M, N, K, ldb, split_k, seed):
    """The same problem through gemm_bf16 (caller workspace) and through the
    entry point without one; returns (host inputs, reference output, output)."""
    a, b, bias, dA, dB, dbias = _inputs(seed, M, N, K, ldb)
    stream = torch.cuda.current_stream().cuda_stream
    out = []
    for fn in ("gemm_bf16", "gemm_bf16_static_workspace"):
        dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        args = _args(dg, M, N, K, dA, ldb, dB, dC, dbias, split_k)
        if fn == "gemm_bf16":
            need = dg.gemm_workspace_size(0, 1, M, N, K, split_k)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
            st = dg.gemm_bf16(*args, ws.data_ptr(), ws.numel(), stream)
        else:
            st = dg.gemm_bf16_static_workspace(*args, stream)
        torch.cuda.synchronize()
        assert st == 0, (fn, dg.gemm_status_string(st))
        out.append(dC.cpu().numpy().astype(np.float64))
    assert dg.gemm_check_device_status(stream) == 0
    return (a, b, bias), out[0], out[1]


def _check_against_oracle(host, got, M, N, K, ldb, seed):
    """Sampled outputs (corners, tile edges, random) against the fp64 oracle,
    at the stated fp32-output tolerance (sqrt(K)-normalised max error)."""
    a, b, bias = host
    rows = sorted({0, 1, 127, 128, M // 2, M - 2, M - 1} & set(range(M)))
    cols = sorted({0, 1, 63, 64, 127, 128, N // 2, N - 2, N - 1} & set(range(N)))
    ii, jj = np.meshgrid(rows, cols, indexing="ij")
    r = datagen.raw64(seed + 77, 2 * 512)
    i = np.concatenate([ii.ravel(), (r[0::2] % np.uint64(M)).astype(np.int64)])
    j = np.concatenate([jj.ravel(), (r[1::2] % np.uint64(N)).astype(np.int64)])
    p = oracle.Problem(ab_dtype="bf16", M=M, N=N, K=K, A=a.ravel(), lda=K, la="row",
                       B=b.ravel(), ldb=ldb, lb="row", c_dtype="f32", bias=bias, act="relu")
    ref = oracle.gemm_sampled(p, None, i, j)
    amax = np.abs(datagen.bf16_bits_to_f32(a)).max()
    bmax = np.abs(datagen.bf16_bits_to_f32(b[:, :N])).max()
    scale = math.sqrt(K) * amax * bmax + np.abs(bias).max()
    assert np.isfinite(got).all()
    assert np.abs(got[i, j] - ref).max() / scale <= 1e-4


def _check_pair(ref, got, K, bias):
    # the entry point against gemm_bf16, at the same fp32-output tolerance
    scale = math.sqrt(K) + float(np.abs(bias).max())
    assert np.abs(got - ref).max() / scale <= 1e-4


def test_static_workspace_explicit_split_twice(dg):
    M, N, K, split = 256, 384, 4096, 8
    st, plan = _plan(dg, M, N, K, N, split, dg.STATIC_WORKSPACE_BYTES)
    assert st == 0 and plan["split_k"] == split and 0 < plan["workspace_bytes"]
    for seed in (101, 202):  # two calls in a row, different data
        host, ref, got = _run_both(dg, M, N, K, N, split, seed)
        _check_pair(ref, got, K, host[2])
        _check_against_oracle(host, got, M, N, K, N, seed)


@pytest.mark.parametrize("M,N,K,ldb", [(1024, 2048, 32768, 2048),   # split-K cut down to fit
                                       (256, 256, 16384, 257)])     # B copied + split-K
def test_static_workspace_automatic_plan_shrinks_to_fit(dg, M, N, K, ldb):
    st, free = _plan(dg, M, N, K, ldb, 0, UNLIMITED)
    assert st == 0
    st, fit = _plan(dg, M, N, K, ldb, 0, dg.STATIC_WORKSPACE_BYTES)
    assert st == 0 and fit["workspace_bytes"] <= dg.STATIC_WORKSPACE_BYTES
    # the plan a free workspace would get needs more than the array holds
    assert free["workspace_bytes"] > dg.STATIC_WORKSPACE_BYTES, free
    assert fit["split_k"] > 1 or fit["stream_k"] > 0, fit   # the scratch is still used
    for seed in (303, 404):
        host, ref, got = _run_both(dg, M, N, K, ldb, 0, seed)
        _check_against_oracle(host, got, M, N, K, ldb, seed)
        # gemm_bf16 got gemm_workspace_size bytes, so its plan may split differently
        _check_pair(ref, got, K, host[2])


def test_static_workspace_refuses_plans_beyond_its_size(dg):
    M, N, K, split = 1024, 1024, 8192, 8   # 8 fp32 partial slices of 4 MiB > the array
    assert split * M * N * 4 > dg.STATIC_WORKSPACE_BYTES
    st, _ = _plan(dg, M, N, K, N, split, dg.STATIC_WORKSPACE_BYTES)
    assert st == dg.Status.ERR_WORKSPACE          # host-only: the planner refuses
    # through the entry point, with buffers of the full problem's size, so that
    # nothing could be read out of bounds even if the refusal were lost
    dA = torch.zeros((M, K), dtype=torch.int16, device="cuda")
    dB = torch.zeros((K, N), dtype=torch.int16, device="cuda")
    dbias = torch.zeros(N, dtype=torch.float32, device="cuda")
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = dg.gemm_bf16_static_workspace(*_args(dg, M, N, K, dA, N, dB, dC, dbias, split), stream)
    torch.cuda.synchronize()
    assert st == dg.Status.ERR_WORKSPACE
    assert torch.isnan(dC).all()                   # nothing was enqueued
