"""Parity at the workloads' full sizes, in the launch configuration bench.py
times: the same inputs (bench.py's own seeded builders) and the same calls.
The oracle computes sampled outputs one by one: every corner, rows and columns
on both sides of tile boundaries, and a counter-chosen random set.  Properties
that hold at any size are checked on every output."""
from __future__ import annotations

import math

import numpy as np
import pytest

import datagen
import oracle

pytestmark = pytest.mark.gpu


def sample_positions(M, N, n_random, seed, batch=1):
    """(b, i, j) index arrays: corners, tile-boundary rows/columns, random."""
    edges_m = sorted({0, 1, 127, 128, 255, 256, M // 2, M - 2, M - 1} & set(range(M)))
    edges_n = sorted({0, 1, 15, 16, 63, 64, 127, 128, 255, 256, N // 2, N - 2, N - 1} & set(range(N)))
    bs, is_, js = [], [], []
    for b in sorted({0, batch - 1}):
        for i in edges_m:
            for j in edges_n:
                bs.append(b)
                is_.append(i)
                js.append(j)
    r = datagen.raw64(seed, 3 * n_random)
    bs += list((r[0::3] % np.uint64(batch)).astype(np.int64))
    is_ += list((r[1::3] % np.uint64(M)).astype(np.int64))
    js += list((r[2::3] % np.uint64(N)).astype(np.int64))
    return np.array(bs), np.array(is_), np.array(js)


def bf16_to_f64(bits):
    return datagen.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16)).astype(np.float64)


def check_16bit(got, ref):
    err = np.abs(got - ref)
    bad = err > 1e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} of {bad.size} samples out of tolerance, worst {err.max():.3g}"


def check_f32(got, ref, scale):
    rel = np.abs(got - ref).max() / scale
    assert rel <= 1e-4, f"normalised max error {rel:.3g} > 1e-4"


# ----------------------------------------------------------------------------- bf16 8192^3

def test_c3_bf16_8192_bias_gelu_full_size():
    """The headline: A row-major, B column-major, bias + GELU(tanh), bf16 out,
    through bench.py's Gemm call (no workspace)."""
    import torch

    import bench
    a, b_cm, bias = bench.c3_host_inputs()
    M, N, K = bench.M, bench.N, bench.K
    dA = torch.from_numpy(a.view(np.int16)).cuda()
    dB = torch.from_numpy(b_cm.view(np.int16)).cuda()
    dbias = torch.from_numpy(bias).cuda()
    dC = torch.empty((M, N), dtype=torch.int16, device="cuda")
    gemm = bench.Gemm(dA, dB, dbias, dC, torch.cuda.current_stream().cuda_stream)
    gemm()
    torch.cuda.synchronize()
    C = dC.cpu().numpy().view(np.uint16)
    # every output: finite and at or above GELU's minimum (about -0.16997 at x = -0.7518)
    vals = bf16_to_f64(C)
    assert np.isfinite(vals).all()
    assert vals.min() >= -0.1701
    _, i, j = sample_positions(M, N, 2048, seed=9001)
    p = oracle.Problem(ab_dtype="bf16", M=M, N=N, K=K, A=a.ravel(), lda=K, la="row",
                       B=b_cm.ravel(), ldb=K, lb="col", c_dtype="bf16", bias=bias,
                       act="gelu_tanh")
    ref = oracle.gemm_sampled(p, None, i, j)
    check_16bit(vals[i, j], ref)


def _c3_layout_call(dA, dB_cm, dC, c_dtype, dbias, epi):
    """One 8192^3 call in the headline's layout (A row-major, B column-major,
    C row-major, no workspace) with the given output type and epilogue;
    returns the plan it ran under."""
    import torch

    import bench
    import dense_gemm_bf16_gb300 as dg
    M, N, K = bench.M, bench.N, bench.K
    args = [0, 1, M, N, K, dA.data_ptr(), K, 0, 0, dB_cm.data_ptr(), K, 1, 0, dC.data_ptr(), N,
            0, 0, c_dtype, 1.0, 0.0, dbias.data_ptr() if dbias is not None else None, epi, 0]
    st, plan = dg.gemm_plan_query(*args, 0)
    assert st == 0
    st = dg.gemm_batched(*args, None, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, dg.gemm_status_string(st)
    return plan.as_dict()


def _planted_zero_gemm_fails(check, got, p):
    """The same check against the oracle run with A = 0 (the GEMM term
    dropped) must fail: the test can see the product."""
    import copy
    zero = copy.copy(p)
    zero.A = np.zeros_like(p.A)
    _, i, j = sample_positions(p.M, p.N, 256, seed=9011)
    ref0 = oracle.gemm_sampled(zero, None, i, j)
    with pytest.raises(AssertionError):
        check(got[i, j], ref0)


def test_c3_layout_scaled_inputs_fp32_out_no_epilogue():
    """The headline's inputs (U(-1,1)/sqrt(K) on both operands) and layout,
    without bias or GELU and with an fp32 output, at the sqrt(K)-normalised
    1e-4 bound.  The product's std is about 1/(3 sqrt(K)) and the bound
    allows 1e-4 of sqrt(K) max|A| max|B| = 1/sqrt(K), so a missing or wrong
    GEMM term fails here where the bias + GELU check cannot see it."""
    import torch

    import bench
    a, b_cm, _ = bench.c3_host_inputs()
    M, N, K = bench.M, bench.N, bench.K
    dA = torch.from_numpy(a.view(np.int16)).cuda()
    dB = torch.from_numpy(b_cm.view(np.int16)).cuda()
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    plan = _c3_layout_call(dA, dB, dC, 2, None, 0)
    # the bench's kernel form: CTA pairs, two K blocks per load, TMA-store epilogue
    assert plan["cta_pair"] == 2 and plan["block_k"] == 128 and plan["fast_epilogue"] == 1, plan
    got = dC.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    _, i, j = sample_positions(M, N, 2048, seed=9005)
    p = oracle.Problem(ab_dtype="bf16", M=M, N=N, K=K, A=a.ravel(), lda=K, la="row",
                       B=b_cm.ravel(), ldb=K, lb="col", c_dtype="f32")
    scale = math.sqrt(K) * bf16_to_f64(a).__abs__().max() * bf16_to_f64(b_cm).__abs__().max()
    check = lambda g, r: check_f32(g, r, scale)   # noqa: E731
    check(got[i, j], oracle.gemm_sampled(p, None, i, j))
    _planted_zero_gemm_fails(check, got, p)


def test_c3_layout_unscaled_inputs_bias_gelu():
    """The headline's call (bias + GELU(tanh), bf16 out, the bench's plan) on
    unscaled U(-1,1) inputs, so that the product (std about sqrt(K/9) = 30)
    dominates the N(0,1) bias: element-wise 1e-2 + 1e-2 |ref|."""
    import torch

    import bench
    M, N, K = bench.M, bench.N, bench.K
    a = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(3, datagen.ROLE_A) + 100, (M, K)))
    b = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(3, datagen.ROLE_B) + 100, (K, N)))
    b_cm = np.ascontiguousarray(b.T)
    del b
    bias = datagen.to_f32(datagen.normal(datagen.seed_for(3, datagen.ROLE_BIAS), (N,)))
    dA = torch.from_numpy(a.view(np.int16)).cuda()
    dB = torch.from_numpy(b_cm.view(np.int16)).cuda()
    dbias = torch.from_numpy(bias).cuda()
    dC = torch.empty((M, N), dtype=torch.int16, device="cuda")
    gemm = bench.Gemm(dA, dB, dbias, dC, torch.cuda.current_stream().cuda_stream)
    assert gemm.plan["cta_pair"] == 2 and gemm.plan["block_k"] == 128, gemm.plan
    gemm()
    torch.cuda.synchronize()
    got = bf16_to_f64(dC.cpu().numpy().view(np.uint16))
    assert np.isfinite(got).all() and got.min() >= -0.1701
    _, i, j = sample_positions(M, N, 2048, seed=9006)
    p = oracle.Problem(ab_dtype="bf16", M=M, N=N, K=K, A=a.ravel(), lda=K, la="row",
                       B=b_cm.ravel(), ldb=K, lb="col", c_dtype="bf16", bias=bias,
                       act="gelu_tanh")
    check_16bit(got[i, j], oracle.gemm_sampled(p, None, i, j))
    _planted_zero_gemm_fails(check_16bit, got, p)


# ----------------------------------------------------------------------------- bench.py rows

def _row(name):
    import torch

    import bench
    fn, flops, nbytes, bound, plan, keep = bench.build_row(name, torch.device("cuda", 0))
    return fn, plan, keep


@pytest.mark.parametrize("name,M,N,K", [("ragged_4097x3001x1000", 4097, 3001, 1000),
                                        ("splitk_256x256x65536", 256, 256, 65536),
                                        ("skinny_16x8192x8192", 16, 8192, 8192)])
def test_c4_boundary_and_skinny_full_size(name, M, N, K):
    """fp32 outputs of the boundary, split-K and skinny workloads."""
    import torch
    fn, plan, keep = _row(name)
    A, B, C = keep[0], keep[1], keep[2]
    fn()
    torch.cuda.synchronize()
    a = A.cpu().numpy().view(np.uint16)
    b = B.cpu().numpy().view(np.uint16)
    got = C.cpu().numpy()
    assert np.isfinite(got).all()
    _, i, j = sample_positions(M, N, 1024, seed=9002 + K)
    p = oracle.Problem(ab_dtype="bf16", M=M, N=N, K=K, A=a.ravel(), lda=K, la="row",
                       B=b.ravel(), ldb=N, lb="row", c_dtype="f32")
    ref = oracle.gemm_sampled(p, None, i, j)
    amax = bf16_to_f64(a).__abs__().max()
    bmax = bf16_to_f64(b).__abs__().max()
    check_f32(got[i, j], ref, math.sqrt(K) * amax * bmax)


@pytest.mark.parametrize("name", ["flat_4096x4096x16", "flat_4096x4096x16_f32"])
def test_flat_small_k_full_size(name):
    """The flat product (K = 16), bf16 and fp32 output: every element against
    the full oracle."""
    import torch
    fn, plan, keep = _row(name)
    A, B, C = keep[0], keep[1], keep[2]
    n, k = 4096, 16
    # no stale value may pass as a result (bf16 bits 0xFFFF are a NaN)
    C.fill_(float("nan") if C.dtype == torch.float32 else -1)
    fn()
    torch.cuda.synchronize()
    a = A.cpu().numpy().view(np.uint16)
    b = B.cpu().numpy().view(np.uint16)
    f32 = name.endswith("f32")
    p = oracle.Problem(ab_dtype="bf16", M=n, N=n, K=k, A=a.ravel(), lda=k, la="row",
                       B=b.ravel(), ldb=n, lb="row", c_dtype="f32" if f32 else "bf16")
    ref = oracle.gemm(p)[0]
    if f32:
        got = C.cpu().numpy().astype(np.float64)
        amax = np.abs(bf16_to_f64(a)).max()
        bmax = np.abs(bf16_to_f64(b)).max()
        check_f32(got, ref, math.sqrt(k) * amax * bmax)
    else:
        check_16bit(bf16_to_f64(C.cpu().numpy().view(np.uint16)), ref)


@pytest.mark.parametrize("name", ["streamk_2560x2560x16384", "streamk_off_2560x2560x16384"])
def test_stream_k_row_full_size(name):
    """2560 x 2560 x 16384, bf16 output, with stream-K cutting the partial
    wave along K and with it switched off, as the bench rows run it."""
    import torch

    import bench
    import dense_gemm_bf16_gb300 as dg
    opts = bench.ROW_OPTIONS.get(name, {})
    saved = {k: dg.gemm_get_option(dg.Option[k]) for k in opts}
    try:
        for k_, v in opts.items():
            assert dg.gemm_set_option(dg.Option[k_], v) == 0
        fn, plan, keep = _row(name)
        assert (plan["stream_k"] == 0) == bool(opts), plan
        A, B, C = keep[0], keep[1], keep[2]
        C.fill_(-1)  # bf16 bits 0xFFFF: a NaN
        fn()
        torch.cuda.synchronize()
    finally:
        for k_, v in saved.items():
            dg.gemm_set_option(dg.Option[k_], v)
    n, k = 2560, 16384
    a = A.cpu().numpy().view(np.uint16)
    b = B.cpu().numpy().view(np.uint16)
    got = bf16_to_f64(C.cpu().numpy().view(np.uint16))
    _, i, j = sample_positions(n, n, 1024, seed=9005)
    p = oracle.Problem(ab_dtype="bf16", M=n, N=n, K=k, A=a.ravel(), lda=k, la="row",
                       B=b.ravel(), ldb=n, lb="row", c_dtype="bf16")
    check_16bit(got[i, j], oracle.gemm_sampled(p, None, i, j))


@pytest.mark.parametrize("name", ["batched_64x1024", "batched_64x1024_bcast"])
def test_c5_batched_full_size(name):
    """alpha 0.5, beta 1 on a bf16 N(0,1) C, per-batch or broadcast B."""
    import torch
    fn, plan, keep = _row(name)
    A, B, C = keep[0], keep[1], keep[2]
    bt, s = 64, 1024
    c0 = C.cpu().numpy().view(np.uint16).copy()
    fn()
    torch.cuda.synchronize()
    got = bf16_to_f64(C.cpu().numpy().view(np.uint16))
    assert np.isfinite(got).all()
    bcast = name.endswith("bcast")
    a = A.cpu().numpy().view(np.uint16).ravel()
    b = B.cpu().numpy().view(np.uint16).ravel()
    bidx, i, j = sample_positions(s, s, 1024, seed=9003, batch=bt)
    p = oracle.Problem(ab_dtype="bf16", M=s, N=s, K=s, A=a, lda=s, la="row", B=b, ldb=s,
                       lb="row", c_dtype="bf16", C0=c0.ravel(), ldc=s, batch=bt,
                       stride_a=s * s, stride_b=0 if bcast else s * s, stride_c=s * s,
                       alpha=0.5, beta=1.0)
    ref = oracle.gemm_sampled(p, bidx, i, j)
    check_16bit(got.reshape(bt, s, s)[bidx, i, j], ref)


def test_c2_sgemm_4096_full_size():
    """fp32 SGEMM 4096^3, alpha 1.5, beta 0.5, through bench.py's call."""
    import torch
    fn, plan, keep = _row("sgemm_4096")
    A, B, C = keep
    n = 4096
    c0 = C.cpu().numpy().copy()
    fn()
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    assert np.isfinite(got).all()
    a = A.cpu().numpy().ravel()
    b = B.cpu().numpy().ravel()
    _, i, j = sample_positions(n, n, 1024, seed=9004)
    p = oracle.Problem(ab_dtype="f32", M=n, N=n, K=n, A=a, lda=n, la="row", B=b, ldb=n,
                       lb="row", c_dtype="f32", C0=c0.ravel(), ldc=n, alpha=1.5, beta=0.5)
    ref = oracle.gemm_sampled(p, None, i, j)
    scale = math.sqrt(n) * 1.5 * np.abs(a).max() * np.abs(b).max() + 0.5 * np.abs(c0).max()
    check_f32(got[i, j], ref, scale)


def test_c1_bf16_256_full():
    """The small workload, every output against the full oracle."""
    import torch

    import dense_gemm_bf16_gb300 as dg
    n = 256
    a = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(1, datagen.ROLE_A), (n, n)))
    b = datagen.to_bf16_bits(datagen.uniform(datagen.seed_for(1, datagen.ROLE_B), (n, n)))
    dA = torch.from_numpy(a.view(np.int16)).cuda()
    dB = torch.from_numpy(b.view(np.int16)).cuda()
    dC = torch.empty((n, n), dtype=torch.int16, device="cuda")
    st = dg.gemm_bf16(n, n, n, dA.data_ptr(), n, 0, dB.data_ptr(), n, 0, dC.data_ptr(), n, 0,
                      0, 1.0, 0.0, None, 0, 0, None, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    got = bf16_to_f64(dC.cpu().numpy().view(np.uint16))
    p = oracle.Problem(ab_dtype="bf16", M=n, N=n, K=n, A=a.ravel(), lda=n, la="row",
                       B=b.ravel(), ldb=n, lb="row", c_dtype="bf16")
    check_16bit(got, oracle.gemm(p)[0])
