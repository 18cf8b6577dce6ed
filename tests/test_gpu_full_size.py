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
