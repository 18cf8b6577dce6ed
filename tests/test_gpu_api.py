"""``dense_gemm_bf16_gb300.gemm`` (the tensor-level call) against the oracle:
views read through their own strides (transposed, padded, expanded batch),
the epilogue by name, the output allocated by the call, and the workspace
allocated from the plan.  Small-integer inputs make fp32 results exact."""
import numpy as np
import pytest
import torch

import datagen
import dense_gemm_bf16_gb300 as dg
import oracle

pytestmark = pytest.mark.gpu


def ints(seed, shape, lo=-4, hi=4, dtype=torch.bfloat16):
    return torch.from_numpy(datagen.small_ints(seed, shape, lo, hi).astype(np.float32)).to(dtype)


def bits(t):
    """Storage of a contiguous CPU tensor as the oracle reads it."""
    t = t.contiguous()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.numpy().reshape(-1)


DT = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


def run(A, B, C=None, **kw):
    dev = torch.device("cuda:0")
    out = dg.gemm(A.to(dev), B.to(dev), None if C is None else C.to(dev), **kw)
    torch.cuda.synchronize()
    return out.cpu()


def test_transposed_and_padded_views():
    M, N, K = 300, 260, 200
    A = ints(91001, (M, 256))[:, :K]              # padded rows: ld 256
    Bt = ints(91002, (N, K))                      # B = Bt.t(): column-major
    out = run(A, Bt.t(), out_dtype=torch.float32)
    p = oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K,
                       A=bits(ints(91001, (M, 256))), B=bits(Bt),
                       strides=((256, 1), (1, K), (N, 1)))
    ref = oracle.gemm(p)[0]
    assert out.shape == (M, N) and out.dtype == torch.float32
    assert np.array_equal(out.numpy().astype(np.float64), ref)


def test_broadcast_batch_row_bias_relu_in_place():
    bt, M, N, K = 4, 128, 136, 96
    A = ints(92001, (bt, M, K))
    B = ints(92002, (K, N))
    C0 = ints(92003, (bt, M, N), dtype=torch.float32)
    bias = ints(92004, (M,), dtype=torch.float32)
    dev = torch.device("cuda:0")
    C = C0.to(dev)
    ret = dg.gemm(A.to(dev), B.to(dev).expand(bt, K, N), C, alpha=2.0, beta=1.0,
                  bias=bias.to(dev), epilogue="row_bias_relu")
    torch.cuda.synchronize()
    assert ret.data_ptr() == C.data_ptr()
    p = oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K, batch=bt,
                       A=bits(A), B=bits(B), C0=bits(C0), stride_a=M * K, stride_b=0,
                       stride_c=M * N, alpha=2.0, beta=1.0, bias=bias.numpy(), act="relu",
                       bias_rows=True, strides=((K, 1), (N, 1), (N, 1)))
    assert np.array_equal(C.cpu().numpy().astype(np.float64), oracle.gemm(p))


def test_long_k_allocates_its_workspace():
    M, N, K = 128, 128, 16384
    A, B = ints(93001, (M, K), -2, 2), ints(93002, (K, N), -2, 2)
    plan = dg.plan(A, B, torch.empty(M, N, dtype=torch.float32))
    assert plan["workspace_bytes"] > 0
    out = run(A, B, out_dtype=torch.float32)
    p = oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K, A=bits(A), B=bits(B),
                       strides=((K, 1), (N, 1), (N, 1)))
    assert np.array_equal(out.numpy().astype(np.float64), oracle.gemm(p)[0])


def test_bf16_output_with_bias_gelu():
    M, N, K = 257, 384, 320
    A = torch.from_numpy(datagen.uniform(94001, (M, K)).astype(np.float32)).to(torch.bfloat16)
    B = torch.from_numpy(datagen.uniform(94002, (K, N)).astype(np.float32)).to(torch.bfloat16)
    bias = torch.from_numpy(datagen.normal(94004, (N,)).astype(np.float32))
    dev = torch.device("cuda:0")
    out = dg.gemm(A.to(dev), B.to(dev), bias=bias.to(dev), epilogue="bias_gelu_tanh",
                  alpha=0.5).cpu()
    p = oracle.Problem(ab_dtype="bf16", c_dtype="bf16", M=M, N=N, K=K, A=bits(A), B=bits(B),
                       alpha=0.5, bias=bias.numpy(), act="gelu_tanh",
                       strides=((K, 1), (N, 1), (N, 1)))
    ref = oracle.gemm(p)[0]
    got = out.float().numpy().astype(np.float64)
    assert out.dtype == torch.bfloat16
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))


def test_fp32_inputs_run_the_cuda_core_sgemm():
    M, N, K = 100, 90, 70
    A = ints(95001, (M, K), dtype=torch.float32)
    B = ints(95002, (K, N), dtype=torch.float32)
    assert dg.plan(A, B, torch.empty(M, N))["kernel"] == 2
    out = run(A, B, alpha=1.5)
    p = oracle.Problem(ab_dtype="f32", c_dtype="f32", M=M, N=N, K=K, A=bits(A), B=bits(B),
                       alpha=1.5, strides=((K, 1), (N, 1), (N, 1)))
    assert np.array_equal(out.numpy().astype(np.float64), oracle.gemm(p)[0])


def test_strided_views_run_through_gemm_strided():
    M, N, K = 96, 80, 72
    base_a = ints(96001, (M, 2 * K))
    row = ints(96002, (1, N))
    base_b = row.expand(K, N)                     # every row of B the same
    dev = torch.device("cuda:0")
    out = dg.gemm(base_a.to(dev)[:, ::2], row.to(dev).expand(K, N),
                  out_dtype=torch.float32).cpu()
    A = base_a[:, ::2].contiguous()
    p = oracle.Problem(ab_dtype="bf16", c_dtype="f32", M=M, N=N, K=K, A=bits(A),
                       B=bits(base_b.contiguous()), strides=((K, 1), (N, 1), (N, 1)))
    assert np.array_equal(out.numpy().astype(np.float64), oracle.gemm(p)[0])
