"""The tensor-level binding (``api.plan`` / ``api.gemm``'s argument reading)
without a GPU: matrix descriptors read off torch tensors, argument checks, and
plans for CPU tensors on the simulated 152-SM device (planning only reads the
pointers' alignment)."""
import pytest
import torch

import dense_gemm_bf16_gb300 as dg
from dense_gemm_bf16_gb300 import Epi, Layout, Option, Status
from dense_gemm_bf16_gb300 import api


@pytest.fixture(scope="module", autouse=True)
def simulated_device():
    dg.build()
    dg.lib()
    assert dg.gemm_set_option(Option.TEST_SIM_SMS, 152) == Status.OK
    yield
    dg.gemm_set_option(Option.TEST_SIM_SMS, 0)


def test_matrix_desc_layouts():
    a = torch.empty(300, 200, dtype=torch.bfloat16)
    assert api.matrix_desc(a)[1:] == (200, Layout.ROW_MAJOR, 1, 0)
    assert api.matrix_desc(a.t())[1:] == (200, Layout.COL_MAJOR, 1, 0)
    padded = torch.empty(300, 256, dtype=torch.bfloat16)[:, :200]
    assert api.matrix_desc(padded)[1:] == (256, Layout.ROW_MAJOR, 1, 0)
    assert api.matrix_desc(padded.t())[1:] == (256, Layout.COL_MAJOR, 1, 0)
    b3 = torch.empty(4, 300, 200, dtype=torch.float16)
    assert api.matrix_desc(b3)[1:] == (200, Layout.ROW_MAJOR, 4, 60000)
    assert api.matrix_desc(b3.transpose(1, 2))[1:] == (200, Layout.COL_MAJOR, 4, 60000)
    # a broadcast batch (stride 0) and a batch of one both give batch stride 0
    assert api.matrix_desc(a.expand(4, 300, 200))[3:] == (4, 0)
    assert api.matrix_desc(a.unsqueeze(0))[3:] == (1, 0)


def test_matrix_desc_vectors_take_any_stride_on_their_unit_dimension():
    col = torch.empty(300, 8, dtype=torch.bfloat16)[:, 3:4]       # [300, 1], strides (8, 1)
    assert api.matrix_desc(col)[1:3] == (8, Layout.ROW_MAJOR)
    row = torch.empty(8, 300, dtype=torch.bfloat16)[3:4, :]       # [1, 300], strides (300, 1)
    assert api.matrix_desc(row)[1:3] == (300, Layout.ROW_MAJOR)
    row_t = torch.empty(300, 8, dtype=torch.bfloat16).t()[3:4]    # [1, 300], strides (1, 8)
    assert api.matrix_desc(row_t)[1:3] == (8, Layout.COL_MAJOR)    # column c at c * 8


@pytest.mark.parametrize("make", [
    lambda: torch.empty(1, 200, dtype=torch.bfloat16).expand(300, 200),   # rows of stride 0
    lambda: torch.empty(300, 1, dtype=torch.bfloat16).expand(300, 200).t(),
    lambda: torch.empty(300, 400, dtype=torch.bfloat16)[:, ::2],          # inner stride 2
    lambda: torch.empty(300, dtype=torch.bfloat16),                       # not a matrix
    lambda: torch.empty(2, 2, 30, 20, dtype=torch.bfloat16),
])
def test_matrix_desc_rejects_what_the_abi_cannot_address(make):
    with pytest.raises(ValueError):
        api.matrix_desc(make())


def bf(*shape):
    return torch.empty(*shape, dtype=torch.bfloat16)


def test_plan_of_the_headline_workload_through_tensors():
    M = N = K = 8192
    A, B = bf(M, K), bf(N, K).t()         # B column-major
    C, bias = bf(M, N), torch.empty(N, dtype=torch.float32)
    p = api.plan(A, B, C, bias=bias, epilogue="bias_gelu_tanh", workspace_bytes=0)
    assert p["kernel"] == 1 and p["cta_pair"] == 2 and p["block_n"] == 256
    assert p["block_k"] == 128 and p["grid"] == 152 and p["fast_epilogue"] == 1
    assert api.plan(A, B, C, bias=bias, epilogue=Epi.BIAS_GELU_TANH, workspace_bytes=0) == p


def test_plan_defaults_to_a_bias_epilogue_when_given_a_bias():
    A, B, C = bf(256, 512), bf(512, 384), bf(256, 384)
    bias = torch.empty(384, dtype=torch.float32)
    assert api.plan(A, B, C, bias=bias) == api.plan(A, B, C, bias=bias, epilogue="bias")


def test_every_epilogue_name_is_accepted_with_the_right_bias():
    M, N, K = 256, 384, 512
    A, B, C = bf(M, K), bf(K, N), bf(M, N)
    for e in Epi:
        bias = None
        if e & Epi.BIAS:
            bias = torch.empty(M if e & 8 else N, dtype=torch.float32)
        p = api.plan(A, B, C, bias=bias, epilogue=e.name.lower())
        assert p["kernel"] == 1


def test_argument_errors():
    M, N, K = 256, 384, 512
    A, B, C = bf(M, K), bf(K, N), bf(M, N)
    col_bias = torch.empty(N, dtype=torch.float32)
    with pytest.raises(ValueError, match="length 256"):
        api.plan(A, B, C, bias=col_bias, epilogue="row_bias")
    with pytest.raises(ValueError, match="takes no bias"):
        api.plan(A, B, C, bias=col_bias, epilogue="relu")
    with pytest.raises(ValueError, match="needs a bias"):
        api.plan(A, B, C, epilogue="bias_relu")
    with pytest.raises(ValueError, match="unknown epilogue"):
        api.plan(A, B, C, epilogue="swish")
    with pytest.raises(ValueError, match="fp32 vector"):
        api.plan(A, B, C, bias=torch.empty(N, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="fp32 vector"):
        api.plan(A, B, C, bias=torch.empty(2 * N, dtype=torch.float32)[::2])
    with pytest.raises(TypeError):
        api.plan(A, B.half(), C)
    with pytest.raises(ValueError, match="shape mismatch"):
        api.plan(A, bf(K + 1, N), C)
    with pytest.raises(ValueError, match="do not broadcast"):
        api.plan(bf(3, M, K), bf(4, K, N), bf(4, M, N))
    with pytest.raises(ValueError, match="full batch"):
        api.plan(bf(4, M, K), B, C)


def test_batched_plans_through_tensors():
    s = 1024
    A, B, C = bf(64, s, s), bf(64, s, s), bf(64, s, s)
    p = api.plan(A, B, C, alpha=0.5, beta=1.0)
    # beta * C by TMA loads, on eight epilogue warps (short K)
    assert p["fast_epilogue"] == 4 and p["cta_pair"] == 2
    pb = api.plan(A, bf(s, s).expand(64, s, s), C, alpha=0.5, beta=1.0)
    assert pb["fast_epilogue"] == 4


def test_workspace_defaults_to_what_the_plan_needs():
    A, B = bf(256, 65536), bf(65536, 256)
    C = torch.empty(256, 256, dtype=torch.float32)
    p = api.plan(A, B, C)
    assert p["stream_k"] == 4 and p["workspace_bytes"] > 0     # the atomic split-K
    assert api.plan(A, B, C, workspace_bytes=p["workspace_bytes"]) == p
    assert api.plan(A, B, C, workspace_bytes=0)["stream_k"] == 0


def _capture(monkeypatch, name, status=0):
    # these tests read the arguments a call would pass, with host tensors
    monkeypatch.setattr(api, "_require_cuda", lambda **kw: None)
    seen = []

    def fake(*args):
        seen.append(args)
        return status
    monkeypatch.setattr(api._abi, name, fake)
    return seen


def test_views_that_are_not_matrices_go_through_gemm_strided(monkeypatch):
    M, N, K = 64, 48, 32
    base_a = bf(M, 2 * K)
    A = base_a[:, ::2]                                   # a step of 2 along K
    row = bf(1, N)
    B = row.expand(K, N)                                 # every row the same
    C = torch.empty(M, N, dtype=torch.float32)
    sizes = _capture(monkeypatch, "gemm_strided_workspace_size", 4096)
    calls = _capture(monkeypatch, "gemm_strided")
    batched = _capture(monkeypatch, "gemm_batched")
    out = api.gemm(A, B, C, alpha=0.5, stream=0)
    assert out is C and batched == [] and len(calls) == 1
    args = calls[0]
    assert args[:5] == (0, 1, M, N, K)
    assert args[5:9] == (A.data_ptr(), 2 * K, 2, 0)      # A: row stride, column stride, batch
    assert args[9:13] == (B.data_ptr(), 0, 1, 0)          # B: rows of stride 0
    assert args[13:17] == (C.data_ptr(), N, 1, 0)
    assert args[17:23] == (2, 0.5, 0.0, 0, 0, 0)
    assert args[24] >= 4096                              # the workspace it was told to need
    assert sizes[0] == (0, 2, 1, M, N, K, 2 * K, 2, 0, 0, 1, 0, N, 1, 0, 0)


def test_batched_views_pass_their_batch_strides(monkeypatch):
    bt, M, N, K = 3, 32, 40, 24
    A = bf(bt, M, 3 * K)[:, :, ::3]
    B = bf(K, N)                                         # broadcast over the batch
    C = torch.empty(bt, M, N, dtype=torch.bfloat16)
    _capture(monkeypatch, "gemm_strided_workspace_size", 0)
    calls = _capture(monkeypatch, "gemm_strided")
    api.gemm(A, B, C, stream=0)
    args = calls[0]
    assert args[1] == bt and args[5:9] == (A.data_ptr(), 3 * K, 3, M * 3 * K)
    assert args[9:13] == (B.data_ptr(), N, 1, 0) and args[13:17] == (C.data_ptr(), N, 1, M * N)
    assert args[23] == 0 and args[24] == 0               # no workspace needed, none passed


def test_matrix_views_stay_on_gemm_batched(monkeypatch):
    A, B = bf(64, 32), bf(48, 32).t()
    C = torch.empty(64, 48, dtype=torch.float32)
    calls = _capture(monkeypatch, "gemm_batched")
    strided = _capture(monkeypatch, "gemm_strided")
    api.gemm(A, B, C, stream=0)
    assert strided == [] and len(calls) == 1
    assert calls[0][5:9] == (A.data_ptr(), 32, int(Layout.ROW_MAJOR), 0)
    assert calls[0][9:13] == (B.data_ptr(), 32, int(Layout.COL_MAJOR), 0)


def test_host_tensors_are_refused_before_any_call():
    A, B = bf(64, 32), bf(32, 48)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        api.gemm(A, B, stream=0)


def test_an_output_with_repeated_rows_is_rejected_by_the_library(monkeypatch):
    monkeypatch.setattr(api, "_require_cuda", lambda **kw: None)
    A, B = bf(64, 32), bf(32, 48)
    C = torch.empty(1, 48, dtype=torch.float32).expand(64, 48)
    with pytest.raises(dg.GemmError) as e:
        api.gemm(A, B, C, stream=0)
    assert e.value.status == Status.ERR_INVALID_ARG


def test_plan_of_a_strided_view_counts_its_copy():
    A = bf(300, 400)[:, ::2]                     # a step of 2 along K = 200
    B, C = bf(200, 256), torch.empty(300, 256, dtype=torch.float32)
    p = api.plan(A, B, C)
    dense = api.plan(A.contiguous(), B, C)
    assert p["pack_a"] == 1 and dense["pack_a"] == 0
    assert p["launches"] == dense["launches"] + 1
