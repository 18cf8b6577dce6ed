"""gemm_bf16_static_workspace: the bf16 GEMM for callers that cannot allocate
device memory (a host framework that has reserved the device's memory, a
plugin hook that forbids allocation, a loop that must not enter the
allocator).  Its scratch is a library-owned device array, so the caller
passes only inputs and outputs.

Checked through the C ABI against gemm_bf16 with a caller workspace, on two
calls in a row (the array keeps the previous call's contents), with a
split-K plan so that the scratch is really used.  This file is collected last
on purpose.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import dense_gemm_bf16_gb300 as dg
    dg.build()
    dg.lib()
    return dg


def _inputs(seed, M, N, K):
    import datagen
    a = datagen.to_bf16_bits(datagen.uniform(seed, (M, K)))
    b = datagen.to_bf16_bits(datagen.uniform(seed + 1, (K, N)))
    bias = datagen.to_f32(datagen.normal(seed + 2, (N,)))
    dA = torch.from_numpy(a.view(np.int16)).cuda()
    dB = torch.from_numpy(b.view(np.int16)).cuda()
    return dA, dB, torch.from_numpy(bias).cuda()


def _call(dg, fn, M, N, K, dA, dB, dbias, split_k, workspace=None):
    dC = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    common = (M, N, K, dA.data_ptr(), K, 0, dB.data_ptr(), N, 0, dC.data_ptr(), N, 0,
              int(dg.DType.F32), 1.0, 0.0, dbias.data_ptr(), int(dg.Epi.BIAS), split_k)
    if workspace is None:
        st = fn(*common, stream)
    else:
        st = fn(*common, workspace.data_ptr(), workspace.numel(), stream)
    torch.cuda.synchronize()
    return st, dC.cpu().numpy().astype(np.float64)


def test_static_workspace_matches_gemm_bf16_twice(dg):
    M, N, K, split = 256, 384, 4096, 8
    # the split-K partials must fit the library's array
    assert split * M * N * 4 <= dg.STATIC_WORKSPACE_BYTES
    st, plan = dg.gemm_plan_query(0, 1, M, N, K, 16, K, 0, 0, 16, N, 0, 0, 16, N, 0, 0, 2, 1.0,
                                  0.0, 16, 1, split, dg.STATIC_WORKSPACE_BYTES)
    assert st == 0 and plan.split_k == split and plan.workspace_bytes > 0
    for seed in (101, 202):  # two calls in a row, different data
        dA, dB, dbias = _inputs(seed, M, N, K)
        ws = torch.empty(dg.gemm_workspace_size(0, 1, M, N, K, split), dtype=torch.uint8,
                         device="cuda")
        st_ref, ref = _call(dg, dg.gemm_bf16, M, N, K, dA, dB, dbias, split, ws)
        st_new, got = _call(dg, dg.gemm_bf16_static_workspace, M, N, K, dA, dB, dbias, split)
        assert st_ref == 0 and st_new == 0
        assert np.all(np.isfinite(got))
        scale = np.sqrt(K) * 1.0 + float(dbias.abs().max())
        assert np.abs(got - ref).max() / scale <= 1e-4
    stream = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_check_device_status(stream) == 0


def test_static_workspace_rejects_plans_beyond_its_size(dg):
    M, N, K = 2048, 2048, 65536
    split = 8  # 8 slices x 16 MiB of fp32 partials > the array
    assert split * M * N * 4 > dg.STATIC_WORKSPACE_BYTES
    dummy = torch.empty(64, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = dg.gemm_bf16_static_workspace(M, N, K, p, K, 0, p, N, 0, p, N, 0, int(dg.DType.F32),
                                       1.0, 0.0, None, 0, split,
                                       torch.cuda.current_stream().cuda_stream)
    assert st == dg.Status.ERR_WORKSPACE
