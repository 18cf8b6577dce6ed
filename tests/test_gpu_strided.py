"""GPU parity of gemm_strided (matrices given by element strides) against the
oracle's strided form, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest

import datagen
import oracle

pytestmark = pytest.mark.gpu

ES = {"bf16": 2, "f16": 2, "f32": 4}
DT_CODE = {"bf16": 0, "f16": 1, "f32": 2}
NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}


def place(vals, rs, cs, bs, dt):
    """Logical [nb, R, C] values at b*bs + r*rs + c*cs in a NaN-poisoned buffer;
    returns (storage, mask of used slots)."""
    vals = np.asarray(vals, dtype=np.float64)
    nb, R, C = vals.shape
    size = (nb - 1) * bs + (R - 1) * rs + (C - 1) * cs + 1 if vals.size else 1
    buf = np.zeros(size)
    used = np.zeros(size, dtype=bool)
    for b in range(nb):
        for r in range(R):
            idx = b * bs + r * rs + np.arange(C) * cs
            buf[idx] = vals[b, r]
            used[idx] = True
    out = datagen.encode(buf, dt)
    if dt == "f32":
        out[~used] = np.nan
    else:
        out[~used] = NAN_BITS[dt]
    return out, used


def decode(bits, dt):
    if dt == "bf16":
        return datagen.bf16_bits_to_f32(bits).astype(np.float64)
    if dt == "f16":
        return datagen.f16_bits_to_f32(bits).astype(np.float64)
    return bits.astype(np.float64)


def values(kind, seed, shape):
    if kind == "ints":
        return datagen.small_ints(seed, shape).astype(np.float64)
    return datagen.uniform(seed, shape)


def run_strided(ab, M, N, K, a_st, b_st, c_st, *, c_dtype="f32", batch=1, alpha=1.0, beta=0.0,
                bias=False, act="none", split_k=0, kind="ints", seed=1, ws_bytes=None):
    """a_st / b_st / c_st: (rs, cs, batch stride).  Returns (status, got, ref,
    C storage after, C storage before, used mask of C)."""
    import torch
    import dense_gemm_bf16_gb300 as dg
    nb_a = batch if a_st[2] else 1
    nb_b = batch if b_st[2] else 1
    A = datagen.encode(values(kind, seed, (nb_a, M, K)), ab)
    B = datagen.encode(values(kind, seed + 1, (nb_b, K, N)), ab)
    c0 = (values("ints", seed + 2, (batch, M, N)) if kind == "ints"
          else datagen.normal(seed + 2, (batch, M, N)))
    C0 = datagen.encode(c0, c_dtype)
    fa, _ = place(decode(A, ab).reshape(nb_a, M, K), *a_st, ab)
    fb, _ = place(decode(B, ab).reshape(nb_b, K, N), *b_st, ab)
    fc, used_c = place(decode(C0, c_dtype).reshape(batch, M, N), *c_st, c_dtype)
    bias_v = datagen.to_f32(datagen.normal(seed + 3, (N,))) if bias else None
    p = oracle.Problem(ab_dtype=ab, M=M, N=N, K=K, A=fa, B=fb, c_dtype=c_dtype, C0=fc,
                       batch=batch, stride_a=a_st[2], stride_b=b_st[2], stride_c=c_st[2],
                       alpha=alpha, beta=beta, bias=bias_v, act=act,
                       strides=[a_st[:2], b_st[:2], c_st[:2]])
    ref = oracle.gemm(p)

    def dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    dA, dB, dC = dev(fa), dev(fb), dev(fc)
    dbias = dev(bias_v) if bias else None
    need = dg.gemm_strided_workspace_size(DT_CODE[ab], DT_CODE[c_dtype], batch, M, N, K, *a_st,
                                          *b_st, *c_st, split_k)
    nbytes = need if ws_bytes is None else ws_bytes
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    epi = (1 if bias else 0) | ({"none": 0, "gelu_tanh": 1, "relu": 2, "gelu_erf": 3}[act] << 1)
    st = dg.gemm_strided(DT_CODE[ab], batch, M, N, K, dA.data_ptr(), *a_st, dB.data_ptr(), *b_st,
                         dC.data_ptr(), *c_st, DT_CODE[c_dtype], alpha, beta,
                         dbias.data_ptr() if bias else None, epi, split_k,
                         ws.data_ptr() if nbytes else None, nbytes,
                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    got = np.zeros((batch, M, N))
    vals = decode(out, c_dtype)
    for b in range(batch):
        for r in range(M):
            got[b, r] = vals[b * c_st[2] + r * c_st[0] + np.arange(N) * c_st[1]]
    return st, got, ref, out, fc, used_c


def check(st, got, ref, out, before, used, exact=True, c_dtype="f32", scale=None):
    """exact: bit for bit.  Otherwise the stated tolerances: a 16-bit output
    element by element, |err| <= 1e-2 + 1e-2 |ref|; an fp32 output by its
    sqrt(K)-normalised maximum error, max |err| / scale <= 1e-4."""
    assert st == 0, f"status {st}"
    if exact:
        assert np.array_equal(got, ref), f"max |diff| {np.abs(got - ref).max()}"
    elif c_dtype != "f32":
        err = np.abs(got - ref)
        bad = err > 1e-2 + 1e-2 * np.abs(ref)
        assert not bad.any(), f"{bad.sum()} elements out of tolerance, worst {err.max():.3g}"
    else:
        assert scale is not None and scale > 0
        assert np.abs(got - ref).max() / scale <= 1e-4
    # the slots between C's elements keep their bytes
    assert np.array_equal(out.view(np.uint8).reshape(out.size, -1)[~used],
                          before.view(np.uint8).reshape(before.size, -1)[~used])


def test_a_with_non_unit_inner_stride():
    M, N, K = 70, 90, 130
    check(*run_strided("bf16", M, N, K, (2 * K + 3, 2, 0), (N, 1, 0), (N, 1, 0)))


def test_b_general_a_column_major():
    M, N, K = 65, 80, 100
    check(*run_strided("bf16", M, N, K, (1, M + 5, 0), (3, 3 * K + 1, 0), (N, 1, 0)))


def test_c_general_with_beta():
    M, N, K = 50, 70, 60
    check(*run_strided("bf16", M, N, K, (K, 1, 0), (N, 1, 0), (2 * N + 1, 2, 0), beta=1.0))


def test_all_dense_strides_take_no_copy():
    import dense_gemm_bf16_gb300 as dg
    M, N, K = 128, 96, 64
    assert dg.gemm_strided_workspace_size(0, 2, 1, M, N, K, K, 1, 0, 1, K, 0, 1, M, 0, 1) == \
        dg.gemm_workspace_size(0, 1, M, N, K, 1)
    check(*run_strided("bf16", M, N, K, (K, 1, 0), (1, K, 0), (1, M, 0), split_k=1))


def test_fp32_general_strides():
    M, N, K = 67, 45, 33
    check(*run_strided("f32", M, N, K, (3, 3 * M + 2, 0), (N + 7, 1, 0), (1, M + 1, 0),
                       alpha=1.5, beta=0.5))


def test_batched_broadcast_b_general_a():
    M, N, K, nb = 40, 48, 56, 3
    check(*run_strided("f16", M, N, K, (2 * K, 2, 2 * K * M + 10), (N, 1, 0),
                       (N, 1, M * N), batch=nb, alpha=0.5))


def test_split_k_and_epilogue_through_copies():
    M, N, K = 100, 120, 2048
    st, got, ref, out, before, used = run_strided(
        "bf16", M, N, K, (2 * K, 2, 0), (N, 1, 0), (2 * N, 2, 0), c_dtype="bf16", beta=0.5,
        bias=True, act="gelu_erf", split_k=4, kind="uniform", seed=7)
    check(st, got, ref, out, before, used, exact=False, c_dtype="bf16")


def test_workspace_too_small_and_bad_strides():
    import dense_gemm_bf16_gb300 as dg
    st = run_strided("bf16", 40, 40, 40, (80, 2, 0), (40, 1, 0), (40, 1, 0), ws_bytes=0)[0]
    assert st == int(dg.Status.ERR_WORKSPACE)
    assert dg.gemm_strided_workspace_size(0, 2, 1, 40, 40, 40, 40, 1, 0, 40, 1, 0, 0, 1, 0, 0) == 0
    assert dg.gemm_strided_workspace_size(0, 2, 1, 40, 40, 40, -1, 1, 0, 40, 1, 0, 40, 1, 0, 0) == 0
