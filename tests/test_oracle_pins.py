"""Pins for the CPU oracle (no GPU).

The oracle is the plain definition of the GEMM ("2 . La GEMM, de zero a
cuBLAS", section 2.1; epilogue per "Skill: Write a Triton GEMM Kernel",
Required reasoning process step 6).  These tests tie it to things other than
itself:

* format decoding against bit patterns whose values the binary16 / bfloat16
  definitions fix (tests/golden/float_formats.txt);
* exact rational brute force (Python ``fractions``) on tiny ragged shapes, in
  every layout, with padding poisoned by NaN, within the textbook error bound
  of an fp64 dot product (Higham, Accuracy and Stability of Numerical
  Algorithms, eq. 3.5: |fl(x.y) - x.y| <= gamma_K |x|.|y|);
* closed forms: identity B, all-ones, rank-1 outer products, and small-integer
  inputs that reduce to numpy's exact int64 matmul;
* invariants: layout/padding invariance, batch stride 0 = broadcast,
  beta == 0 does not read C, K == 0;
* GELU(tanh): odd-part identity, value at 0, the Taylor coefficients of the
  closed form (which pin sqrt(2/pi) and 0.044715), the large-|x| limits, and
  closeness to the exact erf GELU of the same paper;
* GELU(erf) = x Phi(x): standard normal table values of Phi, the odd-part
  identity, and its curvature at 0 (2 phi(0) = sqrt(2/pi), which pins the
  sqrt(2) inside erf); ReLU on signed values and NaN;
* the epilogue's wiring of each activation (equal to the activation applied
  to the identity-activation result), bias along columns or rows (closed
  form with identity B on non-square shapes), and storage by arbitrary
  (row, column) strides (closed form, and equal to the row-major result).
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import datagen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}


# ---------------------------------------------------------------------------
# independent helpers (numpy / struct based; nothing from oracle/)
# ---------------------------------------------------------------------------

def exact_value(bits_or_val, dt) -> Fraction:
    if dt == "bf16":
        f = struct.unpack("<f", struct.pack("<I", int(bits_or_val) << 16))[0]
    elif dt == "f16":
        f = float(np.array([int(bits_or_val)], dtype=np.uint16).view(np.float16)[0])
    else:
        f = float(np.float32(bits_or_val))
    return Fraction(f)


def store(vals, dt, layout, pad=0, bpad=0):
    """Store logical [batch, R, C] fp64 values (already representable in dt)
    with the given layout; padding filled with NaN.  Returns (flat, ld, stride)."""
    vals = np.asarray(vals, dtype=np.float64)
    if vals.ndim == 2:
        vals = vals[None]
    nb, R, C = vals.shape
    ld = (C if layout == "row" else R) + pad
    per = (R if layout == "row" else C) * ld + bpad
    n = max(nb * per, 1)
    if dt in ("bf16", "f16"):
        flat = np.full(n, NAN_BITS[dt], dtype=np.uint16)
        enc = datagen.encode(vals, dt)
    else:
        flat = np.full(n, np.nan, dtype=np.float32)
        enc = datagen.encode(vals, dt)
    for b in range(nb):
        blk = enc[b] if layout == "row" else enc[b].T
        rows, cols = blk.shape
        for r in range(rows):
            flat[b * per + r * ld: b * per + r * ld + cols] = blk[r]
    return flat, ld, per


def representable(x, dt):
    """Round fp64 values to dt and back (so logical values are exact in dt)."""
    enc = datagen.encode(x, dt)
    if dt == "bf16":
        return datagen.bf16_bits_to_f32(enc).astype(np.float64)
    if dt == "f16":
        return datagen.f16_bits_to_f32(enc).astype(np.float64)
    return enc.astype(np.float64)


def make_problem(oracle, A, B, dt, la, lb, *, C0=None, c_dt="f32", lc="row", alpha=1.0,
                 beta=0.0, bias=None, act="none", pad=0, bstride_a=None, bstride_b=None, bias_rows=False):
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    if A.ndim == 2:
        A = A[None]
    if B.ndim == 2:
        B = B[None]
    nb = max(A.shape[0], B.shape[0])
    M, K = A.shape[1:]
    N = B.shape[2]
    fa, lda, sa = store(A, dt, la, pad)
    fb, ldb, sb = store(B, dt, lb, pad)
    if A.shape[0] == 1 and nb > 1:
        sa = 0
    if B.shape[0] == 1 and nb > 1:
        sb = 0
    if bstride_a is not None:
        sa = bstride_a
    if bstride_b is not None:
        sb = bstride_b
    fc, ldc, sc = (None, N if lc == "row" else M, 0)
    if C0 is not None:
        C0 = np.asarray(C0, dtype=np.float64)
        if C0.ndim == 2:
            C0 = C0[None]
        fc, ldc, sc = store(C0, c_dt, lc, pad)
    return oracle.Problem(ab_dtype=dt, M=M, N=N, K=K, A=fa, lda=lda, la=la, B=fb, ldb=ldb,
                          lb=lb, c_dtype=c_dt, C0=fc, ldc=ldc, lc=lc, batch=nb,
                          stride_a=sa, stride_b=sb, stride_c=sc, alpha=alpha, beta=beta,
                          bias=bias, act=act, bias_rows=bias_rows)


# ---------------------------------------------------------------------------
# format decoding
# ---------------------------------------------------------------------------

def _golden_formats():
    rows = []
    with open(os.path.join(GOLDEN, "float_formats.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            fmt, bits, val = line.split()
            rows.append((fmt, int(bits, 16), val))
    return rows


def _parse_value(s):
    if s in ("inf", "-inf"):
        return float(s)
    if s == "-0":
        return -0.0
    num, _, den = s.partition("/")
    v = Fraction(1)
    for part in num.split("*"):
        v *= Fraction(int(part))
    return v / (int(den) if den else 1)


@pytest.mark.parametrize("fmt,bits,val", _golden_formats())
def test_decode_matches_format_definition(oracle_mod, fmt, bits, val):
    got = oracle_mod.decode_bf16(bits) if fmt == "bf16" else oracle_mod.decode_f16(bits)
    want = _parse_value(val)
    if isinstance(want, float):
        assert got == want and math.copysign(1, got) == math.copysign(1, want)
    else:
        assert Fraction(got) == want


def test_decode_nan(oracle_mod):
    assert math.isnan(oracle_mod.decode_bf16(0x7FC0))
    assert math.isnan(oracle_mod.decode_f16(0x7E00))


def test_decode_all_f16_against_numpy(oracle_mod):
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    got = oracle_mod.decode(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    both_nan = np.isnan(got) & np.isnan(want)
    assert np.all((got == want) | both_nan)


# ---------------------------------------------------------------------------
# exact brute force on tiny ragged shapes
# ---------------------------------------------------------------------------

def exact_gemm(A, B, C0, alpha, beta, bias):
    nb = max(A.shape[0], B.shape[0])
    M, K = A.shape[1:]
    N = B.shape[2]
    fa, fb = Fraction(alpha), Fraction(beta)
    R = np.empty((nb, M, N), dtype=object)
    bound = np.empty((nb, M, N), dtype=np.float64)
    for b in range(nb):
        a = A[min(b, A.shape[0] - 1)]
        bb = B[min(b, B.shape[0] - 1)]
        for i in range(M):
            for j in range(N):
                s = Fraction(0)
                sabs = Fraction(0)
                for k in range(K):
                    p = Fraction(a[i, k]) * Fraction(bb[k, j])
                    s += p
                    sabs += abs(p)
                v = fa * s
                mag = abs(fa) * sabs
                if beta != 0.0:
                    v += fb * Fraction(C0[b, i, j])
                    mag += abs(fb * Fraction(C0[b, i, j]))
                if bias is not None:
                    v += Fraction(float(bias[j]))
                    mag += abs(Fraction(float(bias[j])))
                R[b, i, j] = v
                bound[b, i, j] = float(mag)
    return R, bound


SHAPES = [(1, 1, 1), (3, 2, 5), (7, 5, 3), (2, 17, 9), (17, 3, 16), (5, 7, 1)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("la,lb,lc", [("row", "row", "row"), ("row", "col", "row"),
                                      ("col", "row", "col"), ("col", "col", "row")])
def test_brute_force_exact(oracle_mod, M, N, K, dt, la, lb, lc):
    seed = 7 * M + 11 * N + 13 * K
    A = representable(datagen.uniform(seed, (1, M, K)), dt)
    B = representable(datagen.uniform(seed + 1, (1, K, N)), dt)
    C0 = representable(datagen.normal(seed + 2, (1, M, N)), "f32")
    bias = datagen.to_f32(datagen.normal(seed + 3, (N,)))
    alpha, beta = 1.25, -0.75
    p = make_problem(oracle_mod, A, B, dt, la, lb, C0=C0, lc=lc, alpha=alpha, beta=beta,
                     bias=bias, pad=3)
    got = oracle_mod.gemm(p)
    want, mag = exact_gemm(A, B, C0, alpha, beta, bias)
    u = 2.0 ** -53
    tol = (K + 4) * u * 1.01 * mag + 1e-300
    err = np.abs(got - want.astype(np.float64))
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"max err {err.max()} vs tol {tol.max()}"


def test_brute_force_batched_broadcast(oracle_mod):
    nb, M, N, K = 3, 4, 5, 6
    A = representable(datagen.uniform(51, (nb, M, K)), "bf16")
    B = representable(datagen.uniform(52, (1, K, N)), "bf16")
    C0 = representable(datagen.normal(53, (nb, M, N)), "bf16")
    p = make_problem(oracle_mod, A, B, "bf16", "row", "row", C0=C0, c_dt="bf16",
                     alpha=0.5, beta=1.0, pad=2)
    assert p.stride_b == 0
    got = oracle_mod.gemm(p)
    want, mag = exact_gemm(A, B, C0, 0.5, 1.0, None)
    assert np.all(np.abs(got - want.astype(np.float64)) <= (K + 4) * 2.0 ** -53 * 1.01 * mag)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def test_identity_B(oracle_mod):
    M, K = 9, 12
    A = representable(datagen.uniform(61, (M, K)), "bf16")
    C0 = representable(datagen.uniform(62, (M, K)), "f32")
    p = make_problem(oracle_mod, A, np.eye(K), "bf16", "row", "row", C0=C0,
                     alpha=1.5, beta=0.5)
    got = oracle_mod.gemm(p)[0]
    assert np.array_equal(got, 1.5 * A + 0.5 * C0)


@pytest.mark.parametrize("K", [1, 2, 64, 1000])
def test_all_ones(oracle_mod, K):
    M, N = 3, 4
    C0 = representable(datagen.uniform(63, (M, N)), "f32")
    bias = np.array([1.0, -2.0, 0.5, 0.0], dtype=np.float32)
    p = make_problem(oracle_mod, np.ones((M, K)), np.ones((K, N)), "bf16", "row", "col",
                     C0=C0, alpha=2.0, beta=-1.0, bias=bias)
    got = oracle_mod.gemm(p)[0]
    assert np.array_equal(got, 2.0 * K - C0 + bias.astype(np.float64)[None, :])


def test_rank_one(oracle_mod):
    M, N, K = 6, 7, 33
    u = datagen.small_ints(71, (M,), -4, 4)
    s = datagen.small_ints(72, (K,), -4, 4)
    t = datagen.small_ints(73, (K,), -4, 4)
    v = datagen.small_ints(74, (N,), -4, 4)
    A = np.outer(u, s)
    B = np.outer(t, v)
    p = make_problem(oracle_mod, A, B, "bf16", "row", "row", alpha=3.0)
    got = oracle_mod.gemm(p)[0]
    assert np.array_equal(got, 3.0 * np.outer(u, v) * float(np.dot(s, t)))


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_small_integers_match_int64_matmul(oracle_mod, dt):
    nb, M, N, K = 2, 13, 11, 29
    A = datagen.small_ints(81, (nb, M, K))
    B = datagen.small_ints(82, (nb, K, N))
    p = make_problem(oracle_mod, A, B, dt, "col", "row", pad=1)
    got = oracle_mod.gemm(p)
    want = np.matmul(A.astype(np.int64), B.astype(np.int64)).astype(np.float64)
    assert np.array_equal(got, want)


def test_transposed_operands_differ(oracle_mod):
    """A transposed operand must give a different answer (non-symmetric data)."""
    n = 8
    A = representable(datagen.uniform(91, (n, n)), "bf16")
    B = representable(datagen.uniform(92, (n, n)), "bf16")
    r = oracle_mod.gemm(make_problem(oracle_mod, A, B, "bf16", "row", "row"))[0]
    rt = oracle_mod.gemm(make_problem(oracle_mod, A, B.T, "bf16", "row", "row"))[0]
    assert not np.allclose(r, rt)
    assert np.allclose(r, A @ B, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants and edge cases
# ---------------------------------------------------------------------------

def test_layout_and_padding_invariance(oracle_mod):
    M, N, K = 10, 7, 19
    A = representable(datagen.uniform(101, (M, K)), "f16")
    B = representable(datagen.uniform(102, (K, N)), "f16")
    C0 = representable(datagen.uniform(103, (M, N)), "f16")
    ref = None
    for la in ("row", "col"):
        for lb in ("row", "col"):
            for lc in ("row", "col"):
                for pad in (0, 5):
                    p = make_problem(oracle_mod, A, B, "f16", la, lb, C0=C0, c_dt="f16",
                                     lc=lc, alpha=0.5, beta=2.0, pad=pad)
                    r = oracle_mod.gemm(p)
                    if ref is None:
                        ref = r
                    assert np.array_equal(r, ref)


def test_batched_equals_per_batch(oracle_mod):
    nb, M, N, K = 4, 5, 6, 7
    A = representable(datagen.uniform(111, (nb, M, K)), "bf16")
    B = representable(datagen.uniform(112, (nb, K, N)), "bf16")
    full = oracle_mod.gemm(make_problem(oracle_mod, A, B, "bf16", "row", "col", pad=1))
    for b in range(nb):
        one = oracle_mod.gemm(make_problem(oracle_mod, A[b], B[b], "bf16", "row", "col"))
        assert np.array_equal(full[b], one[0])


def test_broadcast_stride_zero_equals_copies(oracle_mod):
    nb, M, N, K = 3, 4, 5, 6
    A = representable(datagen.uniform(121, (nb, M, K)), "bf16")
    B1 = representable(datagen.uniform(122, (1, K, N)), "bf16")
    bc = oracle_mod.gemm(make_problem(oracle_mod, A, B1, "bf16", "row", "row"))
    cp = oracle_mod.gemm(make_problem(oracle_mod, A, np.repeat(B1, nb, axis=0), "bf16",
                                      "row", "row"))
    assert np.array_equal(bc, cp)


def test_beta_zero_does_not_read_C(oracle_mod):
    M, N, K = 3, 3, 4
    A = np.ones((M, K))
    B = np.ones((K, N))
    C0 = np.full((M, N), np.nan)
    p = make_problem(oracle_mod, A, B, "bf16", "row", "row", C0=C0, alpha=1.0, beta=0.0)
    assert np.array_equal(oracle_mod.gemm(p)[0], np.full((M, N), 4.0))


def test_k_zero(oracle_mod):
    M, N = 4, 3
    C0 = representable(datagen.uniform(131, (M, N)), "f32")
    bias = np.array([0.5, -1.0, 2.0], dtype=np.float32)
    fa = np.zeros(1, dtype=np.uint16)
    fc, ldc, _ = store(C0, "f32", "row")
    p = oracle_mod.Problem(ab_dtype="bf16", M=M, N=N, K=0, A=fa, lda=1, la="row", B=fa,
                           ldb=N, lb="row", c_dtype="f32", C0=fc, ldc=ldc, alpha=3.0,
                           beta=0.25, bias=bias)
    assert np.array_equal(oracle_mod.gemm(p)[0], 0.25 * C0 + bias.astype(np.float64))


def test_sampled_equals_full(oracle_mod):
    nb, M, N, K = 2, 9, 10, 11
    A = representable(datagen.uniform(141, (nb, M, K)), "bf16")
    B = representable(datagen.uniform(142, (nb, K, N)), "bf16")
    C0 = representable(datagen.uniform(143, (nb, M, N)), "bf16")
    bias = datagen.to_f32(datagen.normal(144, (N,)))
    p = make_problem(oracle_mod, A, B, "bf16", "row", "col", C0=C0, c_dt="bf16", alpha=0.5,
                     beta=1.0, bias=bias, act="gelu_tanh")
    full = oracle_mod.gemm(p)
    bs, is_, js = np.meshgrid(np.arange(nb), np.arange(M), np.arange(N), indexing="ij")
    s = oracle_mod.gemm_sampled(p, bs.ravel(), is_.ravel(), js.ravel())
    assert np.array_equal(s, full.ravel())


def test_rejects_out_of_range_sample(oracle_mod):
    A = np.ones((2, 2))
    p = make_problem(oracle_mod, A, A, "bf16", "row", "row")
    with pytest.raises(ValueError):
        oracle_mod.gemm_sampled(p, [0], [2], [0])


# ---------------------------------------------------------------------------
# GELU (tanh form)
# ---------------------------------------------------------------------------

def test_gelu_zero_and_limits(oracle_mod):
    g = oracle_mod.gelu_tanh
    assert g(0.0) == 0.0
    for x in (10.0, 25.0, 1e3):
        assert g(x) == x
    for x in (-10.0, -25.0):
        assert abs(g(x)) < 1e-30


def test_gelu_odd_part_identity(oracle_mod):
    # tanh is odd, so gelu(x) - gelu(-x) = x exactly in real arithmetic
    g = oracle_mod.gelu_tanh
    for x in np.linspace(-6, 6, 241):
        assert abs((g(x) - g(-x)) - x) <= 4e-16 * max(1.0, abs(x))


def test_gelu_taylor_coefficients(oracle_mod):
    # even part: gelu(h) + gelu(-h) = h tanh(c (h + a h^3)) = c h^2 + (c a - c^3/3) h^4 + O(h^6)
    # with c = sqrt(2/pi) and a = 0.044715 (Hendrycks & Gimpel 2016, section 2)
    g = oracle_mod.gelu_tanh
    c = math.sqrt(2.0 / math.pi)
    a = 0.044715
    h = 1e-3
    even = g(h) + g(-h)
    assert abs(even / h ** 2 - c) < 1e-5
    c4 = (even / h ** 2 - c) / h ** 2
    assert abs(c4 - (c * a - c ** 3 / 3.0)) < 1e-3 * abs(c * a - c ** 3 / 3.0)
    # first derivative at 0 is 1/2
    assert abs((g(h) - g(-h)) / (2 * h) - 0.5) < 1e-12


def test_gelu_close_to_erf_form(oracle_mod):
    # the tanh form approximates x * Phi(x) (the exact GELU) to within ~5e-4
    g = oracle_mod.gelu_tanh
    worst = 0.0
    for x in np.linspace(-8, 8, 1601):
        exact = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))
        worst = max(worst, abs(g(x) - exact))
    assert worst < 5e-4
    assert worst > 1e-5  # it is the tanh form, not erf itself


def test_gelu_applied_after_bias(oracle_mod):
    # A = 0: R = gelu(beta*C0 + bias) elementwise; check against the oracle's own scalar gelu
    M, N, K = 2, 3, 4
    C0 = np.array([[1.0, -1.0, 0.5], [2.0, -3.0, 0.0]])
    bias = np.array([0.25, 0.5, -1.0], dtype=np.float32)
    p = make_problem(oracle_mod, np.zeros((M, K)), np.ones((K, N)), "bf16", "row", "row",
                     C0=C0, alpha=1.0, beta=2.0, bias=bias, act="gelu_tanh")
    got = oracle_mod.gemm(p)[0]
    for i in range(M):
        for j in range(N):
            assert got[i, j] == oracle_mod.gelu_tanh(2.0 * C0[i, j] + float(bias[j]))


# ---------------------------------------------------------------------------
# GELU (erf form), ReLU, bias orientation, general strides
# ---------------------------------------------------------------------------

# Phi(x) of the standard normal distribution, from standard normal tables
# (values to 16 digits, e.g. Abramowitz & Stegun, table 26.1).
PHI_TABLE = {1.0: 0.8413447460685429, 1.96: 0.9750021048517795, -0.5: 0.3085375387259869,
             2.5: 0.9937903346742238}


@pytest.mark.parametrize("x", sorted(PHI_TABLE))
def test_gelu_erf_is_x_phi(oracle_mod, x):
    assert oracle_mod.gelu_erf(x) == pytest.approx(x * PHI_TABLE[x], rel=1e-14)


def test_gelu_erf_odd_part_and_curvature(oracle_mod):
    g = oracle_mod.gelu_erf
    assert g(0.0) == 0.0
    for x in (0.1, 0.7, 1.3, 4.0):
        # Phi(x) + Phi(-x) = 1  =>  g(x) - g(-x) = x
        assert g(x) - g(-x) == pytest.approx(x, rel=1e-14)
    # g'(0) = Phi(0) = 1/2 and g''(0) = 2 phi(0) = sqrt(2/pi): central differences
    h = 1e-4
    assert (g(h) - g(-h)) / (2 * h) == pytest.approx(0.5, abs=1e-9)
    assert (g(h) - 2 * g(0.0) + g(-h)) / h ** 2 == pytest.approx(math.sqrt(2 / math.pi), rel=1e-5)


def test_relu_definition(oracle_mod):
    r = oracle_mod.relu
    assert [r(x) for x in (-2.0, -0.0, 0.0, 3.5, 1e-300)] == [0.0, 0.0, 0.0, 3.5, 1e-300]
    assert r(float("nan")) == 0.0


def _wiring_case(oracle_mod, act, bias_rows=False):
    M, N, K = 7, 5, 9
    A = representable(datagen.uniform(71, (M, K)), "bf16")
    B = representable(datagen.uniform(72, (K, N)), "bf16")
    bias = representable(datagen.normal(73, (M if bias_rows else N,)), "f32")
    p = make_problem(oracle_mod, A, B, "bf16", "row", "row", alpha=1.5, bias=bias,
                     act=act, bias_rows=bias_rows)
    return oracle_mod.gemm(p)[0], A, B, bias


@pytest.mark.parametrize("act", ["relu", "gelu_erf", "gelu_tanh"])
@pytest.mark.parametrize("bias_rows", [False, True])
def test_activation_applied_to_identity_result(oracle_mod, act, bias_rows):
    got, *_ = _wiring_case(oracle_mod, act, bias_rows)
    ident, *_ = _wiring_case(oracle_mod, "none", bias_rows)
    fn = {"relu": oracle_mod.relu, "gelu_erf": oracle_mod.gelu_erf,
          "gelu_tanh": oracle_mod.gelu_tanh}[act]
    want = np.vectorize(fn)(ident)
    assert np.array_equal(got, want)
    if act == "relu":
        assert np.array_equal(got, np.maximum(ident, 0.0))


@pytest.mark.parametrize("M,N", [(9, 4), (4, 9)])
def test_bias_orientation_closed_form(oracle_mod, M, N):
    # B = identity (N = K): R = alpha * A + bias, bias along columns (length N)
    # or along rows (length M); non-square so that the orientations differ
    A = representable(datagen.uniform(74, (M, N)), "bf16")
    bias_c = representable(datagen.normal(75, (N,)), "f32")
    bias_r = representable(datagen.normal(76, (M,)), "f32")
    pc = make_problem(oracle_mod, A, np.eye(N), "bf16", "row", "row", alpha=0.5, bias=bias_c)
    pr = make_problem(oracle_mod, A, np.eye(N), "bf16", "row", "row", alpha=0.5, bias=bias_r,
                      bias_rows=True)
    assert np.array_equal(oracle_mod.gemm(pc)[0], 0.5 * A + bias_c[None, :])
    assert np.array_equal(oracle_mod.gemm(pr)[0], 0.5 * A + bias_r[:, None])


def _store_strided(vals, rs, cs, dt, size):
    """Logical [R, C] values placed at r*rs + c*cs in a NaN-filled buffer."""
    R, C = vals.shape
    buf = np.zeros(size)
    used = np.zeros(size, dtype=bool)
    for r in range(R):
        for c in range(C):
            buf[r * rs + c * cs] = vals[r, c]
            used[r * rs + c * cs] = True
    assert used.sum() == R * C  # the map is injective
    out = datagen.encode(buf, dt)
    out[~used] = np.nan if dt == "f32" else NAN_BITS[dt]
    return out


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_strided_storage(oracle_mod, dt):
    M, N, K = 5, 6, 7
    A = representable(datagen.uniform(77, (M, K)), dt)
    B = representable(datagen.uniform(78, (K, N)), dt)
    C0 = representable(datagen.normal(79, (M, N)), "f32")
    # A with row stride 3 and column stride 17, B transposed with a gap, C
    # interleaved: every map is injective and none is row- or column-major
    fa = _store_strided(A, 3, 17, dt, 3 * M + 17 * K)
    fb = _store_strided(B, 2, 2 * K + 3, dt, 2 * K + (2 * K + 3) * N)
    fc = _store_strided(C0, 2 * N + 1, 2, "f32", (2 * N + 1) * M + 2 * N)
    strided = oracle_mod.Problem(ab_dtype=dt, M=M, N=N, K=K, A=fa, B=fb, c_dtype="f32", C0=fc,
                                 alpha=1.25, beta=-0.5,
                                 strides=[(3, 17), (2, 2 * K + 3), (2 * N + 1, 2)])
    dense = make_problem(oracle_mod, A, B, dt, "row", "row", C0=C0, alpha=1.25, beta=-0.5)
    got = oracle_mod.gemm(strided)
    assert np.array_equal(got, oracle_mod.gemm(dense))
    # closed form with B = identity, stored with strides
    fi = _store_strided(np.eye(K), 1, K + 2, dt, (K + 2) * K)
    pid = oracle_mod.Problem(ab_dtype=dt, M=M, N=K, K=K, A=fa, B=fi, c_dtype="f32",
                             alpha=2.0, strides=[(3, 17), (1, K + 2), (K, 1)])
    assert np.array_equal(oracle_mod.gemm(pid)[0], 2.0 * A)


def test_strided_sampled_equals_strided_full(oracle_mod):
    # the one-by-one form of the strided oracle against its full form, with a
    # batch, batch strides, a broadcast B, a bias along rows and an activation
    nb, M, N, K = 2, 5, 6, 7
    A = representable(datagen.uniform(181, (nb, M, K)), "bf16")
    B = representable(datagen.uniform(182, (K, N)), "bf16")
    C0 = representable(datagen.normal(183, (nb, M, N)), "f32")
    bias = datagen.to_f32(datagen.normal(184, (M,)))
    sa = 3 * M + 17 * K
    fa = np.concatenate([_store_strided(A[b], 3, 17, "bf16", sa) for b in range(nb)])
    fb = _store_strided(B, 2, 2 * K + 3, "bf16", 2 * K + (2 * K + 3) * N)
    sc = (2 * N + 1) * M + 2 * N
    fc = np.concatenate([_store_strided(C0[b], 2 * N + 1, 2, "f32", sc) for b in range(nb)])
    p = oracle_mod.Problem(ab_dtype="bf16", M=M, N=N, K=K, batch=nb, A=fa, B=fb, c_dtype="f32",
                           C0=fc, stride_a=sa, stride_b=0, stride_c=sc, alpha=0.75, beta=0.5,
                           bias=bias, bias_rows=True, act="gelu_tanh",
                           strides=[(3, 17), (2, 2 * K + 3), (2 * N + 1, 2)])
    full = oracle_mod.gemm(p)
    bs, is_, js = np.meshgrid(np.arange(nb), np.arange(M), np.arange(N), indexing="ij")
    s = oracle_mod.gemm_sampled(p, bs.ravel(), is_.ravel(), js.ravel())
    assert np.array_equal(s, full.ravel())
    # and the full form against the dense definition, batch by batch
    for b in range(nb):
        dense = make_problem(oracle_mod, A[b], B, "bf16", "row", "row", C0=C0[b], alpha=0.75,
                             beta=0.5, bias=bias, bias_rows=True, act="gelu_tanh")
        assert np.array_equal(full[b], oracle_mod.gemm(dense)[0])
