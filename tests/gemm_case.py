"""One GEMM test case: seeded storage buffers (any layout, padding, batch stride,
pointer offset), the oracle's answer on the same bits, and the CUDA path's
answer through the C ABI (``gemm_batched``).  Shared by the GPU tests, the
smoke test and the bench's correctness checks."""
from __future__ import annotations

import numpy as np

import datagen
import oracle

ES = {"bf16": 2, "f16": 2, "f32": 4}
NAN_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}
DT_CODE = {"bf16": 0, "f16": 1, "f32": 2}
LAYOUT = {"row": 0, "col": 1}
ACT_CODE = {"none": 0, "gelu_tanh": 1, "relu": 2, "gelu_erf": 3}


def epi_code(use_bias, act, row_bias=False):
    """gemm_epilogue_t: bit 0 bias, bits 1-2 activation, bit 3 bias along rows."""
    return (1 if use_bias else 0) | (ACT_CODE[act] << 1) | (8 if row_bias else 0)


def _values(kind, seed, shape, K):
    if kind == "ints":
        return datagen.small_ints(seed, shape, -4, 4)
    if kind == "scaled":
        return datagen.uniform(seed, shape) / np.sqrt(K)
    if kind == "normal":
        return datagen.normal(seed, shape)
    return datagen.uniform(seed, shape)


def _poison(n, dt):
    if dt in ("bf16", "f16"):
        return np.full(n, NAN_BITS[dt], dtype=np.uint16)
    return np.full(n, np.nan, dtype=np.float32)


def store(enc, dt, layout, pad, offset, nb_alloc):
    """enc: encoded [nb, R, C] storage values.  Returns (flat, ld, stride, offset)."""
    nb, R, C = enc.shape
    ld = (C if layout == "row" else R) + pad
    outer = R if layout == "row" else C
    stride = outer * ld
    flat = _poison(offset + max(nb_alloc * stride, 1) + 64, dt)
    for b in range(nb):
        blk = enc[b] if layout == "row" else enc[b].T
        rows, cols = blk.shape
        base = offset + b * stride
        view = flat[base: base + rows * ld].reshape(rows, ld)
        view[:, :cols] = blk
    return flat, ld, stride, offset


def read(flat, dt, layout, ld, stride, offset, nb, R, C):
    """Logical [nb, R, C] fp64 values of a storage buffer."""
    out = np.empty((nb, R, C), dtype=np.float64)
    for b in range(nb):
        base = offset + b * stride
        if layout == "row":
            blk = flat[base: base + R * ld].reshape(R, ld)[:, :C]
        else:
            blk = flat[base: base + C * ld].reshape(C, ld)[:, :R].T
        if dt == "bf16":
            out[b] = datagen.bf16_bits_to_f32(np.ascontiguousarray(blk))
        elif dt == "f16":
            out[b] = datagen.f16_bits_to_f32(np.ascontiguousarray(blk))
        else:
            out[b] = blk
    return out


class Case:
    def __init__(self, ab="bf16", M=64, N=64, K=64, *, batch=1, la="row", lb="row", lc="row",
                 c_dtype="f32", pads=(0, 0, 0), offsets=(0, 0, 0), alpha=1.0, beta=0.0,
                 bias=False, act="none", row_bias=False, broadcast_b=False, values="uniform",
                 c_values="normal",
                 seed=1, split_k=0):
        self.ab, self.M, self.N, self.K, self.batch = ab, M, N, K, batch
        self.la, self.lb, self.lc, self.c_dtype = la, lb, lc, c_dtype
        self.alpha, self.beta, self.act, self.split_k = alpha, beta, act, split_k
        self.use_bias = bias
        self.row_bias = bool(row_bias and bias)
        sa, sb, sc, sbias = (seed * 10 + r for r in range(4))
        nb_b = 1 if broadcast_b else batch
        A = datagen.encode(_values(values, sa, (batch, M, K), K), ab)
        B = datagen.encode(_values(values, sb, (nb_b, K, N), K), ab)
        self.A, self.lda, self.stride_a, self.off_a = store(A, ab, la, pads[0], offsets[0], batch)
        self.B, self.ldb, self.stride_b, self.off_b = store(B, ab, lb, pads[1], offsets[1], nb_b)
        if broadcast_b:
            self.stride_b = 0
        if beta != 0.0:
            C0 = datagen.encode(_values(c_values, sc, (batch, M, N), K), c_dtype)
        else:
            C0 = _poison(batch * M * N, c_dtype).reshape(batch, M, N)  # must not be read
        self.C0, self.ldc, self.stride_c, self.off_c = store(C0, c_dtype, lc, pads[2], offsets[2],
                                                            batch)
        self.bias = (datagen.to_f32(datagen.normal(sbias, (M if self.row_bias else N,)))
                     if bias else None)

    # ------------------------------------------------------------------ oracle
    def problem(self):
        return oracle.Problem(
            ab_dtype=self.ab, M=self.M, N=self.N, K=self.K, batch=self.batch,
            A=self.A[self.off_a:], lda=self.lda, la=self.la, stride_a=self.stride_a,
            B=self.B[self.off_b:], ldb=self.ldb, lb=self.lb, stride_b=self.stride_b,
            c_dtype=self.c_dtype, C0=self.C0[self.off_c:] if self.beta != 0.0 else None,
            ldc=self.ldc, lc=self.lc, stride_c=self.stride_c, alpha=self.alpha, beta=self.beta,
            bias=self.bias, act=self.act, bias_rows=self.row_bias)

    def oracle_full(self):
        return oracle.gemm(self.problem())

    def oracle_sampled(self, b, i, j):
        return oracle.gemm_sampled(self.problem(), b, i, j)

    # ------------------------------------------------------------------ GPU
    def run_gpu(self, stream=None, workspace=None, L=None):
        """Runs through the C ABI; returns (status, C storage after the call).
        L: a loaded library (ctypes) to call instead of the product one, e.g.
        the debug build."""
        import ctypes

        import torch
        import dense_gemm_bf16_gb300 as dg
        L = L or dg.lib()

        def up(flat):
            t = torch.from_numpy(flat.copy())
            return t.cuda()
        dA, dB, dC = up(self.A), up(self.B), up(self.C0)
        dbias = torch.from_numpy(self.bias).cuda() if self.bias is not None else None
        es = ES[self.ab]
        pa = dA.data_ptr() + self.off_a * es
        pb = dB.data_ptr() + self.off_b * es
        pc = dC.data_ptr() + self.off_c * ES[self.c_dtype]
        epi = epi_code(self.use_bias, self.act, self.row_bias)
        args = [DT_CODE[self.ab], self.batch, self.M, self.N, self.K,
                pa, self.lda, LAYOUT[self.la], self.stride_a if self.batch > 1 else 0,
                pb, self.ldb, LAYOUT[self.lb], self.stride_b if self.batch > 1 else 0,
                pc, self.ldc, LAYOUT[self.lc], self.stride_c if self.batch > 1 else 0,
                DT_CODE[self.c_dtype], self.alpha, self.beta,
                dbias.data_ptr() if dbias is not None else None, epi, self.split_k]
        if workspace is None:
            plan = dg.Plan()
            st = L.gemm_plan_query(*args, 1 << 62, ctypes.byref(plan))
            self.plan = plan.as_dict()
            need = int(plan.workspace_bytes) if st == 0 else 0
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        st = L.gemm_batched(*args, workspace.data_ptr(), workspace.numel(), stream)
        torch.cuda.synchronize()
        out = dC.cpu().numpy()
        return st, out

    def result(self, out):
        return read(out, self.c_dtype, self.lc, self.ldc, self.stride_c, self.off_c, self.batch,
                    self.M, self.N)

    def untouched_padding(self, out):
        """Every element of C's buffer outside the logical matrix still holds its poison."""
        mask = np.ones(out.shape[0], dtype=bool)
        for b in range(self.batch):
            base = self.off_c + b * self.stride_c
            outer = self.M if self.lc == "row" else self.N
            inner = self.N if self.lc == "row" else self.M
            for r in range(outer):
                mask[base + r * self.ldc: base + r * self.ldc + inner] = False
        if self.c_dtype == "f32":
            return bool(np.all(np.isnan(out[mask])))
        return bool(np.all(out[mask] == NAN_BITS[self.c_dtype]))

    # ------------------------------------------------------------------ tolerance
    def scale(self):
        """sqrt(K)-growth scale of one output: sqrt(K)|alpha| max|A| max|B| + |beta| max|C0| + max|bias|."""
        a = np.abs(read(self.A, self.ab, self.la, self.lda, self.stride_a, self.off_a, self.batch,
                        self.M, self.K)).max() if self.M * self.K else 0.0
        nb = 1 if self.stride_b == 0 else self.batch
        b = np.abs(read(self.B, self.ab, self.lb, self.ldb, self.stride_b, self.off_b, nb, self.K,
                        self.N)).max() if self.K * self.N else 0.0
        s = np.sqrt(self.K) * abs(self.alpha) * a * b
        if self.beta != 0.0:
            s += abs(self.beta) * np.abs(read(self.C0, self.c_dtype, self.lc, self.ldc,
                                              self.stride_c, self.off_c, self.batch, self.M,
                                              self.N)).max()
        if self.bias is not None:
            s += np.abs(self.bias).max()
        return max(float(s), 1e-30)


def check_close(case: Case, got: np.ndarray, ref: np.ndarray):
    """The stated tolerances: 16-bit outputs |err| <= 1e-2 + 1e-2|ref|; fp32
    outputs max|err| / scale <= 1e-4 with the sqrt(K) scale of Case.scale()."""
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    if case.c_dtype in ("bf16", "f16"):
        bad = err > 1e-2 + 1e-2 * np.abs(ref)
        assert not bad.any(), (f"{bad.sum()} elements out of tolerance, worst err "
                               f"{err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    else:
        rel = err.max() / case.scale() if err.size else 0.0
        assert rel <= 1e-4, f"normalised max error {rel:.3g} > 1e-4"
