/*
 * CPU oracle for the dense GEMM  C = epi(alpha * A @ B + beta * C0 + bias).
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference leg load this library.  It shares no
 * code, header, table or helper with the CUDA library; it decodes the
 * storage formats itself and accumulates in fp64.
 *
 * What it computes (the plain definition, not an algorithm):
 *   BLAS level-3 GEMM, "2 . La GEMM, de zero a cuBLAS", section 2.1:
 *       C(MxN) = alpha * A(MxK) B(KxN) + beta * C
 *   with the fused epilogue of "Skill: Write a Triton GEMM Kernel",
 *   Required reasoning process step 6 (alpha scaling, bias, activation,
 *   applied after the K loop) and Common failure modes (beta*C applied once,
 *   after accumulation):
 *       R[b,i,j] = act( alpha * sum_k A[b,i,k] * B[b,k,j] + beta * C0[b,i,j] + bias )
 *   - the sum runs over k = 0..K-1 in ascending order, in double;
 *     bf16 / fp16 / fp32 inputs widen to double exactly.  The pages ask the
 *     kernel for an fp32 accumulator at least ("GEMM Kernel Optimization",
 *     Core Technique) and ask for a float64 reference to check it against
 *     ("Skill: Write a Triton GEMM Kernel", Required reasoning process,
 *     step 8).
 *   - act is the identity, GELU with the tanh form
 *       gelu_tanh(x) = 0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) )),
 *     GELU itself, gelu_erf(x) = x Phi(x) = 0.5 x (1 + erf(x / sqrt(2)))
 *     (Hendrycks & Gimpel, "Gaussian Error Linear Units", 2016, defines the
 *     second and gives the first as its approximation; the pages name no
 *     GELU variant), or the rectifier relu(x) = x for x > 0, else 0 (so NaN
 *     maps to 0).  The pages ask for "an activation function" in the
 *     epilogue without naming one ("Skill: Write a Triton GEMM Kernel",
 *     Inputs the agent should gather first, item 5).
 *   - bias is an fp32 vector added before the activation and not scaled by
 *     alpha: bias[j] (length N, the same for every row) or, with bias_rows,
 *     bias[i] (length M, the same for every column).
 *   - beta == 0 means C0 is not read (BLAS convention): NaN in C0 does not
 *     propagate.  K == 0 gives act(beta * C0 + bias).
 *   - storage: element (r, c) of batch b sits at index
 *     b*stride + r*rs + c*cs.  A row-major matrix with leading dimension ld
 *     has (rs, cs) = (ld, 1), a column-major one (1, ld); oracle_gemm_strided
 *     takes any (rs, cs) ("Skill: Write a Triton GEMM Kernel", Kernel design
 *     rules: strides are arguments, so non-contiguous tensors work).  Batch
 *     stride 0 broadcasts ("Skill: Write a Triton GEMM Kernel", Correctness
 *     requirements, batched GEMM).
 *
 * The loop visits rows of A one at a time and, for each k in ascending
 * order, adds A[i,k]*B[k,j] into a row of fp64 accumulators: per element this
 * is the same ascending-k sum as the textbook i-j-k triple loop (the naive
 * kernel of "2 . La GEMM, de zero a cuBLAS", section 2.2), only with B read
 * row by row.  Single-threaded on purpose.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* storage types (the oracle's own numbering) */
enum { OR_BF16 = 0, OR_F16 = 1, OR_F32 = 2, OR_F64 = 3 };
/* layouts */
enum { OR_ROW = 0, OR_COL = 1 };
/* activations */
enum { OR_ACT_NONE = 0, OR_ACT_GELU_TANH = 1, OR_ACT_RELU = 2, OR_ACT_GELU_ERF = 3 };

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
double oracle_decode_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double load_elem(const void* base, int dt, int64_t idx) {
    switch (dt) {
    case OR_BF16: return oracle_decode_bf16(((const uint16_t*)base)[idx]);
    case OR_F16:  return oracle_decode_f16(((const uint16_t*)base)[idx]);
    case OR_F32:  return (double)((const float*)base)[idx];
    default:      return ((const double*)base)[idx];
    }
}

/* element (r, c) of batch b of a matrix stored with strides (rs, cs, stride) */
static double mat(const void* base, int dt, int64_t rs, int64_t cs, int64_t stride,
                  int64_t b, int64_t r, int64_t c) {
    int64_t idx = b * stride + r * rs + c * cs;
    return load_elem(base, dt, idx);
}

/* (row stride, column stride) of a matrix stored with (ld, layout) */
static void strides_of(int layout, int64_t ld, int64_t* rs, int64_t* cs) {
    *rs = layout == OR_ROW ? ld : 1;
    *cs = layout == OR_ROW ? 1 : ld;
}

double oracle_gelu_tanh(double x) {
    const double k0 = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(k0 * (x + 0.044715 * x * x * x)));
}

double oracle_gelu_erf(double x) {
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

double oracle_relu(double x) {
    return x > 0.0 ? x : 0.0;
}

static double epilogue(double acc, double alpha, double beta, const void* C0, int c_dt,
                       int64_t crs, int64_t ccs, int64_t sc, int64_t b, int64_t i, int64_t j,
                       const float* bias, int bias_rows, int act) {
    double v = alpha * acc;
    if (beta != 0.0) v += beta * mat(C0, c_dt, crs, ccs, sc, b, i, j);
    if (bias) v += (double)bias[bias_rows ? i : j];
    if (act == OR_ACT_GELU_TANH) v = oracle_gelu_tanh(v);
    else if (act == OR_ACT_RELU) v = oracle_relu(v);
    else if (act == OR_ACT_GELU_ERF) v = oracle_gelu_erf(v);
    return v;
}

/*
 * Full result, written dense row-major into R[batch][M][N] (fp64).
 * Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 */
int oracle_gemm_strided(int ab_dt, int c_dt, int64_t batch, int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t ars, int64_t acs, int64_t sa,
                        const void* B, int64_t brs, int64_t bcs, int64_t sb,
                        const void* C0, int64_t crs, int64_t ccs, int64_t sc,
                        double alpha, double beta, const float* bias, int bias_rows, int act,
                        double* R) {
    if (batch < 0 || M < 0 || N < 0 || K < 0 || !R) return -1;
    if (beta != 0.0 && !C0) return -1;
    double* acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!acc) return -2;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t i = 0; i < M; ++i) {
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = mat(A, ab_dt, ars, acs, sa, b, i, k);
                for (int64_t j = 0; j < N; ++j)
                    acc[j] += a * mat(B, ab_dt, brs, bcs, sb, b, k, j);
            }
            for (int64_t j = 0; j < N; ++j)
                R[(b * M + i) * N + j] =
                    epilogue(acc[j], alpha, beta, C0, c_dt, crs, ccs, sc, b, i, j, bias, bias_rows,
                             act);
        }
    }
    free(acc);
    return 0;
}

/*
 * Selected elements only: out[s] = R[bs[s], is[s], js[s]], each computed one
 * by one with the same ascending-k fp64 sum (for checks at full size).
 */
int oracle_gemm_strided_sampled(int ab_dt, int c_dt, int64_t batch, int64_t M, int64_t N,
                                int64_t K, const void* A, int64_t ars, int64_t acs, int64_t sa,
                                const void* B, int64_t brs, int64_t bcs, int64_t sb,
                                const void* C0, int64_t crs, int64_t ccs, int64_t sc,
                                double alpha, double beta, const float* bias, int bias_rows,
                                int act, int64_t nsamples, const int64_t* bs, const int64_t* is,
                                const int64_t* js, double* out) {
    if (batch < 0 || M < 0 || N < 0 || K < 0 || nsamples < 0 || !out) return -1;
    if (beta != 0.0 && !C0) return -1;
    for (int64_t s = 0; s < nsamples; ++s) {
        int64_t b = bs ? bs[s] : 0, i = is[s], j = js[s];
        if (b < 0 || b >= batch || i < 0 || i >= M || j < 0 || j >= N) return -1;
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += mat(A, ab_dt, ars, acs, sa, b, i, k) * mat(B, ab_dt, brs, bcs, sb, b, k, j);
        out[s] = epilogue(acc, alpha, beta, C0, c_dt, crs, ccs, sc, b, i, j, bias, bias_rows, act);
    }
    return 0;
}

/* The same two functions with every matrix given as (ld, layout). */
int oracle_gemm(int ab_dt, int c_dt, int64_t batch, int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, int la, int64_t sa,
                const void* B, int64_t ldb, int lb, int64_t sb,
                const void* C0, int64_t ldc, int lc, int64_t sc,
                double alpha, double beta, const float* bias, int bias_rows, int act, double* R) {
    int64_t ars, acs, brs, bcs, crs, ccs;
    strides_of(la, lda, &ars, &acs);
    strides_of(lb, ldb, &brs, &bcs);
    strides_of(lc, ldc, &crs, &ccs);
    return oracle_gemm_strided(ab_dt, c_dt, batch, M, N, K, A, ars, acs, sa, B, brs, bcs, sb,
                               C0, crs, ccs, sc, alpha, beta, bias, bias_rows, act, R);
}

int oracle_gemm_sampled(int ab_dt, int c_dt, int64_t batch, int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, int la, int64_t sa,
                        const void* B, int64_t ldb, int lb, int64_t sb,
                        const void* C0, int64_t ldc, int lc, int64_t sc,
                        double alpha, double beta, const float* bias, int bias_rows, int act,
                        int64_t nsamples, const int64_t* bs, const int64_t* is,
                        const int64_t* js, double* out) {
    int64_t ars, acs, brs, bcs, crs, ccs;
    strides_of(la, lda, &ars, &acs);
    strides_of(lb, ldb, &brs, &bcs);
    strides_of(lc, ldc, &crs, &ccs);
    return oracle_gemm_strided_sampled(ab_dt, c_dt, batch, M, N, K, A, ars, acs, sa, B, brs, bcs,
                                       sb, C0, crs, ccs, sc, alpha, beta, bias, bias_rows, act,
                                       nsamples, bs, is, js, out);
}
