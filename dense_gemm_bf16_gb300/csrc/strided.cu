// gemm_strided: the GEMM with every matrix given by element strides,
// element (r, c) of batch b at b*stride + r*rs + c*cs ("Skill: Write a Triton
// GEMM Kernel", Kernel design rules: strides are kernel arguments, so
// non-contiguous tensors work).
//
// A matrix whose strides describe a row-major (cs == 1) or column-major
// (rs == 1) layout with a valid leading dimension goes to gemm_batched as is.
// Any other operand is first gathered into a dense row-major copy in the
// caller's workspace; any other C is computed into a dense row-major buffer
// in the workspace (gathered from C first when beta != 0) and scattered back.
// The tensor-core and CUDA-core kernels see only dense layouts.
#include <stdint.h>

#include <algorithm>

#include "gemm.h"
#include "internal.h"
#include "span_check.h"

namespace dg {
namespace {

constexpr int kThreads = 256;

// dst[b][r][c] (pitch ld, batch pitch dbs) = src[b*bs + r*rs + c*cs].  One
// thread per column of a row; blocks walk rows and batches in grid-stride
// loops.  The writes are coalesced; the reads follow the caller's strides.
template <typename T>
__global__ void gather_kernel(const T* __restrict__ src, int64_t rs, int64_t cs, int64_t bs,
                              int64_t R, int64_t C, int64_t nb, T* __restrict__ dst, int64_t ld,
                              int64_t dbs) {
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= C) return;
    for (int64_t b = blockIdx.z; b < nb; b += gridDim.z)
        for (int64_t r = blockIdx.y; r < R; r += gridDim.y)
            dst[b * dbs + r * ld + c] = src[b * bs + r * rs + c * cs];
}

// The inverse: dst[b*bs + r*rs + c*cs] = src[b][r][c].
template <typename T>
__global__ void scatter_kernel(const T* __restrict__ src, int64_t ld, int64_t sbs, int64_t R,
                               int64_t C, int64_t nb, T* __restrict__ dst, int64_t rs, int64_t cs,
                               int64_t bs) {
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= C) return;
    for (int64_t b = blockIdx.z; b < nb; b += gridDim.z)
        for (int64_t r = blockIdx.y; r < R; r += gridDim.y)
            dst[b * bs + r * rs + c * cs] = src[b * sbs + r * ld + c];
}

dim3 copy_grid(int64_t R, int64_t C, int64_t nb) {
    const int64_t gx = (C + kThreads - 1) / kThreads;
    return dim3(static_cast<unsigned>(gx), static_cast<unsigned>(std::min<int64_t>(R, 65535)),
                static_cast<unsigned>(std::min<int64_t>(nb, 65535)));
}

cudaError_t gather(const void* src, int es, int64_t rs, int64_t cs, int64_t bs, int64_t R,
                   int64_t C, int64_t nb, void* dst, int64_t ld, int64_t dbs, cudaStream_t st) {
    if (R == 0 || C == 0 || nb == 0) return cudaSuccess;
    const dim3 g = copy_grid(R, C, nb);
    if (es == 2)
        gather_kernel<uint16_t><<<g, kThreads, 0, st>>>(static_cast<const uint16_t*>(src), rs, cs,
                                                       bs, R, C, nb, static_cast<uint16_t*>(dst),
                                                       ld, dbs);
    else
        gather_kernel<uint32_t><<<g, kThreads, 0, st>>>(static_cast<const uint32_t*>(src), rs, cs,
                                                       bs, R, C, nb, static_cast<uint32_t*>(dst),
                                                       ld, dbs);
    return cudaGetLastError();
}

cudaError_t scatter(const void* src, int es, int64_t ld, int64_t sbs, int64_t R, int64_t C,
                    int64_t nb, void* dst, int64_t rs, int64_t cs, int64_t bs, cudaStream_t st) {
    if (R == 0 || C == 0 || nb == 0) return cudaSuccess;
    const dim3 g = copy_grid(R, C, nb);
    if (es == 2)
        scatter_kernel<uint16_t><<<g, kThreads, 0, st>>>(static_cast<const uint16_t*>(src), ld,
                                                        sbs, R, C, nb, static_cast<uint16_t*>(dst),
                                                        rs, cs, bs);
    else
        scatter_kernel<uint32_t><<<g, kThreads, 0, st>>>(static_cast<const uint32_t*>(src), ld,
                                                        sbs, R, C, nb, static_cast<uint32_t*>(dst),
                                                        rs, cs, bs);
    return cudaGetLastError();
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// How one R x C matrix reaches gemm_batched: as row- or column-major storage
// with a leading dimension, or through a dense row-major copy of pitch `pitch`.
struct MatPlan {
    bool copy = false;
    gemm_layout_t layout = GEMM_ROW_MAJOR;
    int64_t ld = 0;
    int64_t pitch = 0;     // copy: elements per row
    int64_t batches = 0;   // copy: batches stored (1 when the batch stride is 0)
    size_t bytes = 0;      // copy: bytes of workspace, 256-aligned
};

MatPlan plan_matrix(int64_t R, int64_t C, int64_t rs, int64_t cs, int64_t bs, int64_t batch,
                    int es) {
    MatPlan m;
    const int64_t one = 1;
    if (cs == 1 && (rs >= C || R <= 1)) {
        m.layout = GEMM_ROW_MAJOR;
        m.ld = std::max({rs, C, one});
        return m;
    }
    if (rs == 1 && (cs >= R || C <= 1)) {
        m.layout = GEMM_COL_MAJOR;
        m.ld = std::max({cs, R, one});
        return m;
    }
    m.copy = true;
    m.layout = GEMM_ROW_MAJOR;
    m.pitch = round_up(std::max(C, one), 16 / es);  // 16-byte rows: TMA- and float4-friendly
    m.ld = m.pitch;
    m.batches = (batch > 1 && bs != 0) ? batch : 1;
    m.bytes = static_cast<size_t>(round_up(m.batches * R * m.pitch * es, 256));
    return m;
}

struct StridedPlan {
    MatPlan a, b, c;
    size_t inner_bytes = 0;
    size_t total = 0;
};

gemm_status_t make_strided_plan(gemm_dtype_t ab, gemm_dtype_t cdt, int64_t batch, int64_t M,
                                int64_t N, int64_t K, int64_t a_rs, int64_t a_cs, int64_t sa,
                                int64_t b_rs, int64_t b_cs, int64_t sb, int64_t c_rs,
                                int64_t c_cs, int64_t sc, int split_k, StridedPlan& sp) {
    if (ab != GEMM_DT_BF16 && ab != GEMM_DT_F16 && ab != GEMM_DT_F32) return GEMM_ERR_INVALID_ARG;
    if (cdt != GEMM_DT_BF16 && cdt != GEMM_DT_F16 && cdt != GEMM_DT_F32) return GEMM_ERR_INVALID_ARG;
    if (batch < 0 || M < 0 || N < 0 || K < 0 || split_k < 0) return GEMM_ERR_INVALID_ARG;
    if (a_rs < 0 || a_cs < 0 || sa < 0 || b_rs < 0 || b_cs < 0 || sb < 0 || c_rs < 0 ||
        c_cs < 0 || sc < 0)
        return GEMM_ERR_INVALID_ARG;
    // distinct output elements need distinct addresses along each extent
    if ((M > 1 && c_rs == 0) || (N > 1 && c_cs == 0) || (batch > 1 && sc == 0))
        return GEMM_ERR_INVALID_ARG;
    const int64_t lim = 0x7FFFFFFF;
    if (batch > lim || M > lim || N > lim || K > lim) return GEMM_ERR_INVALID_ARG;
    if (batch > 0 && M > 0 && N > 0) {
        if (!strided_span_ok(M, N, c_rs, c_cs, batch, sc) || !count_ok(batch, M, N))
            return GEMM_ERR_INVALID_ARG;
        if (K > 0 && (!strided_span_ok(M, K, a_rs, a_cs, batch, sa) ||
                      !strided_span_ok(K, N, b_rs, b_cs, batch, sb) ||
                      !count_ok(batch, M, K) || !count_ok(batch, K, N)))
            return GEMM_ERR_INVALID_ARG;
    }
    const int es_ab = ab == GEMM_DT_F32 ? 4 : 2;
    const int es_c = cdt == GEMM_DT_F32 ? 4 : 2;
    sp.a = plan_matrix(M, K, a_rs, a_cs, sa, batch, es_ab);
    sp.b = plan_matrix(K, N, b_rs, b_cs, sb, batch, es_ab);
    sp.c = plan_matrix(M, N, c_rs, c_cs, sc, batch, es_c);
    if (sp.c.copy) {
        sp.c.batches = std::max<int64_t>(batch, 1);
        sp.c.bytes = static_cast<size_t>(round_up(sp.c.batches * M * sp.c.pitch * es_c, 256));
    }
    sp.inner_bytes = gemm_workspace_size(ab, batch, M, N, K, split_k);
    sp.total = (sp.a.copy ? sp.a.bytes : 0) + (sp.b.copy ? sp.b.bytes : 0) +
               (sp.c.copy ? sp.c.bytes : 0) + sp.inner_bytes;
    return GEMM_OK;
}

}  // namespace
}  // namespace dg

extern "C" {

size_t gemm_strided_workspace_size(gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype, int64_t batch,
                                   int64_t M, int64_t N, int64_t K, int64_t a_rs, int64_t a_cs,
                                   int64_t stride_a, int64_t b_rs, int64_t b_cs, int64_t stride_b,
                                   int64_t c_rs, int64_t c_cs, int64_t stride_c, int split_k) {
    dg::StridedPlan sp;
    if (dg::make_strided_plan(ab_dtype, c_dtype, batch, M, N, K, a_rs, a_cs, stride_a, b_rs, b_cs,
                              stride_b, c_rs, c_cs, stride_c, split_k, sp) != GEMM_OK)
        return 0;
    return sp.total;
}

gemm_status_t gemm_strided(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N, int64_t K,
                           const void* A, int64_t a_rs, int64_t a_cs, int64_t stride_a,
                           const void* B, int64_t b_rs, int64_t b_cs, int64_t stride_b,
                           void* C, int64_t c_rs, int64_t c_cs, int64_t stride_c,
                           gemm_dtype_t c_dtype, float alpha, float beta, const float* bias,
                           gemm_epilogue_t epi, int split_k, void* workspace,
                           size_t workspace_bytes, gemm_stream_t stream) {
    using namespace dg;
    StridedPlan sp;
    gemm_status_t st = make_strided_plan(ab_dtype, c_dtype, batch, M, N, K, a_rs, a_cs, stride_a,
                                         b_rs, b_cs, stride_b, c_rs, c_cs, stride_c, split_k, sp);
    if (st != GEMM_OK) return st;
    if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
    const bool any_copy = sp.a.copy || sp.b.copy || sp.c.copy;
    if (!any_copy)
        return gemm_batched(ab_dtype, batch, M, N, K, A, sp.a.ld, sp.a.layout, stride_a, B,
                            sp.b.ld, sp.b.layout, stride_b, C, sp.c.ld, sp.c.layout, stride_c,
                            c_dtype, alpha, beta, bias, epi, split_k, workspace, workspace_bytes,
                            stream);
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return workspace == nullptr ? GEMM_ERR_WORKSPACE : GEMM_ERR_INVALID_ARG;
    const size_t copies = sp.total - sp.inner_bytes;
    if (workspace_bytes < copies) return GEMM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const int es_ab = ab_dtype == GEMM_DT_F32 ? 4 : 2;
    const int es_c = c_dtype == GEMM_DT_F32 ? 4 : 2;
    const bool need_ab = K > 0 && alpha != 0.0f;
    const void* a = A;
    const void* b = B;
    void* c = C;
    int64_t sa = stride_a, sb = stride_b, scc = stride_c;
    if (sp.a.copy) {
        if (need_ab && gather(A, es_ab, a_rs, a_cs, stride_a, M, K, sp.a.batches, ws, sp.a.pitch,
                              M * sp.a.pitch, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        a = ws;
        sa = sp.a.batches > 1 ? M * sp.a.pitch : 0;
        ws += sp.a.bytes;
    }
    if (sp.b.copy) {
        if (need_ab && gather(B, es_ab, b_rs, b_cs, stride_b, K, N, sp.b.batches, ws, sp.b.pitch,
                              K * sp.b.pitch, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        b = ws;
        sb = sp.b.batches > 1 ? K * sp.b.pitch : 0;
        ws += sp.b.bytes;
    }
    if (sp.c.copy) {
        if (beta != 0.0f && gather(C, es_c, c_rs, c_cs, stride_c, M, N, sp.c.batches, ws,
                                   sp.c.pitch, M * sp.c.pitch, s) != cudaSuccess)
            return GEMM_ERR_CUDA;
        c = ws;
        scc = M * sp.c.pitch;
        ws += sp.c.bytes;
    }
    st = gemm_batched(ab_dtype, batch, M, N, K, a, sp.a.ld, sp.a.layout, sa, b, sp.b.ld,
                      sp.b.layout, sb, c, sp.c.ld, sp.c.layout, scc, c_dtype, alpha, beta, bias,
                      epi, split_k, ws, workspace_bytes - copies, stream);
    if (st != GEMM_OK) return st;
    if (sp.c.copy && scatter(c, es_c, sp.c.pitch, M * sp.c.pitch, M, N, sp.c.batches, C, c_rs,
                             c_cs, stride_c, s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

gemm_status_t gemm_strided_plan_query(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N,
                                      int64_t K, const void* A, int64_t a_rs, int64_t a_cs,
                                      int64_t stride_a, const void* B, int64_t b_rs, int64_t b_cs,
                                      int64_t stride_b, void* C, int64_t c_rs, int64_t c_cs,
                                      int64_t stride_c, gemm_dtype_t c_dtype, float alpha,
                                      float beta, const float* bias, gemm_epilogue_t epi,
                                      int split_k, size_t workspace_bytes, gemm_plan_t* plan) {
    using namespace dg;
    if (plan == nullptr) return GEMM_ERR_INVALID_ARG;
    StridedPlan sp;
    gemm_status_t st = make_strided_plan(ab_dtype, c_dtype, batch, M, N, K, a_rs, a_cs, stride_a,
                                         b_rs, b_cs, stride_b, c_rs, c_cs, stride_c, split_k, sp);
    if (st != GEMM_OK) return st;
    const bool any_copy = sp.a.copy || sp.b.copy || sp.c.copy;
    const size_t copies = any_copy ? sp.total - sp.inner_bytes : 0;
    if (any_copy && workspace_bytes < copies) return GEMM_ERR_WORKSPACE;
    // the copies sit in the workspace, which is 256-byte aligned: planning reads
    // only the alignment of their addresses, so an aligned stand-in serves
    alignas(256) static const char copy_standin[256] = {0};
    const bool need_ab = K > 0 && alpha != 0.0f;
    const void* a = sp.a.copy ? static_cast<const void*>(copy_standin) : A;
    const void* b = sp.b.copy ? static_cast<const void*>(copy_standin) : B;
    void* c = sp.c.copy ? const_cast<char*>(copy_standin) : C;
    const int64_t sa = sp.a.copy ? (sp.a.batches > 1 ? M * sp.a.pitch : 0) : stride_a;
    const int64_t sb = sp.b.copy ? (sp.b.batches > 1 ? K * sp.b.pitch : 0) : stride_b;
    const int64_t sc = sp.c.copy ? M * sp.c.pitch : stride_c;
    st = gemm_plan_query(ab_dtype, batch, M, N, K, a, sp.a.ld, sp.a.layout, sa, b, sp.b.ld,
                         sp.b.layout, sb, c, sp.c.ld, sp.c.layout, sc, c_dtype, alpha, beta, bias,
                         epi, split_k, workspace_bytes - copies, plan);
    if (st != GEMM_OK) return st;
    if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
    plan->pack_a = plan->pack_a || sp.a.copy;
    plan->pack_b = plan->pack_b || sp.b.copy;
    plan->launches += (sp.a.copy && need_ab) + (sp.b.copy && need_ab) +
                      (sp.c.copy ? 1 + (beta != 0.0f) : 0);
    plan->workspace_bytes += static_cast<int64_t>(copies);
    return GEMM_OK;
}

}  // extern "C"
