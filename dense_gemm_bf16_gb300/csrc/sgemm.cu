// True-fp32 GEMM on the CUDA cores (FFMA pipe; no tensor cores, no TF32).
//
// The register-tiled design of "2 . La GEMM, de zero a cuBLAS", sections
// 2.3-2.8, for sm_103a:
//   - a 128 x 128 output tile per CTA of 256 threads, K consumed 8 at a time
//     (section 2.6: BM = BN = 128, BK = 8, TM = TN = 8);
//   - each thread accumulates an 8 x 8 block as outer products of 8 values of
//     A and 8 values of B per k: 16 shared-memory reads for 64 FMAs
//     (section 2.6); its rows are {4ty..4ty+3, 64+4ty..64+4ty+3} and its
//     columns {4tx..4tx+3, 64+4tx..64+4tx+3}, so every read is a float4 and
//     the reads of one warp touch each bank at most once per wavefront;
//   - the A tile is stored transposed, As[k][m], so a thread's column of A is
//     contiguous and vectorisable (section 2.7);
//   - global loads are float4 (LDG.128) when alignment allows (section 2.7)
//     and land in the second of two shared buffers while the first is
//     consumed (section 2.8), one __syncthreads per K step;
//   - consecutive threads read consecutive addresses of each operand row
//     (coalescing, section 2.3);
//   - ragged M / N / K edges are masked with zero fill, and the store is
//     masked on M and N.
// Tiles are ordered by the grouped schedule of tile_order.h; batch is the slowest
// index of the 1-D grid.
#include <stdint.h>

#include "epilogue.cuh"
#include "internal.h"
#include "tile_order.h"

namespace dg {
namespace {

constexpr int SBM = 128, SBN = 128, SBK = 8, STHREADS = 256;

template <bool A_ROW>
__device__ __forceinline__ float4 load_a(const SgemmParams& p, const float* A, int m0, int k0,
                                         int tid) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (A_ROW) {
        // 128 rows x 8 k: thread -> row tid/2, k offset 4*(tid%2), float4 along k
        const int m = m0 + (tid >> 1);
        const int k = k0 + ((tid & 1) << 2);
        if (m < p.M) {
            const float* src = A + static_cast<int64_t>(m) * p.lda + k;
            if (p.a_vec_ok && k + 3 < p.K) {
                v = *reinterpret_cast<const float4*>(src);
            } else {
                if (k + 0 < p.K) v.x = src[0];
                if (k + 1 < p.K) v.y = src[1];
                if (k + 2 < p.K) v.z = src[2];
                if (k + 3 < p.K) v.w = src[3];
            }
        }
    } else {
        // column-major A: 8 k x 128 m, thread -> k tid/32, m offset 4*(tid%32), float4 along m
        const int k = k0 + (tid >> 5);
        const int m = m0 + ((tid & 31) << 2);
        if (k < p.K) {
            const float* src = A + static_cast<int64_t>(k) * p.lda + m;
            if (p.a_vec_ok && m + 3 < p.M) {
                v = *reinterpret_cast<const float4*>(src);
            } else {
                if (m + 0 < p.M) v.x = src[0];
                if (m + 1 < p.M) v.y = src[1];
                if (m + 2 < p.M) v.z = src[2];
                if (m + 3 < p.M) v.w = src[3];
            }
        }
    }
    return v;
}

template <bool B_ROW>
__device__ __forceinline__ float4 load_b(const SgemmParams& p, const float* B, int n0, int k0,
                                         int tid) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (B_ROW) {
        // 8 k x 128 n: thread -> k tid/32, n offset 4*(tid%32), float4 along n
        const int k = k0 + (tid >> 5);
        const int n = n0 + ((tid & 31) << 2);
        if (k < p.K) {
            const float* src = B + static_cast<int64_t>(k) * p.ldb + n;
            if (p.b_vec_ok && n + 3 < p.N) {
                v = *reinterpret_cast<const float4*>(src);
            } else {
                if (n + 0 < p.N) v.x = src[0];
                if (n + 1 < p.N) v.y = src[1];
                if (n + 2 < p.N) v.z = src[2];
                if (n + 3 < p.N) v.w = src[3];
            }
        }
    } else {
        // column-major B: thread -> column n tid/2, k offset 4*(tid%2), float4 along k
        const int n = n0 + (tid >> 1);
        const int k = k0 + ((tid & 1) << 2);
        if (n < p.N) {
            const float* src = B + static_cast<int64_t>(n) * p.ldb + k;
            if (p.b_vec_ok && k + 3 < p.K) {
                v = *reinterpret_cast<const float4*>(src);
            } else {
                if (k + 0 < p.K) v.x = src[0];
                if (k + 1 < p.K) v.y = src[1];
                if (k + 2 < p.K) v.z = src[2];
                if (k + 3 < p.K) v.w = src[3];
            }
        }
    }
    return v;
}

template <bool A_ROW>
__device__ __forceinline__ void store_a(float (*As)[SBM], float4 v, int tid) {
    if (A_ROW) {
        const int m = tid >> 1, k = (tid & 1) << 2;
        As[k + 0][m] = v.x;
        As[k + 1][m] = v.y;
        As[k + 2][m] = v.z;
        As[k + 3][m] = v.w;
    } else {
        const int k = tid >> 5, m = (tid & 31) << 2;
        *reinterpret_cast<float4*>(&As[k][m]) = v;
    }
}

template <bool B_ROW>
__device__ __forceinline__ void store_b(float (*Bs)[SBN], float4 v, int tid) {
    if (B_ROW) {
        const int k = tid >> 5, n = (tid & 31) << 2;
        *reinterpret_cast<float4*>(&Bs[k][n]) = v;
    } else {
        const int n = tid >> 1, k = (tid & 1) << 2;
        Bs[k + 0][n] = v.x;
        Bs[k + 1][n] = v.y;
        Bs[k + 2][n] = v.z;
        Bs[k + 3][n] = v.w;
    }
}

template <bool A_ROW, bool B_ROW>
__global__ void __launch_bounds__(STHREADS, 2) sgemm_kernel(const __grid_constant__ SgemmParams p) {
    __shared__ __align__(16) float As[2][SBK][SBM];
    __shared__ __align__(16) float Bs[2][SBK][SBN];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int tiles = p.num_pid_m * p.num_pid_n;
    const int b = blockIdx.x / tiles;
    int pid_m, pid_n;
    tile_coord(blockIdx.x - b * tiles, p.num_pid_m, p.num_pid_n, p.group_m, pid_m, pid_n);
    const int m0 = pid_m * SBM, n0 = pid_n * SBN;
    const float* A = p.A + static_cast<int64_t>(b) * p.stride_a;
    const float* B = p.B + static_cast<int64_t>(b) * p.stride_b;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int nk = (p.K + SBK - 1) / SBK;
    float4 ra = load_a<A_ROW>(p, A, m0, 0, tid);
    float4 rb = load_b<B_ROW>(p, B, n0, 0, tid);
    store_a<A_ROW>(As[0], ra, tid);
    store_b<B_ROW>(Bs[0], rb, tid);
    __syncthreads();

    for (int kt = 0; kt < nk; ++kt) {
        const int cur = kt & 1;
        const bool more = kt + 1 < nk;
        if (more) {
            ra = load_a<A_ROW>(p, A, m0, (kt + 1) * SBK, tid);
            rb = load_b<B_ROW>(p, B, n0, (kt + 1) * SBK, tid);
        }
#pragma unroll
        for (int k = 0; k < SBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][64 + tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) {
            store_a<A_ROW>(As[cur ^ 1], ra, tid);
            store_b<B_ROW>(Bs[cur ^ 1], rb, tid);
        }
        __syncthreads();
    }

    // epilogue: rows 4ty+i (+64), columns 4tx+j (+64)
    const Epilogue& e = p.epi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= p.M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h * 64 + tx * 4;
            if (e.c_row_major && e.c_vec_ok && n + 3 < p.N) {
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = e.alpha * acc[i][4 * h + j];
                float4* c = reinterpret_cast<float4*>(c_addr(e, b, m, n));
                if (e.beta != 0.f) {
                    const float4 o = *c;
                    v[0] = fmaf(e.beta, o.x, v[0]);
                    v[1] = fmaf(e.beta, o.y, v[1]);
                    v[2] = fmaf(e.beta, o.z, v[2]);
                    v[3] = fmaf(e.beta, o.w, v[3]);
                }
                if (e.bias) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] += e.bias[n + j];
                }
                if (e.act == ACT_GELU_TANH) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) v[j] = gelu_tanh(v[j]);
                }
                *c = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < p.N) epilogue_store(e, b, m, n + j, acc[i][4 * h + j]);
            }
        }
    }
}

}  // namespace

cudaError_t sgemm_launch(const SgemmParams& p, cudaStream_t stream) {
    const int64_t grid = static_cast<int64_t>(p.batch) * p.num_pid_m * p.num_pid_n;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const dim3 g(static_cast<unsigned>(grid));
    if (p.a_row && p.b_row)
        sgemm_kernel<true, true><<<g, STHREADS, 0, stream>>>(p);
    else if (p.a_row)
        sgemm_kernel<true, false><<<g, STHREADS, 0, stream>>>(p);
    else if (p.b_row)
        sgemm_kernel<false, true><<<g, STHREADS, 0, stream>>>(p);
    else
        sgemm_kernel<false, false><<<g, STHREADS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dg
