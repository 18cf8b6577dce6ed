// True-fp32 GEMM on the CUDA cores (FFMA pipe; no tensor cores, no TF32).
//
// The register-tiled design of "2 . La GEMM, de zero a cuBLAS", sections
// 2.3-2.8, for sm_103a:
//   - a 128 x 128 output tile per CTA of 256 threads (section 2.6: BM = BN =
//     128, TM = TN = 8), K consumed 16 at a time (the page's BK = 8 doubled
//     to halve the synchronisations and tile loads per FMA);
//   - each thread accumulates an 8 x 8 block as outer products of 8 values of
//     A and 8 values of B per k: 16 shared-memory reads for 64 FMAs
//     (section 2.6); its rows are {4ty..4ty+3, 64+4ty..64+4ty+3} and its
//     columns {4tx..4tx+3, 64+4tx..64+4tx+3}, so every read is a float4 and
//     the reads of one warp touch each bank at most once per wavefront;
//   - the A tile is stored transposed, As[k][m], so a thread's column of A is
//     contiguous and vectorisable (section 2.7);
//   - global loads are float4 (LDG.128) when alignment allows (section 2.7)
//     and land in the second of two shared buffers while the first is
//     consumed (section 2.8), one __syncthreads per K step; the operand
//     fragments of step k+1 are also read while step k computes;
//   - one CTA per SM (up to 255 registers, no spills), which also gives more
//     waves and a smaller tail at 4096^2;
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

constexpr int SBM = 128, SBN = 128, SBK = 16, STHREADS = 256;

// Global -> register staging of one 128 x 16 A tile and one 16 x 128 B tile:
// two float4 of each per thread.  Mapping (thread t):
//   K-contiguous operand (row-major A, column-major B): row r = t % 64 (+64),
//     k offset 4 * (t / 64); a warp covers 32 consecutive rows at one k
//     offset, so the transposed shared-memory stores hit 32 distinct banks.
//   MN-contiguous operand: k = t / 32 (+8), mn offset 4 * (t % 32); a warp
//     reads 512 contiguous bytes and stores one float4 each.
struct Frag4 {
    float4 v[2];
};

template <bool KCONTIG>
__device__ __forceinline__ Frag4 load_tile(const float* __restrict__ X, int64_t ld, int mn0,
                                           int mn_ext, int k0, int K, bool vec_ok, int tid) {
    Frag4 f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (KCONTIG) {
            const int r = mn0 + (tid & 63) + 64 * h;
            const int k = k0 + ((tid >> 6) << 2);
            if (r < mn_ext) {
                const float* src = X + static_cast<int64_t>(r) * ld + k;
                if (vec_ok && k + 3 < K) {
                    v = *reinterpret_cast<const float4*>(src);
                } else {
                    if (k + 0 < K) v.x = src[0];
                    if (k + 1 < K) v.y = src[1];
                    if (k + 2 < K) v.z = src[2];
                    if (k + 3 < K) v.w = src[3];
                }
            }
        } else {
            const int k = k0 + (tid >> 5) + 8 * h;
            const int r = mn0 + ((tid & 31) << 2);
            if (k < K) {
                const float* src = X + static_cast<int64_t>(k) * ld + r;
                if (vec_ok && r + 3 < mn_ext) {
                    v = *reinterpret_cast<const float4*>(src);
                } else {
                    if (r + 0 < mn_ext) v.x = src[0];
                    if (r + 1 < mn_ext) v.y = src[1];
                    if (r + 2 < mn_ext) v.z = src[2];
                    if (r + 3 < mn_ext) v.w = src[3];
                }
            }
        }
        f.v[h] = v;
    }
    return f;
}

// Store a staged tile as S[k][mn] (k-major rows of 128 floats).
template <bool KCONTIG>
__device__ __forceinline__ void store_tile(float (*S)[SBM], const Frag4& f, int tid) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (KCONTIG) {
            const int r = (tid & 63) + 64 * h;
            const int k = (tid >> 6) << 2;
            S[k + 0][r] = f.v[h].x;
            S[k + 1][r] = f.v[h].y;
            S[k + 2][r] = f.v[h].z;
            S[k + 3][r] = f.v[h].w;
        } else {
            const int k = (tid >> 5) + 8 * h;
            const int r = (tid & 31) << 2;
            *reinterpret_cast<float4*>(&S[k][r]) = f.v[h];
        }
    }
}

template <bool A_ROW, bool B_ROW>
__global__ void __launch_bounds__(STHREADS, 1) sgemm_kernel(const __grid_constant__ SgemmParams p) {
    __shared__ __align__(16) float As[2][SBK][SBM];
    __shared__ __align__(16) float Bs[2][SBK][SBN];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int tiles = p.num_pid_m * p.num_pid_n;
    const int b = blockIdx.x / tiles;
    int pid_m, pid_n;
    tile_coord(blockIdx.x - b * tiles, p.num_pid_m, p.num_pid_n, p.group_m, pid_m, pid_n);
    const int m0 = pid_m * SBM, n0 = pid_n * SBN;
    const float* __restrict__ A = p.A + static_cast<int64_t>(b) * p.stride_a;
    const float* __restrict__ B = p.B + static_cast<int64_t>(b) * p.stride_b;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int nk = (p.K + SBK - 1) / SBK;
    // A is K-contiguous when row-major; B is K-contiguous when column-major
    Frag4 fa = load_tile<A_ROW>(A, p.lda, m0, p.M, 0, p.K, p.a_vec_ok, tid);
    Frag4 fb = load_tile<!B_ROW>(B, p.ldb, n0, p.N, 0, p.K, p.b_vec_ok, tid);
    store_tile<A_ROW>(As[0], fa, tid);
    store_tile<!B_ROW>(Bs[0], fb, tid);
    __syncthreads();

    for (int kt = 0; kt < nk; ++kt) {
        const int cur = kt & 1;
        const bool more = kt + 1 < nk;
        if (more) {
            fa = load_tile<A_ROW>(A, p.lda, m0, p.M, (kt + 1) * SBK, p.K, p.a_vec_ok, tid);
            fb = load_tile<!B_ROW>(B, p.ldb, n0, p.N, (kt + 1) * SBK, p.K, p.b_vec_ok, tid);
        }
        // outer products; the float4 fragments of step k+1 are read while step
        // k computes and are used in place (no copies between the load and the FMAs)
        float4 xa0[2], xa1[2], xb0[2], xb1[2];
        xa0[0] = *reinterpret_cast<const float4*>(&As[cur][0][ty * 4]);
        xa1[0] = *reinterpret_cast<const float4*>(&As[cur][0][64 + ty * 4]);
        xb0[0] = *reinterpret_cast<const float4*>(&Bs[cur][0][tx * 4]);
        xb1[0] = *reinterpret_cast<const float4*>(&Bs[cur][0][64 + tx * 4]);
#pragma unroll
        for (int k = 0; k < SBK; ++k) {
            const int c = k & 1;
            if (k + 1 < SBK) {
                xa0[c ^ 1] = *reinterpret_cast<const float4*>(&As[cur][k + 1][ty * 4]);
                xa1[c ^ 1] = *reinterpret_cast<const float4*>(&As[cur][k + 1][64 + ty * 4]);
                xb0[c ^ 1] = *reinterpret_cast<const float4*>(&Bs[cur][k + 1][tx * 4]);
                xb1[c ^ 1] = *reinterpret_cast<const float4*>(&Bs[cur][k + 1][64 + tx * 4]);
            }
            const float a[8] = {xa0[c].x, xa0[c].y, xa0[c].z, xa0[c].w,
                                xa1[c].x, xa1[c].y, xa1[c].z, xa1[c].w};
            const float bb[8] = {xb0[c].x, xb0[c].y, xb0[c].z, xb0[c].w,
                                 xb1[c].x, xb1[c].y, xb1[c].z, xb1[c].w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        if (more) {
            store_tile<A_ROW>(As[cur ^ 1], fa, tid);
            store_tile<!B_ROW>(Bs[cur ^ 1], fb, tid);
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
