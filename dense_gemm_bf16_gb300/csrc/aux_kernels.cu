// Memory-bound helper kernels of the GEMM path.
//
//  pack16      copies a 16-bit operand whose base or leading dimension TMA
//              cannot address (not 16-byte aligned) into a dense, aligned
//              buffer of the caller's workspace.  Reads and writes are
//              coalesced along the contiguous dimension.
//  splitk_epi  the second pass of split-K ("Skill: Write a Triton GEMM
//              Kernel", Kernel design rules, split-K): sums the fp32 partial
//              tiles of all K slices in a fixed order (deterministic), then
//              applies the epilogue and the single downcast.  With zero
//              slices it is the K == 0 / alpha == 0 path: C = act(beta*C + bias).
//              With 8 or more slices and a row-major C, eight lanes share
//              each group of four outputs: lane g sums slices g, g + 8, ...,
//              and the eight sums combine by a fixed shuffle tree, so that a
//              small output still spreads over the whole GPU.
#include <stdint.h>

#include "epilogue.cuh"
#include "ptx.cuh"
#include "internal.h"

namespace dg {
namespace {

constexpr int kThreads = 256;

// grid: x covers the contiguous dimension in groups of 8 elements, y groups of
// 4 rows (grid-stride), z the batch.  A thread copies 8 consecutive elements
// of each of its rows: 2-byte loads (the source rows need only be 2-byte
// aligned; a warp's loads still cover 512 contiguous bytes) and one 16-byte
// store (the destination pitch is a multiple of 8 elements and its base
// 256-byte aligned).  Columns past `cols` in the last group are written as 0.
// The GEMM that reads the copy may be launched as this grid's programmatic
// dependent: it is let in at once, sets itself up while the copy runs, and
// waits for the copy's completion before its first operand load.
__global__ void __launch_bounds__(kThreads) pack16_kernel(const uint16_t* __restrict__ src,
                                                          int64_t ld, int64_t stride, int64_t rows,
                                                          int64_t cols, uint16_t* __restrict__ dst,
                                                          int64_t ld_dst) {
    griddep_launch_dependents();
    const int64_t b = blockIdx.z;
    const int64_t c0 = 8 * (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x);
    if (c0 >= cols) return;
    const uint16_t* s = src + b * stride + c0;
    uint16_t* d = dst + b * rows * ld_dst + c0;
    const int nc = cols - c0 < 8 ? static_cast<int>(cols - c0) : 8;
    for (int64_t r0 = 4 * static_cast<int64_t>(blockIdx.y); r0 < rows; r0 += 4 * gridDim.y) {
        uint32_t w[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint16_t* sr = s + (r0 + u) * ld;
            const bool row_ok = r0 + u < rows;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t lo = row_ok && 2 * h < nc ? __ldg(sr + 2 * h) : 0u;
                const uint32_t hi = row_ok && 2 * h + 1 < nc ? __ldg(sr + 2 * h + 1) : 0u;
                w[u][h] = lo | (hi << 16);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (r0 + u < rows)
                *reinterpret_cast<uint4*>(d + (r0 + u) * ld_dst) =
                    make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]);
    }
}

__global__ void __launch_bounds__(kThreads) splitk_epi_kernel(const float* __restrict__ P,
                                                              int splits, int64_t batch, int64_t M,
                                                              int64_t N, Epilogue e) {
    const int64_t mn = M * N;
    const int64_t total = batch * mn;
    for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // idx walks C's own layout densely, so partial reads are coalesced
        const int64_t b = idx / mn;
        const int64_t rem = idx - b * mn;
        int64_t i, j;
        if (e.c_row_major) {
            i = rem / N;
            j = rem - i * N;
        } else {
            j = rem / M;
            i = rem - j * M;
        }
        float acc = 0.0f;
        for (int s = 0; s < splits; ++s) acc += P[static_cast<int64_t>(s) * total + idx];
        epilogue_store(e, b, i, j, acc);
    }
}

// Four consecutive elements of one row per thread (row-major C, N % 4 == 0):
// 16-byte partial loads, eight slices in flight at a time, summed in slice order.
__global__ void __launch_bounds__(kThreads) splitk_epi_vec4_kernel(const float* __restrict__ P,
                                                                   int splits, int64_t batch,
                                                                   int64_t M, int64_t N,
                                                                   Epilogue e) {
    const int64_t mn = M * N;
    const int64_t total = batch * mn;
    const int64_t total4 = total >> 2;
    const float4* __restrict__ P4 = reinterpret_cast<const float4*>(P);
    for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < total4;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int s = 0;
        for (; s + 8 <= splits; s += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = P4[static_cast<int64_t>(s + u) * total4 + q];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
        for (; s < splits; ++s) {
            const float4 v = P4[static_cast<int64_t>(s) * total4 + q];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const int64_t idx = q << 2;
        const int64_t b = idx / mn;
        const int64_t rem = idx - b * mn;
        const int64_t i = rem / N;
        const int64_t j = rem - i * N;
        epilogue_store(e, b, i, j + 0, acc.x);
        epilogue_store(e, b, i, j + 1, acc.y);
        epilogue_store(e, b, i, j + 2, acc.z);
        epilogue_store(e, b, i, j + 3, acc.w);
    }
}

// Eight lanes per float4 of outputs: lane g of the group adds slices
// g, g + 8, g + 16, ... in ascending order, then the group adds its eight sums
// pairwise (distance 4, 2, 1), and lane 0 writes the four results.
__global__ void __launch_bounds__(kThreads) splitk_epi_group8_kernel(const float* __restrict__ P,
                                                                     int splits, int64_t batch,
                                                                     int64_t M, int64_t N,
                                                                     Epilogue e) {
    const int64_t mn = M * N;
    const int64_t total4 = (batch * mn) >> 2;
    const float4* __restrict__ P4 = reinterpret_cast<const float4*>(P);
    const int g = threadIdx.x & 7;
    const int64_t groups = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 3);
    for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x >> 3) + (threadIdx.x >> 3);
         q - (threadIdx.x >> 3) < total4; q += groups) {
        // every lane of the warp stays in the loop for the shuffles
        const bool live = q < total4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
            int s = g;
            for (; s + 24 < splits; s += 32) {
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = P4[static_cast<int64_t>(s + 8 * u) * total4 + q];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc.x += v[u].x;
                    acc.y += v[u].y;
                    acc.z += v[u].z;
                    acc.w += v[u].w;
                }
            }
            for (; s < splits; s += 8) {
                const float4 v = P4[static_cast<int64_t>(s) * total4 + q];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
        }
#pragma unroll
        for (int d = 4; d >= 1; d >>= 1) {
            acc.x += __shfl_down_sync(0xffffffffu, acc.x, d, 8);
            acc.y += __shfl_down_sync(0xffffffffu, acc.y, d, 8);
            acc.z += __shfl_down_sync(0xffffffffu, acc.z, d, 8);
            acc.w += __shfl_down_sync(0xffffffffu, acc.w, d, 8);
        }
        if (live && g == 0) {
            const int64_t idx = q << 2;
            const int64_t b = idx / mn;
            const int64_t rem = idx - b * mn;
            const int64_t i = rem / N;
            const int64_t j = rem - i * N;
            epilogue_store(e, b, i, j + 0, acc.x);
            epilogue_store(e, b, i, j + 1, acc.y);
            epilogue_store(e, b, i, j + 2, acc.z);
            epilogue_store(e, b, i, j + 3, acc.w);
        }
    }
}

int grid_for(int64_t total) {
    int64_t g = (total + kThreads - 1) / kThreads;
    if (g > 152 * 32) g = 152 * 32;  // grid-stride beyond a few waves of the 152 SMs
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t pack16_launch(const void* src, int64_t ld, int64_t stride, int64_t rows, int64_t cols,
                          int64_t batch, void* dst, int64_t ld_dst, cudaStream_t stream) {
    if (batch <= 0 || rows <= 0 || cols <= 0) return cudaSuccess;
    if (batch > 65535) return cudaErrorInvalidValue;
    if ((ld_dst & 7) != 0 || (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
        return cudaErrorInvalidValue;  // the 16-byte stores need an aligned destination
    const int64_t gx = ((cols + 7) / 8 + kThreads - 1) / kThreads;
    const int64_t groups = (rows + 3) / 4;
    const int64_t gy = groups < 4096 ? groups : 4096;
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
    pack16_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                         static_cast<unsigned>(batch)),
                    kThreads, 0, stream>>>(static_cast<const uint16_t*>(src), ld, stride, rows,
                                           cols, static_cast<uint16_t*>(dst), ld_dst);
    return cudaGetLastError();
}

cudaError_t splitk_epilogue_launch(const float* partials, int splits, int64_t batch, int64_t M,
                                   int64_t N, const Epilogue& e, cudaStream_t stream) {
    const int64_t total = batch * M * N;
    if (total <= 0) return cudaSuccess;
    if (partials && e.c_row_major && (N & 3) == 0 && splits >= 8) {
        splitk_epi_group8_kernel<<<grid_for(total << 1), kThreads, 0, stream>>>(partials, splits,
                                                                               batch, M, N, e);
    } else if (partials && e.c_row_major && (N & 3) == 0) {
        splitk_epi_vec4_kernel<<<grid_for(total >> 2), kThreads, 0, stream>>>(partials, splits, batch,
                                                                              M, N, e);
    } else {
        splitk_epi_kernel<<<grid_for(total), kThreads, 0, stream>>>(partials, splits, batch, M, N,
                                                                    e);
    }
    return cudaGetLastError();
}

}  // namespace dg
