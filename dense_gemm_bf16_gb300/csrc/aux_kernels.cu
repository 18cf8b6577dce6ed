// Memory-bound helper kernels of the GEMM path.
//
//  pack16      copies a 16-bit operand whose base or leading dimension TMA
//              cannot address (not 16-byte aligned) into a dense, aligned
//              buffer of the caller's workspace.  Reads and writes are
//              coalesced along the contiguous dimension.
//  splitk_epi  the second pass of split-K ("Skill: Write a Triton GEMM
//              Kernel", Kernel design rules, split-K): sums the fp32 partial
//              tiles of all K slices in slice order (deterministic), then
//              applies the epilogue and the single downcast.  With zero
//              slices it is the K == 0 / alpha == 0 path: C = act(beta*C + bias).
#include <stdint.h>

#include "epilogue.cuh"
#include "internal.h"

namespace dg {
namespace {

constexpr int kThreads = 256;

// grid: x covers the contiguous dimension, y the rows (grid-stride), z the batch
__global__ void __launch_bounds__(kThreads) pack16_kernel(const uint16_t* __restrict__ src,
                                                          int64_t ld, int64_t stride, int64_t rows,
                                                          int64_t cols, uint16_t* __restrict__ dst,
                                                          int64_t ld_dst) {
    const int64_t b = blockIdx.z;
    const int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (c >= cols) return;
    const uint16_t* s = src + b * stride + c;
    uint16_t* d = dst + b * rows * ld_dst + c;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) d[r * ld_dst] = s[r * ld];
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
    const int64_t gx = (cols + kThreads - 1) / kThreads;
    const int64_t gy = rows < 4096 ? rows : 4096;
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
    splitk_epi_kernel<<<grid_for(total), kThreads, 0, stream>>>(partials, splits, batch, M, N, e);
    return cudaGetLastError();
}

}  // namespace dg
