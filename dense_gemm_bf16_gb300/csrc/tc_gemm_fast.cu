// Instantiations of the tensor-core GEMM kernel with the TMA-store-only
// epilogue (beta == 0 or split-K partials), for tile widths of 64 and up.
#include "tc_kernel.cuh"

namespace dg {

cudaError_t tc_prepare_fast(int bn) {
    switch (bn) {
        case 64: return prepare_bn<64, 0, 1>();
        case 128: {
            cudaError_t e = prepare_bn<128, 0, 1>();
            if (e == cudaSuccess) e = prepare_bn<128, 2, 1>();
            return e;
        }
        case 256: {
            cudaError_t e = prepare_bn<256, 0, 1>();
            if (e == cudaSuccess) e = prepare_bn<256, 2, 1>();
            return e;
        }
        case 512: return prepare_bn<512, 2, 1>();
    }
    return cudaSuccess;  // no fast instantiation for narrower tiles
}

cudaError_t tc_launch_fast(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream) {
    if (mode == 2) {
        if (bn == 128) return launch_bn<128, 2, 1>(p, grid, stream);
        if (bn == 256) return launch_bn<256, 2, 1>(p, grid, stream);
        if (bn == 512) return launch_bn<512, 2, 1>(p, grid, stream);
        return cudaErrorInvalidValue;
    }
    switch (bn) {
        case 64: return launch_bn<64, 0, 1>(p, grid, stream);
        case 128: return launch_bn<128, 0, 1>(p, grid, stream);
        case 256: return launch_bn<256, 0, 1>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dg
