// Instantiations of the tensor-core GEMM kernel with the general epilogue.
#include "tc_kernel.cuh"

namespace dg {

cudaError_t tc_prepare_general(int bn) {
    switch (bn) {
        case 16: return prepare_bn<16, 0, 0>();
        case 32: return prepare_bn<32, 0, 0>();
        case 64: return prepare_bn<64, 0, 0>();
        case 128: {
            cudaError_t e = prepare_bn<128, 0, 0>();
            if (e == cudaSuccess) e = prepare_bn<128, 2, 0>();
            return e;
        }
        case 256: {
            cudaError_t e = prepare_bn<256, 0, 0>();
            if (e == cudaSuccess) e = prepare_bn<256, 2, 0>();
            return e;
        }
        case 512: return prepare_bn<512, 2, 0>();
    }
    return cudaErrorInvalidValue;
}

int tc_max_pairs_general(int bn, int mode) {
    if (mode == 2 && bn == 128) return max_clusters_bn<128, 2, 0>();
    if (mode == 2 && bn == 256) return max_clusters_bn<256, 2, 0>();
    if (mode == 2 && bn == 512) return max_clusters_bn<512, 2, 0>();
    return 0;
}

cudaError_t tc_launch_general(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream) {
    if (mode == 2) {
        if (bn == 128) return launch_bn<128, 2, 0>(p, grid, stream);
        if (bn == 256) return launch_bn<256, 2, 0>(p, grid, stream);
        if (bn == 512) return launch_bn<512, 2, 0>(p, grid, stream);
        return cudaErrorInvalidValue;
    }
    switch (bn) {
        case 16: return launch_bn<16, 0, 0>(p, grid, stream);
        case 32: return launch_bn<32, 0, 0>(p, grid, stream);
        case 64: return launch_bn<64, 0, 0>(p, grid, stream);
        case 128: return launch_bn<128, 0, 0>(p, grid, stream);
        case 256: return launch_bn<256, 0, 0>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dg
