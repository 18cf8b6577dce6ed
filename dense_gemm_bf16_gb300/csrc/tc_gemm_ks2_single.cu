// Instantiations of the tensor-core GEMM kernel with one CTA per tile that
// bring two 64-deep K blocks of each operand per TMA load (KS = 2): narrow
// tiles (16-64 columns) with the general epilogue, which skinny products use
// (M <= 64 computed as C^T, whose output is then column-major), and 64-256
// columns with the TMA-store-only epilogue.  Larger loads keep more bytes in
// flight per SM where one SM must stream a long operand panel by itself.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_ks2_single(int bn, int epi) {
    if (epi == 0) return bn == 16 || bn == 32 || bn == 64;
    if (epi == 1) return bn == 64 || bn == 128 || bn == 256;
    return false;
}

int tc_stages_ks2_single(int bn, int epi) {
    if (epi == 0) {
        if (bn == 16) return Cfg<16, 0, 0, 2>::STAGES;
        if (bn == 32) return Cfg<32, 0, 0, 2>::STAGES;
        if (bn == 64) return Cfg<64, 0, 0, 2>::STAGES;
    } else if (epi == 1) {
        if (bn == 64) return Cfg<64, 0, 1, 2>::STAGES;
        if (bn == 128) return Cfg<128, 0, 1, 2>::STAGES;
        if (bn == 256) return Cfg<256, 0, 1, 2>::STAGES;
    }
    return 0;
}

cudaError_t tc_prepare_ks2_single(int bn) {
    switch (bn) {
        case 16: return prepare_bn<16, 0, 0, 2>();
        case 32: return prepare_bn<32, 0, 0, 2>();
        case 64: {
            cudaError_t e = prepare_bn<64, 0, 0, 2>();
            if (e == cudaSuccess) e = prepare_bn<64, 0, 1, 2>();
            return e;
        }
        case 128: return prepare_bn<128, 0, 1, 2>();
        case 256: return prepare_bn<256, 0, 1, 2>();
    }
    return cudaSuccess;  // no instantiation for other tile widths
}

cudaError_t tc_launch_ks2_single(int bn, int epi, const TcParams& p, int grid,
                                 cudaStream_t stream) {
    if (epi == 0) {
        if (bn == 16) return launch_bn<16, 0, 0, 2>(p, grid, stream);
        if (bn == 32) return launch_bn<32, 0, 0, 2>(p, grid, stream);
        if (bn == 64) return launch_bn<64, 0, 0, 2>(p, grid, stream);
    } else if (epi == 1) {
        if (bn == 64) return launch_bn<64, 0, 1, 2>(p, grid, stream);
        if (bn == 128) return launch_bn<128, 0, 1, 2>(p, grid, stream);
        if (bn == 256) return launch_bn<256, 0, 1, 2>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dg
