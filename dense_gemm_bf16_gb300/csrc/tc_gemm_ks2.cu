// Instantiations of the tensor-core GEMM kernel that bring two 64-deep K
// blocks of each K-major operand per TMA load (KS = 2): CTA pairs with
// 128- and 256-column tiles and the TMA-store-only epilogue.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_ks2(int bn, int mode, int epi) { return mode == 2 && epi == 1 && (bn == 128 || bn == 256); }

int tc_stages_ks2(int bn) {
    if (bn == 128) return Cfg<128, 2, 1, 2>::STAGES;
    if (bn == 256) return Cfg<256, 2, 1, 2>::STAGES;
    return 0;
}

cudaError_t tc_prepare_ks2(int bn) {
    if (bn == 128) return prepare_bn<128, 2, 1, 2>();
    if (bn == 256) return prepare_bn<256, 2, 1, 2>();
    return cudaSuccess;  // no instantiation for other tile widths
}

cudaError_t tc_launch_ks2(int bn, const TcParams& p, int grid, cudaStream_t stream) {
    if (bn == 128) return launch_bn<128, 2, 1, 2>(p, grid, stream);
    if (bn == 256) return launch_bn<256, 2, 1, 2>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace dg
