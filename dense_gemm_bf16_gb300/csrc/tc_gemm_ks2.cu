// Instantiations of the tensor-core GEMM kernel that bring two 64-deep K
// blocks of each operand per TMA load (KS = 2): CTA pairs with 128- and
// 256-column tiles and the TMA-store-only epilogue (the single-CTA forms are
// in tc_gemm_ks2_single.cu), and the dispatch over both.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_ks2_single(int bn, int epi);
int tc_stages_ks2_single(int bn, int epi);
cudaError_t tc_prepare_ks2_single(int bn);
cudaError_t tc_launch_ks2_single(int bn, int epi, const TcParams& p, int grid, cudaStream_t stream);

bool tc_has_ks2(int bn, int mode, int epi) {
    if (mode == 2) return epi == 1 && (bn == 128 || bn == 256);
    if (mode == 0) return tc_has_ks2_single(bn, epi);
    return false;
}

int tc_stages_ks2(int bn, int mode, int epi) {
    if (mode == 0) return tc_stages_ks2_single(bn, epi);
    if (mode == 2 && epi == 1) {
        if (bn == 128) return Cfg<128, 2, 1, 2>::STAGES;
        if (bn == 256) return Cfg<256, 2, 1, 2>::STAGES;
    }
    return 0;
}

cudaError_t tc_prepare_ks2(int bn) {
    cudaError_t e = tc_prepare_ks2_single(bn);
    if (e != cudaSuccess) return e;
    if (bn == 128) return prepare_bn<128, 2, 1, 2>();
    if (bn == 256) return prepare_bn<256, 2, 1, 2>();
    return cudaSuccess;  // no pair instantiation for other tile widths
}

cudaError_t tc_launch_ks2(int bn, int mode, int epi, const TcParams& p, int grid,
                          cudaStream_t stream) {
    if (mode == 0) return tc_launch_ks2_single(bn, epi, p, grid, stream);
    if (mode == 2 && epi == 1) {
        if (bn == 128) return launch_bn<128, 2, 1, 2>(p, grid, stream);
        if (bn == 256) return launch_bn<256, 2, 1, 2>(p, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dg
