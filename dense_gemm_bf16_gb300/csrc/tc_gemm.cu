// Host dispatch of the tensor-core GEMM kernel over tile width, CTA mode and
// epilogue form; the instantiations live in tc_gemm_general.cu,
// tc_gemm_epi8.cu, tc_gemm_fast.cu, tc_gemm_beta.cu and tc_gemm_ks2*.cu.
#include "tc_kernel.cuh"

namespace dg {

cudaError_t tc_prepare_general(int bn);
cudaError_t tc_prepare_fast(int bn);
int tc_max_pairs_general(int bn, int mode);
cudaError_t tc_launch_general(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t tc_launch_fast(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t tc_prepare_beta(int bn);
cudaError_t tc_prepare_ks2(int bn);
cudaError_t tc_launch_ks2(int bn, int mode, int epi, const TcParams& p, int grid,
                          cudaStream_t stream);
cudaError_t tc_launch_beta(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t tc_prepare_epi8(int bn);
cudaError_t tc_launch_epi8(int bn, int mode, int epi, const TcParams& p, int grid,
                           cudaStream_t stream);

int tc_stages_for(int bn, int mode) {
    if (mode == 2) {
        if (bn == 128) return Cfg<128, 2>::STAGES;
        if (bn == 256) return Cfg<256, 2>::STAGES;
        if (bn == 512) return Cfg<512, 2>::STAGES;
        return 0;
    }
    switch (bn) {
        case 16: return Cfg<16, 0>::STAGES;
        case 32: return Cfg<32, 0>::STAGES;
        case 64: return Cfg<64, 0>::STAGES;
        case 128: return Cfg<128, 0>::STAGES;
        case 256: return Cfg<256, 0>::STAGES;
    }
    return 0;
}

cudaError_t tc_prepare(int bn) {
    cudaError_t e = tc_prepare_general(bn);
    if (e == cudaSuccess) e = tc_prepare_fast(bn);
    if (e == cudaSuccess) e = tc_prepare_beta(bn);
    if (e == cudaSuccess) e = tc_prepare_ks2(bn);
    if (e == cudaSuccess) e = tc_prepare_epi8(bn);
    return e;
}

bool tc_has_mode(int bn, int mode) {
    if (mode == 0) return bn == 16 || bn == 32 || bn == 64 || bn == 128 || bn == 256;
    if (mode == 2) return bn == 128 || bn == 256 || bn == 512;
    return false;
}

int tc_max_pairs(int bn, int mode) { return tc_max_pairs_general(bn, mode); }

bool tc_has_fast(int bn) { return bn == 64 || bn == 128 || bn == 256 || bn == 512; }

cudaError_t tc_launch(int bn, int mode, int epi, int ks, const TcParams& p, int grid,
                      cudaStream_t stream) {
    if (ks == 2) {
        if (!tc_has_ks2(bn, mode, epi)) return cudaErrorInvalidValue;
        return tc_launch_ks2(bn, mode, epi, p, grid, stream);
    }
    if (epi == 1 && tc_has_fast(bn)) return tc_launch_fast(bn, mode, p, grid, stream);
    if (epi == 2 && tc_has_beta_form(bn, mode)) return tc_launch_beta(bn, mode, p, grid, stream);
    if (epi == 3 || epi == 4) return tc_launch_epi8(bn, mode, epi, p, grid, stream);
    return tc_launch_general(bn, mode, p, grid, stream);
}

}  // namespace dg
