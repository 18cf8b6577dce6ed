// Instantiations of the tensor-core GEMM kernel with the TMA-store epilogue
// that reads beta * C by TMA loads (epilogue form 2): a 16-bit C that takes
// TMA stores, beta != 0.  Single-CTA tiles of 64-256 columns and pair tiles of
// 128 and 256 columns.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_beta_form(int bn, int mode) {
    if (mode == 0) return bn == 64 || bn == 128 || bn == 256;
    if (mode == 2) return bn == 128 || bn == 256;
    return false;
}

int tc_stages_beta(int bn, int mode) {
    if (mode == 2) {
        if (bn == 128) return Cfg<128, 2, 2>::STAGES;
        if (bn == 256) return Cfg<256, 2, 2>::STAGES;
        return 0;
    }
    switch (bn) {
        case 64: return Cfg<64, 0, 2>::STAGES;
        case 128: return Cfg<128, 0, 2>::STAGES;
        case 256: return Cfg<256, 0, 2>::STAGES;
    }
    return 0;
}

cudaError_t tc_prepare_beta(int bn) {
    switch (bn) {
        case 64: return prepare_bn<64, 0, 2>();
        case 128: {
            cudaError_t e = prepare_bn<128, 0, 2>();
            if (e == cudaSuccess) e = prepare_bn<128, 2, 2>();
            return e;
        }
        case 256: {
            cudaError_t e = prepare_bn<256, 0, 2>();
            if (e == cudaSuccess) e = prepare_bn<256, 2, 2>();
            return e;
        }
    }
    return cudaSuccess;  // no instantiation of this form for other tile widths
}

cudaError_t tc_launch_beta(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream) {
    if (mode == 2) {
        if (bn == 128) return launch_bn<128, 2, 2>(p, grid, stream);
        if (bn == 256) return launch_bn<256, 2, 2>(p, grid, stream);
        return cudaErrorInvalidValue;
    }
    if (mode == 0) {
        switch (bn) {
            case 64: return launch_bn<64, 0, 2>(p, grid, stream);
            case 128: return launch_bn<128, 0, 2>(p, grid, stream);
            case 256: return launch_bn<256, 0, 2>(p, grid, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace dg
