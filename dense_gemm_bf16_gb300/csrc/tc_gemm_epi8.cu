// Instantiations of the tensor-core GEMM kernel whose epilogue runs on eight
// warps, two per tensor-memory lane quarter, each writing half of the tile's
// columns: form 3 (the general, plain-store epilogue, for an output the TMA
// unit cannot store, such as fp32 rows that are not 16-byte aligned) and
// form 4 (the TMA-store epilogue that reads beta * C by TMA loads, one output
// box per warp), for CTA pairs with 256-column tiles and whole tiles only.
// A unit of its own so that it compiles in parallel with the other forms.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_epi8(int bn, int mode, int epi) {
    return bn == 256 && mode == 2 && (epi == 3 || epi == 4);
}

int tc_stages_epi8(int bn, int mode, int epi) {
    if (!tc_has_epi8(bn, mode, epi)) return 0;
    return epi == 3 ? Cfg<256, 2, 3>::STAGES : Cfg<256, 2, 4>::STAGES;
}

cudaError_t tc_prepare_epi8(int bn) {
    if (bn != 256) return cudaSuccess;
    cudaError_t e = prepare_bn<256, 2, 3>();
    if (e == cudaSuccess) e = prepare_bn<256, 2, 4>();
    return e;
}

cudaError_t tc_launch_epi8(int bn, int mode, int epi, const TcParams& p, int grid,
                           cudaStream_t stream) {
    if (!tc_has_epi8(bn, mode, epi)) return cudaErrorInvalidValue;
    if (epi == 3) return launch_bn<256, 2, 3>(p, grid, stream);
    return launch_bn<256, 2, 4>(p, grid, stream);
}

}  // namespace dg
