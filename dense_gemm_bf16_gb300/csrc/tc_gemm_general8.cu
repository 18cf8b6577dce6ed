// Instantiation of the tensor-core GEMM kernel in epilogue form 3: the
// general (plain-store) epilogue on eight warps, two per tensor-memory lane
// quarter, each writing half of the tile's columns, for CTA pairs with
// 256-column tiles and whole tiles only (an output TMA cannot store, such as
// fp32 rows that are not 16-byte aligned).  A unit of its own so that it
// compiles in parallel with the other forms.
#include "tc_kernel.cuh"

namespace dg {

bool tc_has_general8(int bn, int mode) { return bn == 256 && mode == 2; }

int tc_stages_general8(int bn, int mode) {
    return tc_has_general8(bn, mode) ? Cfg<256, 2, 3>::STAGES : 0;
}

cudaError_t tc_prepare_general8(int bn) {
    if (bn == 256) return prepare_bn<256, 2, 3>();
    return cudaSuccess;
}

cudaError_t tc_launch_general8(int bn, int mode, const TcParams& p, int grid, cudaStream_t stream) {
    if (tc_has_general8(bn, mode)) return launch_bn<256, 2, 3>(p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace dg
