// gemm_bf16_static_workspace: the bf16 GEMM with its scratch in a fixed
// device array that the library owns, for callers that cannot allocate.
//
// The scratch (split-K partial tiles, aligned copies of operands that TMA
// cannot address) normally lives in a caller-provided workspace.  Here it is
// the file-scope array below, GEMM_STATIC_WORKSPACE_BYTES long, which every
// device that loads this library holds until the process exits.  The host
// code never dereferences or passes the array's host-side name: once per
// device, with that device current, it asks the runtime for the array's
// device address and hands that address to the regular gemm_bf16 entry point
// as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "gemm.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[GEMM_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_device_addr[kMaxDevices];
cudaError_t g_setup_err[kMaxDevices];

}  // namespace

extern "C" gemm_status_t gemm_bf16_static_workspace(
    int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, gemm_layout_t la, const void* B,
    int64_t ldb, gemm_layout_t lb, void* C, int64_t ldc, gemm_layout_t lc, gemm_dtype_t c_dtype,
    float alpha, float beta, const float* bias, gemm_epilogue_t epi, int split_k,
    gemm_stream_t stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    // Set-up on this device's first call (the current device is `dev`).
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_setup_err[dev] = cudaGetSymbolAddress(&p, g_static_workspace);
        g_device_addr[dev] = p;
        if (g_setup_err[dev] != cudaSuccess) cudaGetLastError();
    });
    if (g_setup_err[dev] != cudaSuccess || g_device_addr[dev] == nullptr) return GEMM_ERR_CUDA;
    return gemm_bf16(M, N, K, A, lda, la, B, ldb, lb, C, ldc, lc, c_dtype, alpha, beta, bias, epi,
                     split_k, g_device_addr[dev], GEMM_STATIC_WORKSPACE_BYTES, stream);
}
