// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "debug_check.cuh"

namespace dg {

enum : int { DT_BF16 = 0, DT_F16 = 1, DT_F32 = 2 };
enum : int { ACT_NONE = 0, ACT_GELU_TANH = 1, ACT_RELU = 2, ACT_GELU_ERF = 3 };

// Tile of the tensor-core kernel: BLOCK_M x BLOCK_N output, K consumed in
// BLOCK_K = 64 slices (64 bf16 = one 128-byte swizzle row).
constexpr int TC_BLOCK_M = 128;
constexpr int TC_BLOCK_K = 64;
// threads of the tensor-core kernel's four-warp epilogue forms (0-2): warp 0
// TMA producer, warp 1 MMA issuer, warps 2-5 epilogue (forms 3 and 4 have
// eight epilogue warps, 320 threads: Cfg::THREADS)
constexpr int TC_THREADS = 192;
constexpr int TC_EPI_THREADS = 128;

// Epilogue description shared by the tensor-core kernel and the split-K reduce.
struct Epilogue {
    void* C;                 // output (and beta input), c_dtype
    int64_t ldc;             // leading dimension of C in elements
    int64_t stride_c;        // batch stride of C in elements
    int32_t c_row_major;     // 1: C(i,j) at i*ldc + j; 0: at j*ldc + i
    int32_t c_dtype;         // DT_BF16 / DT_F16 / DT_F32
    int32_t c_vec_ok;        // C base and ldc allow 16-byte vector access along rows
    float alpha, beta;
    const float* bias;       // may be null
    int32_t bias_on_rows;    // 1: bias indexed by row i (swapped problem), 0: by column j
    int32_t act;             // ACT_NONE / ACT_GELU_TANH / ACT_RELU / ACT_GELU_ERF
#if DG_DEBUG
    // debug build only: the bounds the device-side checks hold accesses to
    int* dbg_status;         // device status word
    int64_t dbg_c_elems;     // C element offsets [0, dbg_c_elems) from C may be touched
    int64_t dbg_bias_len;    // entries of bias
    uint32_t* dbg_counts;    // count-writes mode: [batch][M][N] of the caller's C, or null
    int64_t dbg_m, dbg_n;    // the caller's M and N
    int32_t dbg_swap;        // 1: the computed problem is the caller's transposed
#endif
};

// Parameters of the persistent tcgen05 kernel (passed as a __grid_constant__).
struct TcParams {
    CUtensorMap tmap_a;      // A-role operand (rows = M of the computed problem)
    CUtensorMap tmap_b;      // B-role operand (rows = N of the computed problem)
    int32_t M, N, K, batch;
    int32_t num_pid_m, num_pid_n;
    int32_t tiles_per_batch;
    int32_t splits;          // K slices per tile
    int32_t kblocks;         // ceil(K / 64)
    int32_t group_m;
    int32_t total_units;     // batch * splits * tiles_per_batch
    int32_t a_mn, b_mn;      // 1: operand stored MN-contiguous (MN-major), 0: K-contiguous
    int32_t a_3d, b_3d;      // 1: tensor map carries the batch as its third dimension
    uint32_t idesc;          // tcgen05 instruction descriptor
    Epilogue epi;
    CUtensorMap tmap_c;      // output (or split-K partials) for the TMA-store epilogue
    int32_t c_tma;           // 1: epilogue stores through tmap_c
    int32_t c_tma_3d;        // 1: tmap_c has a third (batch or slice) dimension
    float* partials;         // split-K: fp32 partial tiles [split][batch][M][N] in C's layout; else null
    int* status;             // device error word
    uint64_t timeout_ns;     // bound on every wait
    int32_t test_stall;      // test only: 1 leave one stage unfilled; 2 CTA 0 publishes no partial flags
    int32_t l2_hints;        // operand L2 policy: 0 normal; 1 A evict-first, B evict-last; 2 the reverse
    // 1: launched as the programmatic dependent of the operand copy just before
    // it on the stream (never with the cooperative forms): the CTAs set up while
    // the copy runs, and the producer waits for the copy's completion
    // (griddepcontrol.wait) before its first load
    int32_t pdl;
    // Stream-K.  Every cluster first takes dp_per_cluster whole units round
    // robin; the units from dp_units on are then cut along K, in one of two forms.
    // Contiguous (sk_iters > 0): their steps (of KS K blocks) are split evenly
    // over the clusters, each taking one contiguous range; a unit cut at
    // cluster boundaries is finished by the cluster that holds its first step,
    // after each later cluster holding part of it has left its fp32 partial in
    // that cluster's own slot.
    // Split (sk_split > 0): each of the sk_tiles last units is cut into sk_split
    // equal K pieces, one per cluster, so that all pieces start together; piece 0
    // finishes the tile after the other sk_split - 1 have left their partials.
    // With sk_spread every piece leaves its partial, and once all have, piece j
    // sums the j-th of sk_split equal shares of the tile over all partials and
    // writes that share of the output (the launch is cooperative: every piece
    // waits for every other one).
    int32_t dp_per_cluster;
    int32_t dp_units;
    int64_t sk_iters;        // steps (of KS K blocks) of the contiguous form (0: off)
    int32_t sk_split;        // pieces per unit of the split form (0: off)
    int32_t sk_tiles;        // units cut in the split form
    int32_t sk_spread;       // split form: 1 every piece reduces a share of the tile
    // 1: no fix-up at all: every K piece adds alpha * its accumulator into C
    // (fp32, row-major) by TMA reduce-add, after the CTAs have set C to
    // beta * C + bias, each for its share of rows, and published that share's
    // flag (sk_flags[cta]) with the epoch
    int32_t sk_atomic;
    float* sk_partials;      // [slot][cta rank][128][BN] fp32, lane-interleaved per warp
    unsigned long long* sk_flags;  // [slot][cta rank][epilogue warp]: epoch when published
    unsigned long long sk_epoch;   // this launch's flag value
#if DG_DEBUG
    // debug build only: the bounds of the workspace areas and of the tile grid
    int64_t dbg_sk_slots;        // stream-K partial slots the workspace holds (x CTAs per cluster)
    int64_t dbg_partials_elems;  // fp32 elements of the split-K partials
    int32_t dbg_num_pid_n;       // tile columns a work unit may name
#endif
};

// Host-side launchers (defined in tc_gemm.cu / sgemm.cu / aux_kernels.cu).
// Tensor-core kernel modes: 0 one CTA per 128 x BN tile; 2 CTA pair computing
// a 256 x BN tile with cta_group::2 MMAs (each CTA loads its own half of A and
// B; no operand load is multicast).  Epilogue forms: 0 general; 1 TMA store only, for
// beta == 0 or split-K partials, with tmap_c boxes of 128-byte rows
// (tc_has_fast tells the tile widths that have it); 2 the same with beta * C
// read by TMA loads through tmap_c, for a 16-bit C (tc_has_beta_form tells the
// tile widths and modes, tc_stages_beta its pipeline depth); 3 and 4 forms 0
// and 2 on eight epilogue warps, two per tensor-memory lane quarter, each
// writing half of the tile's columns, for whole tiles only (tc_has_epi8 /
// tc_stages_epi8).  ks: 64-deep K
// blocks per stage and per TMA load of each operand, 1 or 2 (tc_has_ks2
// tells where 2 exists; a K-major operand's map is then the three-dimensional
// view 64 K x rows x K blocks, an MN-major one's takes boxes of 128 K rows).
int tc_stages_for(int block_n, int mode);
bool tc_has_mode(int block_n, int mode);
bool tc_has_fast(int block_n);
bool tc_has_beta_form(int block_n, int mode);
int tc_stages_beta(int block_n, int mode);
cudaError_t tc_prepare(int block_n);   // sets the dynamic shared memory attribute (per device)
cudaError_t tc_launch(int block_n, int mode, int epi, int ks, const TcParams& p, int grid,
                      cudaStream_t stream);
bool tc_has_ks2(int block_n, int mode, int epi);
int tc_stages_ks2(int block_n, int mode, int epi);
int tc_max_pairs(int block_n, int mode);  // two-CTA clusters resident at once on this device
bool tc_has_epi8(int block_n, int mode, int epi);
int tc_stages_epi8(int block_n, int mode, int epi);

struct SgemmParams {
    const float* A; int64_t lda; int64_t stride_a; int32_t a_row;
    const float* B; int64_t ldb; int64_t stride_b; int32_t b_row;
    int32_t M, N, K, batch;
    int32_t a_vec_ok, b_vec_ok;   // float4 global loads allowed
    int32_t kernel;               // 0 cp.async packed-FMA kernel (row-major A and B); 1 register-staged
    int32_t num_pid_m, num_pid_n, group_m;
    Epilogue epi;
};
cudaError_t sgemm_launch(const SgemmParams& p, cudaStream_t stream);
cudaError_t sgemm_prepare();  // dynamic shared memory attributes (per device)

// Dense copy of a rows x cols 16-bit matrix stored with (ld, batch stride) into
// dst with leading dimension ld_dst and batch stride rows*ld_dst.
cudaError_t pack16_launch(const void* src, int64_t ld, int64_t stride, int64_t rows,
                          int64_t cols, int64_t batch, void* dst, int64_t ld_dst,
                          cudaStream_t stream);

// C = act(alpha * sum_s P[s] + beta*C + bias) for splits >= 0 partial slices
// stored densely in C's layout ([split][batch][M][N] row-major or its transpose).
cudaError_t splitk_epilogue_launch(const float* partials, int splits, int64_t batch,
                                   int64_t M, int64_t N, const Epilogue& e,
                                   cudaStream_t stream);

}  // namespace dg
