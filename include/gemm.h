/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library (libdgemm_gb300.so).
 *
 * Operation (BLAS level-3 GEMM, "2 . La GEMM, de zero a cuBLAS", section 2.1,
 * with the fused epilogue of "Skill: Write a Triton GEMM Kernel", Required
 * reasoning process step 6):
 *
 *     C[b] <- act( alpha * A[b] @ B[b] + beta * C[b] + bias )      b = 0..batch-1
 *
 *   A[b] is M x K, B[b] is K x N, C[b] is M x N.  Products accumulate in fp32
 *   ("GEMM Kernel Optimization", Core Technique and Tensor Core Utilization);
 *   the downcast to the output type happens once, after accumulation
 *   ("GEMM Kernel Optimization", Common Pitfalls).  bias is an fp32 vector,
 *   along columns (length N) or rows (length M), added before the activation
 *   and not scaled by alpha.  act is the identity, GELU (tanh or erf form) or
 *   ReLU; see gemm_epilogue_t.
 *
 * Storage.  Every matrix is given by a pointer, a leading dimension and a
 * layout flag: element (r, c) of a GEMM_ROW_MAJOR matrix sits at r*ld + c, of
 * a GEMM_COL_MAJOR one at c*ld + r (elements, not bytes).  The inner stride is
 * always 1; ld must be at least the inner extent ("Skill: Write a Triton GEMM
 * Kernel", Kernel design rules: strides are arguments, never recomputed from
 * shapes).  Batch b of an operand starts at ptr + b*stride; a stride of 0
 * broadcasts one matrix to the whole batch (same page, Correctness
 * requirements, batched GEMM).  C is read (when beta != 0) and written in
 * place, in its own dtype.
 *
 * Conventions shared by every entry point:
 *   - All pointers except the workspace and the return codes are DEVICE
 *     pointers on the current CUDA device; the caller owns every buffer.  The
 *     library allocates no device memory in any call and keeps no pointer
 *     after return.  Work is enqueued on `stream` (NULL = legacy default
 *     stream) and runs asynchronously: results are ready when the stream is.
 *   - beta == 0 means C is not read (NaN or Inf in C does not propagate).
 *     alpha == 0 or K == 0 means A and B are not read:
 *     C <- act(beta*C + bias).  M == 0, N == 0 or batch == 0 is a no-op.
 *   - Argument errors are detected before anything is enqueued and are
 *     reported by the return code; nothing aborts, prints or throws.  Among
 *     them: an extent above 2^31 - 1, a matrix whose elements (with its
 *     leading dimension or strides, over the batch) would span more than
 *     2^48 elements of memory, and a matrix of more than 2^56 elements over
 *     the batch.
 *   - Any pointer alignment that the element type allows is accepted.  Fast
 *     TMA paths need 16-byte aligned bases and leading dimensions that are a
 *     multiple of 16 bytes; other operands are first copied into the
 *     caller's workspace (see gemm_workspace_size).
 *   - Calls are thread-safe.  The first call on a device queries device
 *     attributes and may set kernel attributes (no allocation).
 *   - A call may be captured into a CUDA graph once the device has seen one
 *     uncaptured call (which does the one-time setup above).  The plan,
 *     pointers and scalars are fixed at capture.  Plans that hand fp32
 *     partials between the pieces of a tile (stream-K, the one-kernel
 *     split-K) synchronise through flags in the workspace.  Those flags hold
 *     a per-launch value that a replay repeats, so a captured call also
 *     records a clearing of the flags ahead of its kernel.  Replays of one
 *     graph, like calls that share one workspace, must not overlap.
 */
#ifndef DGEMM_GB300_GEMM_H
#define DGEMM_GB300_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t / CUstream); NULL is the legacy stream. */
typedef void* gemm_stream_t;

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;

typedef enum { GEMM_DT_BF16 = 0, GEMM_DT_F16 = 1, GEMM_DT_F32 = 2 } gemm_dtype_t;

/*
 * Epilogue: C = act(alpha*A@B + beta*C + bias), applied once after the K loop
 * ("Skill: Write a Triton GEMM Kernel", Required reasoning process step 6;
 * Inputs the agent should gather first, item 5).  The value is a bit field:
 *   bit 0     add the bias vector (fp32, device memory);
 *   bits 1-2  activation: 0 none, 1 GELU tanh form
 *             0.5x(1 + tanh(sqrt(2/pi)(x + 0.044715x^3))), 2 ReLU (x > 0 ? x : 0,
 *             NaN gives 0), 3 GELU erf form 0.5x(1 + erf(x/sqrt(2)));
 *   bit 3     the bias runs along rows: bias[m], length M (requires bit 0);
 *             without it bias[n], length N.
 * The bias is added before the activation and is not scaled by alpha.
 */
typedef enum {
    GEMM_EPI_NONE = 0,                /* C = alpha*A@B + beta*C              */
    GEMM_EPI_BIAS = 1,                /* ... + bias[n]                       */
    GEMM_EPI_GELU_TANH = 2,           /* gelu_tanh(alpha*A@B + beta*C)       */
    GEMM_EPI_BIAS_GELU_TANH = 3,      /* gelu_tanh(... + bias[n])            */
    GEMM_EPI_RELU = 4,                /* relu(alpha*A@B + beta*C)            */
    GEMM_EPI_BIAS_RELU = 5,           /* relu(... + bias[n])                 */
    GEMM_EPI_GELU_ERF = 6,            /* gelu_erf(alpha*A@B + beta*C)        */
    GEMM_EPI_BIAS_GELU_ERF = 7,       /* gelu_erf(... + bias[n])             */
    GEMM_EPI_ROW_BIAS = 9,            /* ... + bias[m]                       */
    GEMM_EPI_ROW_BIAS_GELU_TANH = 11, /* gelu_tanh(... + bias[m])            */
    GEMM_EPI_ROW_BIAS_RELU = 13,      /* relu(... + bias[m])                 */
    GEMM_EPI_ROW_BIAS_GELU_ERF = 15   /* gelu_erf(... + bias[m])             */
} gemm_epilogue_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,  /* negative size, ld too small, bad enum, NULL pointer, misaligned element */
    GEMM_ERR_UNSUPPORTED = 2,  /* well-formed request this library does not implement (e.g. dtype mix)  */
    GEMM_ERR_WORKSPACE = 3,    /* workspace smaller than the plan needs                                   */
    GEMM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed (launch, attribute, tensor map)      */
    GEMM_ERR_TIMEOUT = 5,      /* a kernel gave up a bounded wait (reported by gemm_check_device_status) */
    GEMM_ERR_NO_DEVICE = 6,    /* no usable sm_103 device is current                                      */
    GEMM_ERR_DEVICE_CHECK = 7  /* debug build only: a device-side check failed and its access was skipped
                                  (reported by gemm_check_device_status)                                  */
} gemm_status_t;

/*
 * gemm_bf16 -- bf16 A and B, fp32 accumulation on the tcgen05 tensor cores.
 *
 *   M, N, K      problem size (>= 0, each below 2^31).
 *   A, lda, la   M x K operand, bf16.           B, ldb, lb  K x N operand, bf16.
 *   C, ldc, lc   M x N result, c_dtype GEMM_DT_BF16 or GEMM_DT_F32; read when beta != 0.
 *   alpha, beta  fp32 scalars.
 *   bias         fp32 device vector of length N (length M for a row bias), 4-byte
 *                aligned; required iff epi uses a bias, else ignored.
 *   epi          epilogue (gemm_epilogue_t).
 *   split_k      0 = choose automatically (split-K or stream-K pieces when they
 *                pay), 1 = no split (every tile summed over the whole K in one
 *                accumulator, no stream-K pieces either), s > 1 = split K into s
 *                slices whose fp32 partial tiles are summed in a fixed order by a
 *                second kernel ("Skill: Write a Triton GEMM Kernel", Kernel
 *                design rules, split-K; "2 . La GEMM, de zero a cuBLAS", section 2.10).
 *                s is clamped to the number of 64-wide K blocks.
 *   workspace    device scratch of workspace_bytes bytes, 256-byte aligned (may be
 *                NULL/0).  Needed
 *                for split-K partials and for copies of operands that TMA cannot
 *                address; gemm_workspace_size() gives a sufficient size.  With
 *                split_k == 0 the plan never asks for more than is given
 *                (it drops to fewer splits); split_k > 1 or an operand that needs
 *                a copy with too small a workspace returns GEMM_ERR_WORKSPACE.
 *   stream       CUDA stream.
 */
gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, gemm_layout_t la,
                        const void* B, int64_t ldb, gemm_layout_t lb,
                        void* C, int64_t ldc, gemm_layout_t lc, gemm_dtype_t c_dtype,
                        float alpha, float beta, const float* bias, gemm_epilogue_t epi,
                        int split_k, void* workspace, size_t workspace_bytes,
                        gemm_stream_t stream);

/* gemm_f16 -- as gemm_bf16 with fp16 A and B; c_dtype GEMM_DT_F16 or GEMM_DT_F32. */
gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, gemm_layout_t la,
                       const void* B, int64_t ldb, gemm_layout_t lb,
                       void* C, int64_t ldc, gemm_layout_t lc, gemm_dtype_t c_dtype,
                       float alpha, float beta, const float* bias, gemm_epilogue_t epi,
                       int split_k, void* workspace, size_t workspace_bytes,
                       gemm_stream_t stream);

/*
 * sgemm_f32 -- true fp32 GEMM on the CUDA cores (FFMA; no tensor cores, no TF32).
 * Register-tiled outer-product kernel ("2 . La GEMM, de zero a cuBLAS",
 * sections 2.6-2.8: 128x128x8 block tile, 8x8 accumulators per thread, float4
 * loads, transposed A tile in shared memory, double buffering).
 * Arguments as gemm_bf16, all matrices fp32; no workspace is used.
 */
gemm_status_t sgemm_f32(int64_t M, int64_t N, int64_t K,
                        const float* A, int64_t lda, gemm_layout_t la,
                        const float* B, int64_t ldb, gemm_layout_t lb,
                        float* C, int64_t ldc, gemm_layout_t lc,
                        float alpha, float beta, const float* bias, gemm_epilogue_t epi,
                        gemm_stream_t stream);

/*
 * gemm_batched -- strided batched GEMM ("Skill: Write a Triton GEMM Kernel",
 * Inputs step 6 and Correctness requirements).
 *
 *   ab_dtype     GEMM_DT_BF16 / GEMM_DT_F16 (tensor cores) or GEMM_DT_F32 (CUDA cores).
 *   batch        number of products (>= 0).
 *   stride_a/b   elements between consecutive A[b] / B[b]; 0 = broadcast.
 *   stride_c     elements between consecutive C[b]; must be > 0 when batch > 1
 *                and large enough that the C[b] do not overlap.
 *   Other arguments as gemm_bf16 (c_dtype: ab_dtype or GEMM_DT_F32; an fp32
 *   ab_dtype needs an fp32 C and ignores split_k and the workspace).
 */
gemm_status_t gemm_batched(gemm_dtype_t ab_dtype, int64_t batch,
                           int64_t M, int64_t N, int64_t K,
                           const void* A, int64_t lda, gemm_layout_t la, int64_t stride_a,
                           const void* B, int64_t ldb, gemm_layout_t lb, int64_t stride_b,
                           void* C, int64_t ldc, gemm_layout_t lc, int64_t stride_c,
                           gemm_dtype_t c_dtype,
                           float alpha, float beta, const float* bias, gemm_epilogue_t epi,
                           int split_k, void* workspace, size_t workspace_bytes,
                           gemm_stream_t stream);

/*
 * gemm_workspace_size -- bytes of workspace that suffice for any call with these
 * sizes, whatever the layouts, leading dimensions and pointer alignment
 * (an upper bound; 0 when no plan can need scratch).  Queries the current
 * device's SM count.  Returns 0 for invalid sizes.
 */
size_t gemm_workspace_size(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N,
                           int64_t K, int split_k);

/*
 * gemm_strided -- gemm_batched with every matrix given by element strides:
 * element (r, c) of batch b of A sits at A + b*stride_a + r*a_rs + c*a_cs, and
 * likewise for B (K x N) and C (M x N) ("Skill: Write a Triton GEMM Kernel",
 * Kernel design rules: strides are arguments, so non-contiguous tensors work).
 *
 *   Strides are in elements and >= 0.  An input stride of 0 repeats a row, a
 *   column or (batch stride) a whole matrix.  C's strides must give distinct
 *   elements distinct addresses; r*c_rs + c*c_cs is not checked for
 *   overlaps beyond c_rs, c_cs > 0 (when M, N > 1) and stride_c > 0 (batch > 1).
 *   A matrix whose strides are a row-major (cs == 1, rs >= columns) or
 *   column-major (rs == 1, cs >= rows) layout is used in place.  Any other A
 *   or B is first gathered into a dense row-major copy in the workspace, and
 *   any other C is computed in a dense row-major buffer in the workspace
 *   (gathered from C first when beta != 0) and then scattered into C.  All of
 *   it is enqueued on `stream`.
 *   The other arguments are those of gemm_batched.  The workspace must hold
 *   gemm_strided_workspace_size() bytes when a copy is needed
 *   (GEMM_ERR_WORKSPACE otherwise) and be 256-byte aligned.
 */
gemm_status_t gemm_strided(gemm_dtype_t ab_dtype, int64_t batch,
                           int64_t M, int64_t N, int64_t K,
                           const void* A, int64_t a_rs, int64_t a_cs, int64_t stride_a,
                           const void* B, int64_t b_rs, int64_t b_cs, int64_t stride_b,
                           void* C, int64_t c_rs, int64_t c_cs, int64_t stride_c,
                           gemm_dtype_t c_dtype,
                           float alpha, float beta, const float* bias, gemm_epilogue_t epi,
                           int split_k, void* workspace, size_t workspace_bytes,
                           gemm_stream_t stream);

/*
 * gemm_strided_workspace_size -- bytes of workspace that suffice for
 * gemm_strided with these sizes and strides: the dense copies it needs plus
 * gemm_workspace_size() for the GEMM itself.  Returns 0 for invalid arguments.
 */
size_t gemm_strided_workspace_size(gemm_dtype_t ab_dtype, gemm_dtype_t c_dtype, int64_t batch,
                                   int64_t M, int64_t N, int64_t K,
                                   int64_t a_rs, int64_t a_cs, int64_t stride_a,
                                   int64_t b_rs, int64_t b_cs, int64_t stride_b,
                                   int64_t c_rs, int64_t c_cs, int64_t stride_c, int split_k);

/* gemm_status_string -- static, human-readable name of a status code. */
const char* gemm_status_string(gemm_status_t status);

/*
 * gemm_check_device_status -- synchronises `stream`, then reads and clears the
 * current device's error word, which a kernel sets when one of its bounded
 * waits expires (or, in the debug build, when a device-side check fails).
 * Returns GEMM_ERR_DEVICE_CHECK if a check failed, else GEMM_ERR_TIMEOUT if a
 * wait expired, GEMM_ERR_CUDA if the synchronisation failed, else GEMM_OK.
 * For tests and debugging; it blocks.
 */
gemm_status_t gemm_check_device_status(gemm_stream_t stream);

/*
 * Debug build (libdgemm_gb300_debug.so: the same sources and entry points
 * compiled with device-side checks; the pages have no counterpart, this is an
 * interface of this library only).  Its kernels check, before each access,
 * that global addresses lie inside the buffers the call described (C's span,
 * the bias, the split-K partials, the stream-K slots and flags), that TMA
 * store boxes start inside the output, that every decoded work unit lies
 * inside the problem, and that shared-memory stages are aligned.  A failed
 * check sets a bit of the device status word and skips the access (no trap,
 * no assert); gemm_check_device_status then returns GEMM_ERR_DEVICE_CHECK.
 *
 * gemm_build_flags -- bit 0 set in the debug build, 0 in the product library.
 */
int32_t gemm_build_flags(void);

/*
 * gemm_debug_count_writes -- count-writes mode of the debug build.  With a
 * non-NULL `counts` (device memory of count_elems uint32 values, zeroed by
 * the caller), every later GEMM call of this process adds one to
 * counts[(b * M + i) * N + j] each time it writes the final value of C(b, i, j)
 * (the caller's batch entry, row and column, whatever C's layout), so that a
 * correct call leaves exactly 1 in each of its batch * M * N counters.  Split-K
 * partials and stream-K partial tiles are not final values and are not
 * counted; gemm_strided's scatter of a dense result is not counted either.
 * Calls whose batch * M * N exceeds count_elems return GEMM_ERR_INVALID_ARG
 * while the mode is on.  NULL turns the mode off.  The caller owns `counts`.
 * Returns GEMM_ERR_UNSUPPORTED in the product library.
 */
gemm_status_t gemm_debug_count_writes(uint32_t* counts, int64_t count_elems);

/*
 * Plan inspection (no launch): fills *plan with the kernel choice that
 * gemm_batched would make for the same arguments.  Pointers are only
 * inspected for alignment, never dereferenced.
 */
typedef struct {
    int32_t kernel;          /* 0 none, 1 tcgen05 tensor-core, 2 CUDA-core fp32, 3 epilogue only */
    int32_t block_m, block_n, block_k;
    int32_t stages;
    int32_t split_k;         /* K slices (1 = none)                                */
    int32_t swap_ab;         /* 1: computed as C^T = B^T A^T                       */
    int32_t pack_a, pack_b;  /* 1: operand copied into the workspace first         */
    int32_t grid;            /* CTAs of the main kernel                            */
    int32_t group_m;         /* tile-order grouping                                */
    int32_t launches;        /* kernels enqueued by the call                       */
    int64_t workspace_bytes; /* workspace the plan uses                            */
    int32_t cta_pair;        /* 0 one CTA per tile; 2 CTA pair computing 256-row tiles
                                with two-CTA (cta_group::2) MMAs, each CTA loading
                                its own half of A and B (1 is not used)            */
    int32_t stream_k;        /* stream-K: 0 off; 1 the K steps of the last one-to-two
                                waves (or, for an automatic split-K, of every tile)
                                split evenly over all CTAs in contiguous ranges;
                                2 each unit of the last partial wave cut into equal
                                K pieces that run side by side; 3 the same with every
                                piece reducing an equal share of its tile; 4 K steps
                                dealt as in 1 with every piece adding its partial
                                into C (GEMM_OPT_SPLIT_REDUCE = 4)                */
    int32_t fast_epilogue;   /* 0: the general epilogue (four warps); 1: the TMA-store-only
                                epilogue; 2: the TMA-store epilogue that reads beta * C by
                                TMA loads (GEMM_OPT_FAST_EPILOGUE); 3 and 4: 0 and 2 on
                                eight warps (GEMM_OPT_EPILOGUE_WARPS)                  */
} gemm_plan_t;

gemm_status_t gemm_plan_query(gemm_dtype_t ab_dtype, int64_t batch,
                              int64_t M, int64_t N, int64_t K,
                              const void* A, int64_t lda, gemm_layout_t la, int64_t stride_a,
                              const void* B, int64_t ldb, gemm_layout_t lb, int64_t stride_b,
                              void* C, int64_t ldc, gemm_layout_t lc, int64_t stride_c,
                              gemm_dtype_t c_dtype, float alpha, float beta,
                              const float* bias, gemm_epilogue_t epi,
                              int split_k, size_t workspace_bytes, gemm_plan_t* plan);

/*
 * gemm_strided_plan_query -- the plan gemm_strided would follow for these
 * arguments, without enqueuing anything (host only; nothing is read through
 * the pointers, whose alignment alone is used).  The plan is that of the
 * gemm_batched call on the dense layouts, with pack_a / pack_b also set for an
 * A or B gathered into a copy, launches counting the gathers and the scatter,
 * and workspace_bytes including the copies.  Returns what gemm_strided would
 * return before enqueuing (GEMM_ERR_WORKSPACE when workspace_bytes cannot hold
 * the copies and the inner plan).  The copies' placement assumes a 256-byte
 * aligned workspace, as gemm_strided requires.
 */
gemm_status_t gemm_strided_plan_query(gemm_dtype_t ab_dtype, int64_t batch,
                                      int64_t M, int64_t N, int64_t K,
                                      const void* A, int64_t a_rs, int64_t a_cs, int64_t stride_a,
                                      const void* B, int64_t b_rs, int64_t b_cs, int64_t stride_b,
                                      void* C, int64_t c_rs, int64_t c_cs, int64_t stride_c,
                                      gemm_dtype_t c_dtype, float alpha, float beta,
                                      const float* bias, gemm_epilogue_t epi, int split_k,
                                      size_t workspace_bytes, gemm_plan_t* plan);

/*
 * Process-wide tuning knobs (for measurements and tests; defaults are what the
 * library ships with).  Returns GEMM_ERR_INVALID_ARG for an unknown option or
 * value out of range.
 *   GEMM_OPT_GROUP_M      tile-order group size ("Skill: Write a Triton GEMM
 *                         Kernel", step 2; 1 = plain row-major tile order), 1..64.
 *   GEMM_OPT_MAX_CTAS     cap on persistent CTAs (0 = one per SM).
 *   GEMM_OPT_TIMEOUT_US   bound on any single in-kernel wait, microseconds (>= 1).
 *   GEMM_OPT_CTA_PAIR     0 (default): two-CTA MMA pairs along M when a problem has a
 *                         full wave of tile pairs and K >= 768; 1: never; 3: two-CTA
 *                         MMA pairs whenever the tile width allows.  2 is refused
 *                         (GEMM_ERR_INVALID_ARG).
 *   GEMM_OPT_SWAP_AB      0 (default): compute C^T = B^T A^T when M <= 64 < N;
 *                         1: never; 2: always.
 *   GEMM_OPT_L2_HINTS     L2 policy of the tensor-core operand loads: 0 (default) normal;
 *                         1: A evict-first, B evict-last; 2: A evict-last, B evict-first.
 *   GEMM_OPT_STREAM_K     stream-K ("2 . La GEMM, de zero a cuBLAS", section 2.10) for a
 *                         partial last wave after at least one whole wave of tiles:
 *                         0 (default): cut each of the r last tiles into S = P / r
 *                         equal K pieces (P: CTAs or CTA pairs of the grid) when a
 *                         cost model says the shorter last wave outweighs the extra
 *                         partial-tile traffic and the workspace holds the partials;
 *                         1: never; 2: force the contiguous form (plan stream_k 1);
 *                         3: force the split form (plan stream_k 2) when S >= 2.
 *                         A call with split_k == 1 never takes stream-K pieces.
 *   GEMM_OPT_FAST_EPILOGUE 0 (default): when no beta * C is read (beta == 0, or split-K
 *                         partials) and C takes TMA stores, use the epilogue built for
 *                         that case alone (64-column steps, fewer registers); when a
 *                         16-bit C that takes TMA stores is read (beta != 0), use the
 *                         same epilogue with beta * C brought in by TMA loads (two
 *                         64-column boxes ahead per epilogue warp); 1: always the
 *                         general epilogue.
 *   GEMM_OPT_SGEMM_KERNEL 0 (default): the fp32 CUDA-core path with row-major A and B
 *                         whose rows are 16-byte aligned uses the kernel that copies
 *                         tiles with cp.async and issues packed fp32 FMAs (128 x 64
 *                         tiles, three CTAs per SM); other layouts use the register-
 *                         staged kernel (128 x 128 tiles); 1: always the register-staged
 *                         kernel.  Both add each output's products in ascending k with
 *                         one rounding per FMA, so their results are identical.
 *   GEMM_OPT_WIDE_TILE    two-CTA MMA pairs with 256 x 512 tiles (two N = 256 MMAs per
 *                         K step, one accumulator): 0 (default) and 1 never (they
 *                         measured slower than 256 x 256 on bf16 8192^3); 2 whenever
 *                         pair MMA runs with 256-wide tiles and N >= 512.
 *   GEMM_OPT_SPLIT_REDUCE how an automatic split-K (split_k = 0, no whole wave of
 *                         tiles) runs in one kernel: 0 (default) with up to 4 K pieces
 *                         per tile, the K steps of all tiles are dealt to every CTA
 *                         in equal contiguous ranges and the piece holding a tile's
 *                         first step adds the others' fp32 partials (plan stream_k 1);
 *                         with more pieces, for an fp32 C that takes TMA stores and no
 *                         activation, the atomic form below (plan stream_k 4), else
 *                         each piece publishes a partial and, once all have, reduces
 *                         one equal share of the tile (plan stream_k 3);
 *                         1 the serial form up to 4 pieces and the two-pass form
 *                         (split_k > 1, a second launch) beyond; 2 the spread form for
 *                         any number of pieces (1 and 2 keep a fixed order of addition,
 *                         so results repeat bit for bit); 3 as 0, but up to 4 pieces
 *                         as equal K pieces, one CTA each (plan stream_k 2); 4 the
 *                         atomic form whenever it applies (an fp32 C that takes TMA
 *                         stores, no activation; plan stream_k 4): K steps dealt to
 *                         every CTA as in 0, and every
 *                         piece adds alpha times its partial into C by TMA reduce-add
 *                         after the CTAs have set C to beta * C + bias (the order of
 *                         the additions varies between runs, so the last bits may
 *                         too); other calls as 0.  The one-kernel forms are
 *                         cooperative launches and need the workspace of
 *                         gemm_workspace_size.
 *   GEMM_OPT_BLOCK_N      tile width of the tensor-core path: 0 (default) chosen by
 *                         the plan, else 16, 32, 64, 128 or 256 (an MN-major B takes
 *                         at least 64).
 *   GEMM_OPT_DOUBLE_K     0 (default): plans whose kernel form has it (CTA pairs with
 *                         128- or 256-column tiles and the TMA-store-only epilogue;
 *                         single CTAs of at least 8 K blocks with 16- to 64-column
 *                         tiles and the general epilogue, or 64- to 256-column tiles
 *                         and the TMA-store-only one), whole tiles or stream-K
 *                         pieces, bring two 64-deep K blocks of each operand per TMA
 *                         load (plan block_k 128); a K-major operand then needs K a
 *                         multiple of 64 and one matrix (one batch entry or a
 *                         broadcast), an MN-major one nothing more; 1: one K block
 *                         per load always.
 *   GEMM_OPT_OVERLAP_COPY 0 (default): when a call first copies an operand TMA cannot
 *                         address, the GEMM is launched as that copy's programmatic
 *                         dependent (not for the cooperative stream-K forms): its
 *                         CTAs set up while the copy runs and wait for the copy's
 *                         completion before their first operand load; 1: the GEMM
 *                         starts after the copy in plain stream order.
 *   GEMM_OPT_EPILOGUE_WARPS 0 (default): whole 256-wide CTA-pair tiles run their
 *                         epilogue on eight warps, each writing half of a lane
 *                         quarter's columns, when their output takes plain stores
 *                         (rows, base or batch stride not 16-byte aligned, or a
 *                         column-major C; plan fast_epilogue 3) or when beta * C
 *                         is read by TMA loads and K is at most 32 blocks of 64
 *                         (plan fast_epilogue 4); 4: four warps always.
 *   GEMM_OPT_TEST_SIM_SMS test only: n > 0 makes gemm_plan_query and
 *                         gemm_workspace_size plan for a simulated sm_103 device of n
 *                         SMs whose CTA pairs of every tile width fit n / 2 at once,
 *                         instead of the current device, so that plans can be
 *                         checked without a GPU (calls that run GEMMs still need
 *                         one); 0 (default) off.
 *   GEMM_OPT_TEST_STALL   test only: 1 makes the next tensor-core launch leave one
 *                         pipeline stage unfilled, so its consumer's bounded wait
 *                         expires and the kernel reports GEMM_ERR_TIMEOUT; 2 makes
 *                         the first CTA of the next launch with stream-K pieces
 *                         leave its partial unpublished, so the waits of the
 *                         pieces that need it expire instead.  The knob resets
 *                         itself after that launch.
 *   GEMM_OPT_TEST_DEBUG_BOUND  debug build, test only: the next tensor-core launch
 *                         gets one bound of its device-side checks set too small
 *                         (the buffers themselves are untouched), so that a check
 *                         fails and its access is skipped: 1 C's span is halved; 2
 *                         the last tile column counts as outside the problem.
 *                         Resets itself after that launch.  The product library
 *                         refuses it (GEMM_ERR_UNSUPPORTED).
 */
typedef enum {
    GEMM_OPT_GROUP_M = 1,
    GEMM_OPT_MAX_CTAS = 2,
    GEMM_OPT_TIMEOUT_US = 3,
    GEMM_OPT_TEST_STALL = 4,
    GEMM_OPT_CTA_PAIR = 5,
    GEMM_OPT_SWAP_AB = 6,
    GEMM_OPT_L2_HINTS = 7,
    GEMM_OPT_STREAM_K = 8,
    GEMM_OPT_FAST_EPILOGUE = 9,
    GEMM_OPT_SGEMM_KERNEL = 10,
    GEMM_OPT_WIDE_TILE = 11,
    GEMM_OPT_SPLIT_REDUCE = 12,
    GEMM_OPT_BLOCK_N = 13,
    GEMM_OPT_DOUBLE_K = 14,
    GEMM_OPT_TEST_SIM_SMS = 15,
    GEMM_OPT_TEST_DEBUG_BOUND = 16,
    GEMM_OPT_OVERLAP_COPY = 17,
    GEMM_OPT_EPILOGUE_WARPS = 18
} gemm_option_t;

gemm_status_t gemm_set_option(gemm_option_t option, int64_t value);
int64_t gemm_get_option(gemm_option_t option);

/*
 * gemm_tile_order -- host copy of the kernels' tile order: writes, for every
 * work index t in [0, num_pid_m*num_pid_n), the tile (pid_m[t], pid_n[t]) it
 * computes, for grouping `group_m` ("Skill: Write a Triton GEMM Kernel",
 * Required reasoning process step 2).  The caller sizes both arrays; invalid
 * arguments write nothing.  Needs no GPU.
 */
void gemm_tile_order(int num_pid_m, int num_pid_n, int group_m, int* pid_m, int* pid_n);

/*
 * gemm_bf16_static_workspace -- gemm_bf16 for callers that cannot allocate
 * device memory.  (The pages have no counterpart: this is an interface of
 * this library only.)
 *
 * Some callers cannot call cudaMalloc or hand over a workspace: code that
 * runs where a host framework has already reserved the device's memory for
 * its own allocator, plugin hooks whose contract forbids allocation during
 * execution, and latency-critical loops that must not enter the allocator
 * (cudaMalloc can synchronise the device).  This entry point takes the same
 * arguments as gemm_bf16 minus the workspace; its scratch (split-K partial
 * tiles and aligned operand copies) is a library-owned device array of
 * GEMM_STATIC_WORKSPACE_BYTES bytes that every GPU loading the library keeps
 * until the process exits.  No call allocates anything.
 *
 *   - Limit: a plan that needs more than GEMM_STATIC_WORKSPACE_BYTES of
 *     scratch is rejected with GEMM_ERR_WORKSPACE before anything is
 *     enqueued (split_k > 1 too large for the array, or operand copies that
 *     do not fit); with split_k == 0 the split is reduced to fit.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture begins.
 *   - All calls share the one array, and it keeps the last call's contents.
 *     Nothing in it needs to start at zero.  Split-K partial tiles and
 *     operand copies are written before they are read.  The stream-K flags
 *     that K pieces poll are read before their publisher writes them, so
 *     they may still hold an earlier call's values; a piece takes a partial
 *     only once its flag equals the launch's epoch, a fresh non-zero value
 *     for every call (and a call made during a stream capture clears the
 *     flags inside the graph first).  Calls whose work overlaps on the GPU
 *     (on different streams, or from different host threads without
 *     ordering) race on the array and may produce wrong results: order them.
 */
#define GEMM_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

gemm_status_t gemm_bf16_static_workspace(int64_t M, int64_t N, int64_t K,
                                         const void* A, int64_t lda, gemm_layout_t la,
                                         const void* B, int64_t ldb, gemm_layout_t lb,
                                         void* C, int64_t ldc, gemm_layout_t lc,
                                         gemm_dtype_t c_dtype, float alpha, float beta,
                                         const float* bias, gemm_epilogue_t epi, int split_k,
                                         gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_GB300_GEMM_H */
