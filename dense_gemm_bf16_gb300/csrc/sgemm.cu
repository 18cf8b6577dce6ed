// True-fp32 GEMM on the CUDA cores (FMA pipe; no tensor cores, no TF32).
//
// Two kernels.  Row-major A and B with 16-byte aligned rows (the common
// layout) take sgemm_rr_kernel, further below: cp.async tile copies and
// packed fp32 FMAs.  Every other layout takes sgemm_kernel, the
// register-tiled design of "2 . La GEMM, de zero a cuBLAS", sections 2.3-2.8,
// for sm_103a:
//   - a 128 x 128 output tile per CTA of 256 threads (section 2.6: BM = BN =
//     128, TM = TN = 8), K consumed 16 at a time (the page's BK = 8 doubled
//     to halve the synchronisations and tile loads per FMA);
//   - each thread accumulates an 8 x 8 block as outer products of 8 values of
//     A and 8 values of B per k: 16 shared-memory reads for 64 FMAs
//     (section 2.6); its rows are {4ty..4ty+3, 64+4ty..64+4ty+3} and its
//     columns {4tx..4tx+3, 64+4tx..64+4tx+3}, so every read is a float4 and
//     the reads of one warp touch each bank at most once per wavefront;
//   - the A tile is stored transposed, As[k][m], so a thread's column of A is
//     contiguous and vectorisable (section 2.7);
//   - global loads are float4 (LDG.128) when alignment allows (section 2.7)
//     and land in the second of two shared buffers while the first is
//     consumed (section 2.8), one __syncthreads per K step; the operand
//     fragments of step k+1 are also read while step k computes;
//   - one CTA per SM (up to 255 registers, no spills), which also gives more
//     waves and a smaller tail at 4096^2;
//   - consecutive threads read consecutive addresses of each operand row
//     (coalescing, section 2.3);
//   - ragged M / N / K edges are masked with zero fill, and the store is
//     masked on M and N.
// Tiles are ordered by the grouped schedule of tile_order.h; batch is the slowest
// index of the 1-D grid.
#include <stdint.h>

#include "epilogue.cuh"
#include "internal.h"
#include "tile_order.h"

namespace dg {
namespace {

constexpr int SBM = 128, SBN = 128, SBK = 16, STHREADS = 256;

// Global -> register staging of one 128 x 16 A tile and one 16 x 128 B tile:
// two float4 of each per thread.  Mapping (thread t):
//   K-contiguous operand (row-major A, column-major B): row r = t % 64 (+64),
//     k offset 4 * (t / 64); a warp covers 32 consecutive rows at one k
//     offset, so the transposed shared-memory stores hit 32 distinct banks.
//   MN-contiguous operand: k = t / 32 (+8), mn offset 4 * (t % 32); a warp
//     reads 512 contiguous bytes and stores one float4 each.
struct Frag4 {
    float4 v[2];
};

template <bool KCONTIG>
__device__ __forceinline__ Frag4 load_tile(const float* __restrict__ X, int64_t ld, int mn0,
                                           int mn_ext, int k0, int K, bool vec_ok, int tid) {
    Frag4 f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (KCONTIG) {
            const int r = mn0 + (tid & 63) + 64 * h;
            const int k = k0 + ((tid >> 6) << 2);
            if (r < mn_ext) {
                const float* src = X + static_cast<int64_t>(r) * ld + k;
                if (vec_ok && k + 3 < K) {
                    v = *reinterpret_cast<const float4*>(src);
                } else {
                    if (k + 0 < K) v.x = src[0];
                    if (k + 1 < K) v.y = src[1];
                    if (k + 2 < K) v.z = src[2];
                    if (k + 3 < K) v.w = src[3];
                }
            }
        } else {
            const int k = k0 + (tid >> 5) + 8 * h;
            const int r = mn0 + ((tid & 31) << 2);
            if (k < K) {
                const float* src = X + static_cast<int64_t>(k) * ld + r;
                if (vec_ok && r + 3 < mn_ext) {
                    v = *reinterpret_cast<const float4*>(src);
                } else {
                    if (r + 0 < mn_ext) v.x = src[0];
                    if (r + 1 < mn_ext) v.y = src[1];
                    if (r + 2 < mn_ext) v.z = src[2];
                    if (r + 3 < mn_ext) v.w = src[3];
                }
            }
        }
        f.v[h] = v;
    }
    return f;
}

// Store a staged tile as S[k][mn] (k-major rows of 128 floats).
template <bool KCONTIG>
__device__ __forceinline__ void store_tile(float (*S)[SBM], const Frag4& f, int tid) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (KCONTIG) {
            const int r = (tid & 63) + 64 * h;
            const int k = (tid >> 6) << 2;
            S[k + 0][r] = f.v[h].x;
            S[k + 1][r] = f.v[h].y;
            S[k + 2][r] = f.v[h].z;
            S[k + 3][r] = f.v[h].w;
        } else {
            const int k = (tid >> 5) + 8 * h;
            const int r = (tid & 31) << 2;
            *reinterpret_cast<float4*>(&S[k][r]) = f.v[h];
        }
    }
}

// Epilogue of one thread's 8 x 8 block: rows 4ty+i (+64), columns 4tx+j (+64).
__device__ __forceinline__ void sgemm_store(const SgemmParams& p, int b, int m0, int n0, int tx,
                                            int ty, const float (&acc)[8][8]) {
    const Epilogue& e = p.epi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= p.M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h * 64 + tx * 4;
            if (e.c_row_major && e.c_vec_ok && n + 3 < p.N) {
                if (!c_span_ok(e, c_off(e, b, m, n), 4)) continue;
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = e.alpha * acc[i][4 * h + j];
                float4* c = reinterpret_cast<float4*>(c_addr(e, b, m, n));
                if (e.beta != 0.f) {
                    const float4 o = *c;
                    v[0] = fmaf(e.beta, o.x, v[0]);
                    v[1] = fmaf(e.beta, o.y, v[1]);
                    v[2] = fmaf(e.beta, o.z, v[2]);
                    v[3] = fmaf(e.beta, o.w, v[3]);
                }
                if (e.bias && bias_ok(e, e.bias_on_rows ? m : n + 3)) {
                    if (e.bias_on_rows) {
                        const float br = e.bias[m];
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[j] += br;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[j] += e.bias[n + j];
                    }
                }
                act_inplace<4>(v, e.act);
                *c = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) count_write(e, b, m, n + j);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < p.N) epilogue_store(e, b, m, n + j, acc[i][4 * h + j]);
            }
        }
    }
}

template <bool A_ROW, bool B_ROW>
__global__ void __launch_bounds__(STHREADS, 1) sgemm_kernel(const __grid_constant__ SgemmParams p) {
    __shared__ __align__(16) float As[2][SBK][SBM];
    __shared__ __align__(16) float Bs[2][SBK][SBN];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int tiles = p.num_pid_m * p.num_pid_n;
    const int b = blockIdx.x / tiles;
    int pid_m, pid_n;
    tile_coord(blockIdx.x - b * tiles, p.num_pid_m, p.num_pid_n, p.group_m, pid_m, pid_n);
    const int m0 = pid_m * SBM, n0 = pid_n * SBN;
    const float* __restrict__ A = p.A + static_cast<int64_t>(b) * p.stride_a;
    const float* __restrict__ B = p.B + static_cast<int64_t>(b) * p.stride_b;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int nk = (p.K + SBK - 1) / SBK;
    // A is K-contiguous when row-major; B is K-contiguous when column-major
    Frag4 fa = load_tile<A_ROW>(A, p.lda, m0, p.M, 0, p.K, p.a_vec_ok, tid);
    Frag4 fb = load_tile<!B_ROW>(B, p.ldb, n0, p.N, 0, p.K, p.b_vec_ok, tid);
    store_tile<A_ROW>(As[0], fa, tid);
    store_tile<!B_ROW>(Bs[0], fb, tid);
    __syncthreads();

    for (int kt = 0; kt < nk; ++kt) {
        const int cur = kt & 1;
        const bool more = kt + 1 < nk;
        if (more) {
            fa = load_tile<A_ROW>(A, p.lda, m0, p.M, (kt + 1) * SBK, p.K, p.a_vec_ok, tid);
            fb = load_tile<!B_ROW>(B, p.ldb, n0, p.N, (kt + 1) * SBK, p.K, p.b_vec_ok, tid);
        }
        // outer products; the float4 fragments of step k+1 are read while step
        // k computes and are used in place (no copies between the load and the FMAs)
        float4 xa0[2], xa1[2], xb0[2], xb1[2];
        xa0[0] = *reinterpret_cast<const float4*>(&As[cur][0][ty * 4]);
        xa1[0] = *reinterpret_cast<const float4*>(&As[cur][0][64 + ty * 4]);
        xb0[0] = *reinterpret_cast<const float4*>(&Bs[cur][0][tx * 4]);
        xb1[0] = *reinterpret_cast<const float4*>(&Bs[cur][0][64 + tx * 4]);
#pragma unroll
        for (int k = 0; k < SBK; ++k) {
            const int c = k & 1;
            if (k + 1 < SBK) {
                xa0[c ^ 1] = *reinterpret_cast<const float4*>(&As[cur][k + 1][ty * 4]);
                xa1[c ^ 1] = *reinterpret_cast<const float4*>(&As[cur][k + 1][64 + ty * 4]);
                xb0[c ^ 1] = *reinterpret_cast<const float4*>(&Bs[cur][k + 1][tx * 4]);
                xb1[c ^ 1] = *reinterpret_cast<const float4*>(&Bs[cur][k + 1][64 + tx * 4]);
            }
            const float a[8] = {xa0[c].x, xa0[c].y, xa0[c].z, xa0[c].w,
                                xa1[c].x, xa1[c].y, xa1[c].z, xa1[c].w};
            const float bb[8] = {xb0[c].x, xb0[c].y, xb0[c].z, xb0[c].w,
                                 xb1[c].x, xb1[c].y, xb1[c].z, xb1[c].w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
        }
        if (more) {
            store_tile<A_ROW>(As[cur ^ 1], fa, tid);
            store_tile<!B_ROW>(Bs[cur ^ 1], fb, tid);
        }
        __syncthreads();
    }

    sgemm_store(p, b, m0, n0, tx, ty, acc);
}

// ------------------------------------------------------------------ row-major A and B
// For row-major A and B with 16-byte aligned rows (the common layout), a
// smaller tile and more warps: a 128 x 64 output tile per CTA of NT threads,
// K consumed BK at a time, each thread an 8 x TN block (rows ty + 16 i,
// columns in float4 groups).  The tiles go global -> shared with cp.async (16
// bytes per copy, zero fill past the M / N / K edges) through a ring of
// STAGES buffers ("2 . La GEMM, de zero a cuBLAS", section 2.8), with no
// register staging and no transpose: A stays [m][k], rows padded by 4 floats,
// and a thread reads each of its rows as a float4 of four consecutive k; B
// stays [k][n] and is read as float4.  Several CTAs share an SM.
// The FMAs are sm_100's packed fma.rn.f32x2 (__ffma2_rn): two IEEE fp32 FMAs
// per instruction, each rounded once, on accumulator pairs along n,
// (a_i, a_i) * (b_2q, b_2q+1) + acc.  They halve the issue slots the FMA work
// takes, which is what held the scalar form near 65 % of the pipe's peak.
// Every output still adds its products in ascending k with one rounding per
// FMA, so the results equal the register-staged kernel's bit for bit.
constexpr int RBM = 128, RBN = 64;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
                 "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ int clamp16(int64_t bytes) {
    return bytes <= 0 ? 0 : (bytes >= 16 ? 16 : static_cast<int>(bytes));
}

template <int NT, int BK, int STAGES>
struct RrCfg {
    static constexpr int SA_LD = BK + 4;           // A row pitch (floats): adjacent rows differ in bank
    static constexpr int A_COPIES = RBM * BK / 4;  // 16-byte copies per A tile
    static constexpr int B_COPIES = BK * RBN / 4;
    static constexpr int A_PER_ROW = BK / 4;
    static constexpr int A_FLOATS = RBM * SA_LD;   // one stage
    static constexpr int B_FLOATS = BK * RBN;
    static constexpr size_t SMEM = size_t(STAGES) * (A_FLOATS + B_FLOATS) * sizeof(float);
    static_assert(A_COPIES % NT == 0 && B_COPIES % NT == 0, "copies divide evenly");
    static constexpr int MIN_BLOCKS = NT == 256 ? 2 : 3;
};

// One stage: copy c of A is row c / (BK / 4), k 4 * (c % (BK / 4)); copy c of
// B is k c / 16, n 4 * (c % 16).  A copy that would start past an edge reads
// nothing and fills zeros, with the operand's base address as its source.
template <int NT, int BK, int STAGES>
__device__ __forceinline__ void sgemm_rr_issue(const SgemmParams& p, const float* A,
                                               const float* B, float* As, float* Bs, int m0,
                                               int n0, int k0, int tid) {
    using R = RrCfg<NT, BK, STAGES>;
#pragma unroll
    for (int h = 0; h < R::A_COPIES / NT; ++h) {
        const int c = tid + h * NT;
        const int r = c / R::A_PER_ROW, kc = (c % R::A_PER_ROW) * 4, k = k0 + kc;
        const bool ok = m0 + r < p.M && k < p.K;
        const int nb = ok ? clamp16(static_cast<int64_t>(p.K - k) * 4) : 0;
        const float* src = ok ? A + static_cast<int64_t>(m0 + r) * p.lda + k : A;
        cp_async16(As + r * R::SA_LD + kc, src, nb);
    }
#pragma unroll
    for (int h = 0; h < R::B_COPIES / NT; ++h) {
        const int c = tid + h * NT;
        const int kr = c >> 4, nc = (c & 15) << 2, n = n0 + nc;
        const bool ok = k0 + kr < p.K && n < p.N;
        const int nb = ok ? clamp16(static_cast<int64_t>(p.N - n) * 4) : 0;
        const float* src = ok ? B + static_cast<int64_t>(k0 + kr) * p.ldb + n : B;
        cp_async16(Bs + kr * RBN + nc, src, nb);
    }
}

// The same copies for a tile that lies wholly inside A and B: the per-thread
// source offsets are computed once and only advance by one K tile.
struct RrOffsets {
    int64_t a0, b0;          // elements from the operand base at k0 = 0 (first copy)
    int64_t a_step, b_step;  // between a thread's successive copies of one tile
};

template <int NT, int BK, int STAGES>
__device__ __forceinline__ void sgemm_rr_issue_interior(const float* A, const float* B,
                                                        const RrOffsets& o, int64_t ldb,
                                                        float* As, float* Bs, int k0, int tid) {
    using R = RrCfg<NT, BK, STAGES>;
    const int ar = tid / R::A_PER_ROW, akc = (tid % R::A_PER_ROW) * 4;
#pragma unroll
    for (int h = 0; h < R::A_COPIES / NT; ++h)
        cp_async16(As + (ar + h * (NT / R::A_PER_ROW)) * R::SA_LD + akc,
                   A + o.a0 + h * o.a_step + k0, 16);
#pragma unroll
    for (int h = 0; h < R::B_COPIES / NT; ++h)
        cp_async16(Bs + ((tid >> 4) + h * (NT / 16)) * RBN + ((tid & 15) << 2),
                   B + o.b0 + h * o.b_step + static_cast<int64_t>(k0) * ldb, 16);
}

// Thread (tx, ty), tx < NT / 16, owns rows ty + 16 i (i < 8) and columns
// 4 (NT / 16) g + 4 tx + j (g < TN / 4, j < 4): 256 threads take 8 x 4
// blocks, 128 threads 8 x 8 blocks.
template <int NT, int BK, int STAGES>
__global__ void __launch_bounds__(NT, (RrCfg<NT, BK, STAGES>::MIN_BLOCKS))
    sgemm_rr_kernel(const __grid_constant__ SgemmParams p) {
    using R = RrCfg<NT, BK, STAGES>;
    constexpr int NTX = NT / 16;   // threads along n
    constexpr int TN = RBN / NTX;  // columns per thread
    constexpr int NG = TN / 4;     // float4 groups per thread row
    extern __shared__ __align__(16) float rr_smem[];
    float* const As0 = rr_smem;                             // [STAGES][RBM][SA_LD]
    float* const Bs0 = rr_smem + STAGES * R::A_FLOATS;      // [STAGES][BK][RBN]

    const int tid = threadIdx.x;
    const int tx = tid % NTX, ty = tid / NTX;
    const int tiles = p.num_pid_m * p.num_pid_n;
    const int b = blockIdx.x / tiles;
    int pid_m, pid_n;
    tile_coord(blockIdx.x - b * tiles, p.num_pid_m, p.num_pid_n, p.group_m, pid_m, pid_n);
    const int m0 = pid_m * RBM, n0 = pid_n * RBN;
    const float* __restrict__ A = p.A + static_cast<int64_t>(b) * p.stride_a;
    const float* __restrict__ B = p.B + static_cast<int64_t>(b) * p.stride_b;

    // accumulator pairs along n: acc2[i][q] = (C(row i, col 2q), C(row i, col 2q + 1))
    float2 acc2[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < TN / 2; ++q) acc2[i][q] = make_float2(0.f, 0.f);

    const int nk = (p.K + BK - 1) / BK;
    // K tiles [0, nk_full) are wholly inside K; with the M and N extents of the
    // CTA also inside, their copies need no bounds
    const bool mn_inside = m0 + RBM <= p.M && n0 + RBN <= p.N;
    const int nk_full = mn_inside ? p.K / BK : 0;
    RrOffsets o;
    o.a0 = static_cast<int64_t>(m0 + tid / R::A_PER_ROW) * p.lda + (tid % R::A_PER_ROW) * 4;
    o.a_step = static_cast<int64_t>(NT / R::A_PER_ROW) * p.lda;
    o.b0 = static_cast<int64_t>(tid >> 4) * p.ldb + n0 + ((tid & 15) << 2);
    o.b_step = static_cast<int64_t>(NT / 16) * p.ldb;
    auto issue = [&](int t, int st) {
        float* as = As0 + st * R::A_FLOATS;
        float* bs = Bs0 + st * R::B_FLOATS;
        if (t < nk_full)
            sgemm_rr_issue_interior<NT, BK, STAGES>(A, B, o, p.ldb, as, bs, t * BK, tid);
        else
            sgemm_rr_issue<NT, BK, STAGES>(p, A, B, as, bs, m0, n0, t * BK, tid);
    };
    // the first STAGES - 1 tiles in flight; one commit group per tile (empty
    // past the end) so that the wait below always refers to tile kt
#pragma unroll
    for (int s0 = 0; s0 < STAGES - 1; ++s0) {
        if (s0 < nk) issue(s0, s0);
        cp_async_commit();
    }
    for (int kt = 0; kt < nk; ++kt) {
        const int cur = kt % STAGES;
        cp_async_wait<STAGES - 2>();
        // every thread's copies of tile kt are visible, and the buffer of tile
        // kt - 1 (refilled next) has been read by everyone
        __syncthreads();
        {
            const int nxt = kt + STAGES - 1;
            if (nxt < nk) issue(nxt, nxt % STAGES);
            cp_async_commit();
        }
        const float* as = As0 + cur * R::A_FLOATS;
        const float* bs = Bs0 + cur * R::B_FLOATS;
#pragma unroll
        for (int k = 0; k < BK; k += 4) {
            float4 av[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                av[i] = *reinterpret_cast<const float4*>(as + (ty + 16 * i) * R::SA_LD + k);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float bb[TN];
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float4 bv = *reinterpret_cast<const float4*>(
                        bs + (k + kk) * RBN + 4 * NTX * g + 4 * tx);
                    bb[4 * g + 0] = bv.x;
                    bb[4 * g + 1] = bv.y;
                    bb[4 * g + 2] = bv.z;
                    bb[4 * g + 3] = bv.w;
                }
                // packed FMAs: (a, a) * (b_2q, b_2q+1) + acc pair
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float a = kk == 0 ? av[i].x : kk == 1 ? av[i].y : kk == 2 ? av[i].z : av[i].w;
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int q = 0; q < TN / 2; ++q)
                        acc2[i][q] = __ffma2_rn(a2, make_float2(bb[2 * q], bb[2 * q + 1]), acc2[i][q]);
                }
            }
        }
    }
    cp_async_wait<0>();
    float acc[8][TN];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < TN / 2; ++q) {
            acc[i][2 * q] = acc2[i][q].x;
            acc[i][2 * q + 1] = acc2[i][q].y;
        }

    // epilogue: rows m0 + ty + 16 i, columns n0 + 4 NTX g + 4 tx .. + 3
    const Epilogue& e = p.epi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + ty + 16 * i;
        if (m >= p.M) continue;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int n = n0 + 4 * NTX * g + tx * 4;
            const float* ag = acc[i] + 4 * g;
            if (e.c_row_major && e.c_vec_ok && n + 3 < p.N) {
                if (!c_span_ok(e, c_off(e, b, m, n), 4)) continue;
                float v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = e.alpha * ag[j];
                float4* c = reinterpret_cast<float4*>(c_addr(e, b, m, n));
                if (e.beta != 0.f) {
                    const float4 o4 = *c;
                    v[0] = fmaf(e.beta, o4.x, v[0]);
                    v[1] = fmaf(e.beta, o4.y, v[1]);
                    v[2] = fmaf(e.beta, o4.z, v[2]);
                    v[3] = fmaf(e.beta, o4.w, v[3]);
                }
                if (e.bias && bias_ok(e, e.bias_on_rows ? m : n + 3)) {
                    if (e.bias_on_rows) {
                        const float br = e.bias[m];
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[j] += br;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[j] += e.bias[n + j];
                    }
                }
                act_inplace<4>(v, e.act);
                *c = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) count_write(e, b, m, n + j);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (n + j < p.N) epilogue_store(e, b, m, n + j, ag[j]);
            }
        }
    }
}

template <int NT, int BK, int STAGES>
cudaError_t rr_prepare() {
    return cudaFuncSetAttribute(sgemm_rr_kernel<NT, BK, STAGES>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(RrCfg<NT, BK, STAGES>::SMEM));
}

template <int NT, int BK, int STAGES>
void rr_launch(const SgemmParams& p, dim3 g, cudaStream_t stream) {
    sgemm_rr_kernel<NT, BK, STAGES><<<g, NT, RrCfg<NT, BK, STAGES>::SMEM, stream>>>(p);
}

}  // namespace

// The configuration of the cp.async kernel: 128 threads (8 x 8 blocks), K
// tiles of 32, two stages; 168 registers and 53 KB of shared memory, so three
// CTAs share an SM.
constexpr int RR_NT = 128, RR_BK = 32, RR_STAGES = 2;

cudaError_t sgemm_prepare() { return rr_prepare<RR_NT, RR_BK, RR_STAGES>(); }

cudaError_t sgemm_launch(const SgemmParams& p, cudaStream_t stream) {
    const int64_t grid = static_cast<int64_t>(p.batch) * p.num_pid_m * p.num_pid_n;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const dim3 g(static_cast<unsigned>(grid));
    if (p.kernel == 0)
        rr_launch<RR_NT, RR_BK, RR_STAGES>(p, g, stream);
    else if (p.a_row && p.b_row)
        sgemm_kernel<true, true><<<g, STHREADS, 0, stream>>>(p);
    else if (p.a_row)
        sgemm_kernel<true, false><<<g, STHREADS, 0, stream>>>(p);
    else if (p.b_row)
        sgemm_kernel<false, true><<<g, STHREADS, 0, stream>>>(p);
    else
        sgemm_kernel<false, false><<<g, STHREADS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dg
