// Persistent, warp-specialised tcgen05 GEMM for sm_103a (bf16 / fp16 in, fp32 accumulate).
//
// The tiled algorithm of "GEMM Kernel Optimization", Core Technique (one
// BLOCK_M x BLOCK_N output tile per work unit, K consumed in BLOCK_K slices,
// fp32 accumulator, cast after the loop) mapped onto GB300:
//
//   warp 0 (one lane)  TMA producer: fills a ring of STAGES shared-memory
//                      stages with the A tile [128 x 64 KS] and the B tile
//                      [BN x 64 KS], 128-byte swizzled, out-of-range elements
//                      zero-filled by the TMA unit (the K / M / N masks of
//                      "Skill: Write a Triton GEMM Kernel", step 5).
//   warp 1 (one lane)  MMA issuer: tcgen05.mma kind::f16, M=128, N=BN, K=16,
//                      4 KS per stage, into one of two TMEM accumulators;
//                      tcgen05.commit frees the stage / publishes the tile.
//   warps 2-5          epilogue: tcgen05.ld of the accumulator (one TMEM lane =
//   (2-9 in forms      one output row per thread), alpha/beta/bias/GELU in fp32,
//   3 and 4)           one rounding to the output type, masked global stores;
//                      or, for split-K, the raw fp32 partial tile.  Forms 3
//                      and 4 put two warps on each TMEM lane quarter, each
//                      writing half of the tile's columns.
//
// The two TMEM accumulators let the epilogue of tile i overlap the main loop
// of tile i+1.  Work units (batch, K slice, tile) are dealt to CTAs round
// robin (persistent grid, one CTA per SM); tiles follow the grouped order of
// tile_order.h.  Every mbarrier wait is bounded: on expiry the kernel records an
// error word, lets its own copies and MMAs drain, frees TMEM and returns.
//
// EPI selects the epilogue's output code: 0 handles every case (beta * C
// read with loads one chunk ahead, TMA store or an st.global fallback for a C
// that TMA cannot address); 1 only the TMA store with beta == 0 or a split-K
// partial, in 64-column steps, and so needs far fewer registers; 2 the same
// TMA store with beta * C of a 16-bit C brought in by TMA loads; 3 and 4 are
// 0 and 2 on eight epilogue warps (whole 256-wide pair tiles).  KS is the
// number of 64-deep K blocks per stage (2: one TMA load brings two K blocks of
// a K-major operand).  The forms are instantiated in separate translation
// units (tc_gemm_general.cu, tc_gemm_fast.cu, tc_gemm_beta.cu, tc_gemm_ks2*.cu,
// tc_gemm_epi8.cu) that compile in parallel.
#pragma once
#include <stdint.h>

#include "epilogue.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tile_order.h"

namespace dg {
namespace {

constexpr int BM = TC_BLOCK_M;
constexpr int BK = TC_BLOCK_K;
constexpr uint32_t kMaxDynSmem = 232448;  // 227 KB opt-in limit per CTA

// Shared memory of each epilogue warp: two 4 KB output boxes (32 rows x 128
// bytes, 128-byte swizzled) for the TMA-store epilogue, or one staging tile
// of 32 rows x 32 fp32 columns for the st.global fallback.  Its rows are
// padded to 36 words: a lane writes its row as 16-byte stores, and the eight
// lanes of each 128-byte phase (words 36 t + c .. 36 t + c + 3, t = 0..7) then
// cover 32 distinct banks; the column-wise reads (word 36 r + t for lane t)
// do too.  The epilogue forms that read beta * C (kind 2: EPI 2
// and 4) add a ring of two more boxes per warp that TMA loads fill with C;
// form 4 keeps one output box per warp.
constexpr int STAGE_LD = 36;
constexpr uint32_t EPI_WARP_BYTES = 8192;
constexpr uint32_t EPI_BOX_BYTES = 4096;
constexpr uint32_t C_RING_WARP_BYTES = 2 * EPI_BOX_BYTES;  // two C boxes per epilogue warp
static_assert(32 * STAGE_LD * 4 <= EPI_WARP_BYTES, "staging tile must fit");
static_assert(STAGE_LD % 4 == 0, "16-byte row writes");

// MODE 0: one CTA per 128 x BN tile.
// MODE 2: two CTAs of a cluster compute one 256 x BN tile with cta_group::2
//         MMAs issued by the even CTA; each CTA holds its own 128 A rows and
//         BN/2 B columns, so a stage is 16 KB + BN*64 bytes per CTA.  With
//         BN = 512 the tile is two N = 256 MMAs per K step into the two halves
//         of tensor memory (one accumulator, no double buffering): every CTA
//         takes in 48 KB per 64-deep K block for twice the work of BN = 256
//         (an option: it measured slower than BN = 256).
// EPI: the epilogue form (only its shared memory matters here).
// KS: 64-deep K blocks per pipeline stage.  With KS = 2 (K-major A and B) one
// TMA load brings two K blocks of an operand through a three-dimensional view
// (64 K x rows x K blocks): half as many loads for the same bytes, which lets
// more of the ring's bytes be in flight at once (an SM's TMA unit keeps a
// bounded number of loads outstanding; measured 3 % faster on 8192^3).
template <int BN, int MODE, int EPI = 0, int KS = 1>
struct Cfg {
    static_assert(MODE == 0 || MODE == 2, "one CTA per tile, or a two-CTA MMA pair");
    static constexpr int CM = MODE == 0 ? 1 : 2;        // CTAs per cluster
    static constexpr int CG = MODE == 2 ? 2 : 1;        // tcgen05 cta_group
    static constexpr int B_ROWS = MODE == 2 ? BN / 2 : BN;  // B rows (N) held per CTA
    static constexpr int NSUB = BN > 256 ? BN / 256 : 1;    // MMAs (N <= 256 each) per K step
    static constexpr int SUB_N = BN / NSUB;
    static constexpr int ACC_BUFS = 2 * BN <= 512 ? 2 : 1;  // accumulators in tensor memory
    static constexpr uint32_t A_BYTES = BM * BK * 2 * KS;
    static constexpr uint32_t B_BYTES = B_ROWS * BK * 2 * KS;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t BAR_BYTES = 512;
    // epilogue warps: four (one per tensor-memory lane quarter), or eight in
    // forms 3 and 4 (two per quarter, each taking half of the tile's columns),
    // which are forms 0 and 2 (KIND) on eight warps; form 4 keeps one output
    // box per warp so that the pipeline keeps four stages
    static constexpr int KIND = EPI == 3 ? 0 : (EPI == 4 ? 2 : EPI);
    static constexpr int EPI_WARPS = EPI >= 3 ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr uint32_t EPI_WARP = EPI == 4 ? EPI_BOX_BYTES : EPI_WARP_BYTES;
    static constexpr uint32_t EPI_SMEM =
        EPI_WARPS * (EPI_WARP + (KIND == 2 ? C_RING_WARP_BYTES : 0));
    static constexpr int STAGES_FIT = (kMaxDynSmem - 1024 - BAR_BYTES - EPI_SMEM) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    static constexpr uint32_t TMEM_COLS = ACC_BUFS * BN < 32 ? 32 : ACC_BUFS * BN;
    static constexpr int CHUNK = BN < 32 ? BN : 32;
    static constexpr size_t SMEM = 1024 + size_t(STAGES) * STAGE_BYTES + BAR_BYTES + EPI_SMEM;
    static_assert(STAGES >= 2, "pipeline needs two stages");
    static_assert((2 * STAGES + 6 + 2 * EPI_WARPS) * 8 + 8 <= BAR_BYTES, "barrier area too small");
    static_assert(B_BYTES % 1024 == 0, "stages must stay 1024-byte aligned");
    static_assert(EPI_BOX_BYTES % 1024 == 0 && EPI_WARP_BYTES % 1024 == 0,
                  "swizzled output boxes must be 1024-byte aligned");
    static_assert(MODE != 2 || BN >= 128, "pair MMA splits B into 64-column atoms");
    static_assert(EPI < 3 || (BN % 128 == 0 && KS == 1), "forms 3, 4: whole 64-column steps per half tile");
    static_assert(BN <= 256 || MODE == 2, "N > 256 only as two pair MMAs");
};

struct Unit {
    int b, split, pid_m, pid_n, kb0, kb1;
    // UNIT_FULL, or a stream-K piece: UNIT_HEAD (finishes the tile) / UNIT_TAIL /
    // UNIT_SPREAD (publishes, then reduces share `piece` of the tile)
    int kind;
    // stream-K partial slots: a TAIL or SPREAD piece publishes into slot `slot`;
    // a HEAD adds the `nslots` partials in slots slot .. slot + nslots - 1; a
    // SPREAD piece reads slots slot - piece .. slot - piece + nslots - 1
    int slot, nslots, piece;
};

enum : int { UNIT_FULL = 0, UNIT_HEAD = 1, UNIT_TAIL = 2, UNIT_SPREAD = 3 };

// Work unit u -> (batch, K slice, tile).  With clusters of CM CTAs along M the
// unit is a CM-tile-high slab and CTA `rank` of the cluster takes tile-row
// pid_m * CM + rank of it.
template <int CM>
__device__ __forceinline__ Unit decode_unit(const TcParams& p, int u, uint32_t rank) {
    const int per_batch = p.splits * p.tiles_per_batch;
    Unit w;
    w.b = u / per_batch;
    const int r = u - w.b * per_batch;
    w.split = r / p.tiles_per_batch;
    const int t = r - w.split * p.tiles_per_batch;
    tile_coord(t, p.num_pid_m, p.num_pid_n, p.group_m, w.pid_m, w.pid_n);
    w.pid_m = w.pid_m * CM + static_cast<int>(rank);
    w.kb0 = static_cast<int>(static_cast<int64_t>(w.split) * p.kblocks / p.splits);
    w.kb1 = static_cast<int>(static_cast<int64_t>(w.split + 1) * p.kblocks / p.splits);
    w.kind = UNIT_FULL;
    w.slot = w.nslots = w.piece = 0;
    return w;
}

// The sequence of work items of one cluster; every role of the CTA walks it.
struct WorkIter {
    int cluster;      // this cluster's index
    int unit_rr;      // next round-robin unit
    int rr_left;      // round-robin units left
    int64_t it, end;  // stream-K K-block range (contiguous form)
    int piece;        // split form: this cluster's piece of the last wave, or -1
};

__device__ __forceinline__ WorkIter work_begin(const TcParams& p, int cta0, int ncta) {
    WorkIter s;
    s.cluster = cta0;
    s.unit_rr = cta0;
    s.it = s.end = 0;
    s.piece = -1;
    if (p.sk_iters > 0) {
        s.rr_left = p.dp_per_cluster;
        s.it = p.sk_iters * cta0 / ncta;
        s.end = p.sk_iters * (cta0 + 1) / ncta;
    } else if (p.sk_split > 0) {
        s.rr_left = p.dp_per_cluster;
        if (cta0 < p.sk_split * p.sk_tiles) s.piece = cta0;
    } else {
        s.rr_left = cta0 < p.total_units ? (p.total_units - 1 - cta0) / ncta + 1 : 0;
    }
    return s;
}

// KS: K blocks per pipeline step; the split form's pieces start and end on
// whole steps (the last may end at an odd kblocks: its last step reads a
// partner block past the end of K, which loads zeros).
template <int CM, int KS = 1>
__device__ __forceinline__ bool work_next_raw(const TcParams& p, WorkIter& s, int ncta,
                                              uint32_t rank, Unit& w) {
    if (s.rr_left > 0) {
        w = decode_unit<CM>(p, s.unit_rr, rank);
        w.kind = UNIT_FULL;
        s.unit_rr += ncta;
        --s.rr_left;
        return true;
    }
    if (s.piece >= 0) {
        // split form: piece j of last-wave tile t covers the steps of KS K
        // blocks [j * steps / S, (j + 1) * steps / S); piece 0 finishes the tile
        const int S = p.sk_split;
        const int j = s.piece / p.sk_tiles;
        const int t = s.piece - j * p.sk_tiles;
        const int64_t steps = (p.kblocks + KS - 1) / KS;
        w = decode_unit<CM>(p, p.dp_units + t, rank);
        w.kb0 = KS * static_cast<int>(static_cast<int64_t>(j) * steps / S);
        const int kb1 = KS * static_cast<int>(static_cast<int64_t>(j + 1) * steps / S);
        w.kb1 = kb1 < p.kblocks ? kb1 : p.kblocks;
        if (p.sk_spread) {
            w.kind = UNIT_SPREAD;
            w.slot = t * S + j;
            w.nslots = S;
        } else {
            w.kind = j == 0 ? UNIT_HEAD : UNIT_TAIL;
            w.slot = t * (S - 1) + (j > 0 ? j - 1 : 0);
            w.nslots = S - 1;
        }
        w.piece = j;
        s.piece = -1;
        return true;
    }
    if (s.it >= s.end) return false;
    // contiguous form: the iterations are steps of KS K blocks, steps_u per unit
    const int64_t steps_u = (p.kblocks + KS - 1) / KS;
    const int64_t u_off = s.it / steps_u;
    const int st0 = static_cast<int>(s.it - u_off * steps_u);
    int64_t lim = (u_off + 1) * steps_u;
    if (lim > s.end) lim = s.end;
    w = decode_unit<CM>(p, static_cast<int>(p.dp_units + u_off), rank);
    w.kb0 = st0 * KS;
    const int kb1 = (st0 + static_cast<int>(lim - s.it)) * KS;
    w.kb1 = kb1 < p.kblocks ? kb1 : p.kblocks;
    w.kind = (w.kb0 == 0 && w.kb1 == p.kblocks) ? UNIT_FULL : (w.kb0 == 0 ? UNIT_HEAD : UNIT_TAIL);
    // A cluster's range starts with at most one piece that continues a unit
    // (a TAIL, published into the cluster's own slot) and ends with at most
    // one that another cluster continues (a HEAD).  The HEAD adds the
    // partials of the clusters that hold the rest of its unit, in order: the
    // next cluster through the one holding the unit's last step.
    if (w.kind == UNIT_TAIL) {
        w.slot = s.cluster;
        w.nslots = 1;
    } else if (w.kind == UNIT_HEAD) {
        const int64_t last = (u_off + 1) * steps_u - 1;  // the unit's last step
        int64_t c = last * ncta / p.sk_iters;             // first guess of its cluster
        while (c + 1 < ncta && p.sk_iters * (c + 1) / ncta <= last) ++c;
        while (c > 0 && p.sk_iters * c / ncta > last) --c;
        w.slot = s.cluster + 1;
        w.nslots = static_cast<int>(c) - s.cluster;
    }
    s.it = lim;
    return true;
}

// Debug build: the decoded unit lies inside the problem (batch entry, K
// slice, tile row and column, K blocks) and the stream-K slots it publishes
// into or reads from inside the workspace's slots.
template <int CM>
__device__ __forceinline__ bool unit_ok(const TcParams& p, const Unit& w) {
#if DG_DEBUG
    bool ok = w.b >= 0 && w.b < p.batch && w.split >= 0 && w.split < p.splits && w.pid_m >= 0 &&
              w.pid_m < p.num_pid_m * CM && w.pid_n >= 0 && w.pid_n < p.dbg_num_pid_n &&
              w.kb0 >= 0 && w.kb0 < w.kb1 && w.kb1 <= p.kblocks;
    if (w.kind != UNIT_FULL && !p.sk_atomic) {
        const int64_t lo = w.kind == UNIT_SPREAD ? w.slot - w.piece : w.slot;
        const int64_t hi = w.kind == UNIT_TAIL ? w.slot + 1 : lo + w.nslots;
        ok = ok && lo >= 0 && hi * CM <= p.dbg_sk_slots && (w.kind != UNIT_HEAD || w.nslots >= 1);
    }
    return DG_CHECK(ok, p.status, STATUS_CHECK_UNIT);
#else
    (void)p, (void)w;
    return true;
#endif
}

// The next work item of this cluster.  The debug build skips (and reports)
// a unit that fails unit_ok; every role of the CTA decodes the same units, so
// all of them skip it together.
template <int CM, int KS = 1>
__device__ __forceinline__ bool work_next(const TcParams& p, WorkIter& s, int ncta, uint32_t rank,
                                          Unit& w) {
#if DG_DEBUG
    while (work_next_raw<CM, KS>(p, s, ncta, rank, w))
        if (unit_ok<CM>(p, w)) return true;
    return false;
#else
    return work_next_raw<CM, KS>(p, s, ncta, rank, w);
#endif
}

__device__ __forceinline__ void st_release_u64(unsigned long long* ptr, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(ptr), "l"(v) : "memory");
}

// Fence with acquire and release semantics at GPU scope: after relaxed loads
// that observed released values, it makes the releasing threads' earlier
// writes visible to this thread.
__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* ptr) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}

// Bounded wait used while draining: ignores the abort flag.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

__device__ __forceinline__ void load_tile(const CUtensorMap* map, uint32_t dst, uint32_t bar, int x,
                                          int y, int z, bool is3d, uint64_t pol) {
    if (is3d)
        tma_load_3d(dst, map, bar, x, y, z, pol);
    else
        tma_load_2d(dst, map, bar, x, y, pol);
}

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float ld_f<__half>(const __half* p) { return __half2float(*p); }

template <typename T>
__device__ __forceinline__ void st_f(T* p, float x);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ void st_f<__half>(__half* p, float x) { *p = __float2half_rn(x); }

// Epilogue terms on a run of H values (each branch taken once per run, so
// unrequested terms never enter the unrolled loops).  cv: beta*C inputs,
// bias_v: per-value bias (already 0 where there is none).
template <int H>
__device__ __forceinline__ void finish_run(const Epilogue& e, float (&v)[H], const float (&cv)[H],
                                           const float (&bias_v)[H], bool has_c, bool has_bias) {
    if (e.alpha != 1.0f) {
#pragma unroll
        for (int i = 0; i < H; ++i) v[i] *= e.alpha;
    }
    if (has_c) {
#pragma unroll
        for (int i = 0; i < H; ++i) v[i] = fmaf(e.beta, cv[i], v[i]);
    }
    if (has_bias) {
#pragma unroll
        for (int i = 0; i < H; ++i) v[i] += bias_v[i];
    }
    act_inplace<H>(v, e.act);
}

// Debug build: the element at ptr lies inside C's span.
template <typename T>
__device__ __forceinline__ bool c_ptr_ok(const Epilogue& e, const T* ptr) {
    return c_span_ok(e, ptr - static_cast<const T*>(e.C));
}

// Row-major C: lane t owns column col0 + t of the warp's 32 rows, read from
// the staging tile.  All beta*C loads of a half-chunk are issued before any
// store (C is read and written in place, so the compiler may not reorder a
// load above an earlier store by itself).
template <int CH, typename T>
__device__ __forceinline__ void rows_out(const Epilogue& e, const Unit& w, int M, int N,
                                         int64_t row_base, int lane, int col0,
                                         const float* stage) {
    constexpr int H = 16;  // rows per half: bounds the registers held by in-flight loads
    const int col = col0 + lane;
    const bool col_ok = lane < CH && col < N;
    const int64_t left = M - row_base;
    const int nrows = left < 32 ? static_cast<int>(left) : 32;
    const int64_t ldc = e.ldc;
    const bool has_c = e.beta != 0.0f;
    const bool has_bias = e.bias != nullptr;
    const float bias_col =
        (has_bias && !e.bias_on_rows && col_ok && bias_ok(e, col)) ? e.bias[col] : 0.0f;
    T* const c0 =
        static_cast<T*>(e.C) + static_cast<int64_t>(w.b) * e.stride_c + row_base * ldc + col;
    if constexpr (CH == 32) {
        // an interior block (32 rows inside M, 32 columns inside N) with no
        // beta * C: no per-row tests, each half's values read from the staging
        // tile before any is stored (the same arithmetic as finish_run)
        if (nrows == 32 && col0 + 32 <= N && !has_c) {
            T* o = c0;
#pragma unroll 1
            for (int h = 0; h < 32; h += H) {
                float v[H];
#pragma unroll
                for (int i = 0; i < H; ++i) v[i] = stage[(h + i) * STAGE_LD + lane];
                if (e.alpha != 1.0f) {
#pragma unroll
                    for (int i = 0; i < H; ++i) v[i] *= e.alpha;
                }
                if (has_bias) {
                    if (e.bias_on_rows) {
#pragma unroll
                        for (int i = 0; i < H; ++i)
                            if (bias_ok(e, row_base + h + i)) v[i] += e.bias[row_base + h + i];
                    } else {
#pragma unroll
                        for (int i = 0; i < H; ++i) v[i] += bias_col;
                    }
                }
                act_inplace<H>(v, e.act);
#pragma unroll
                for (int i = 0; i < H; ++i, o += ldc) {
                    if (!c_ptr_ok(e, o)) continue;
                    st_f(o, v[i]);
                    count_write(e, w.b, row_base + h + i, col);
                }
            }
            return;
        }
    }
#pragma unroll 1
    for (int h = 0; h < 32; h += H) {
        float v[H], cv[H], bv[H];
        const T* q = c0 + h * ldc;
#pragma unroll
        for (int i = 0; i < H; ++i, q += ldc) {
            const bool ok = h + i < nrows && col_ok;
            cv[i] = (has_c && ok && c_ptr_ok(e, q)) ? ld_f(q) : 0.0f;
            v[i] = stage[(h + i) * STAGE_LD + lane];
            bv[i] = bias_col;
        }
        if (has_bias && e.bias_on_rows) {
#pragma unroll
            for (int i = 0; i < H; ++i)
                bv[i] = h + i < nrows && bias_ok(e, row_base + h + i) ? e.bias[row_base + h + i]
                                                                       : 0.0f;
        }
        finish_run<H>(e, v, cv, bv, has_c, has_bias);
        T* o = c0 + h * ldc;
#pragma unroll
        for (int i = 0; i < H; ++i, o += ldc)
            if (h + i < nrows && col_ok && c_ptr_ok(e, o)) {
                st_f(o, v[i]);
                count_write(e, w.b, row_base + h + i, col);
            }
    }
}

// Column-major C: lane t owns row row_base + t; for a fixed column the 32
// lanes address 32 consecutive elements, so the accesses are coalesced.
template <int CH, typename T>
__device__ __forceinline__ void cols_out(const Epilogue& e, const Unit& w, int M, int N,
                                         int64_t row_base, int lane, int col0,
                                         const uint32_t (&r)[32]) {
    constexpr int H = CH < 16 ? CH : 16;
    const int64_t row = row_base + lane;
    if (row >= M) return;
    const int left = N - col0;
    const int ncols = left < CH ? left : CH;
    const int64_t ldc = e.ldc;
    const bool has_c = e.beta != 0.0f;
    const bool has_bias = e.bias != nullptr;
    const float bias_row = (has_bias && e.bias_on_rows && bias_ok(e, row)) ? e.bias[row] : 0.0f;
    T* const c0 = static_cast<T*>(e.C) + static_cast<int64_t>(w.b) * e.stride_c +
                  static_cast<int64_t>(col0) * ldc + row;
#pragma unroll
    for (int h = 0; h < CH; h += H) {
        float v[H], cv[H], bv[H];
        const T* q = c0 + h * ldc;
#pragma unroll
        for (int i = 0; i < H; ++i, q += ldc) {
            const bool ok = h + i < ncols;
            cv[i] = (has_c && ok && c_ptr_ok(e, q)) ? ld_f(q) : 0.0f;
            v[i] = __uint_as_float(r[h + i]);
            bv[i] = bias_row;
        }
        if (has_bias && !e.bias_on_rows) {
#pragma unroll
            for (int i = 0; i < H; ++i)
                bv[i] = h + i < ncols && bias_ok(e, col0 + h + i) ? e.bias[col0 + h + i] : 0.0f;
        }
        finish_run<H>(e, v, cv, bv, has_c, has_bias);
        T* o = c0 + h * ldc;
#pragma unroll
        for (int i = 0; i < H; ++i, o += ldc)
            if (h + i < ncols && c_ptr_ok(e, o)) {
                st_f(o, v[i]);
                count_write(e, w.b, row, col0 + h + i);
            }
    }
}

// CTA-pair load: bytes complete on `bar`, which may be the peer's barrier.
__device__ __forceinline__ void load_pair(const CUtensorMap* map, uint32_t dst, uint32_t bar, int x,
                                          int y, int z, bool is3d, uint64_t pol) {
    if (is3d)
        tma_load_3d_pair(dst, map, bar, x, y, z, pol);
    else
        tma_load_2d_pair(dst, map, bar, x, y, pol);
}

// Debug build: element `at` of the split-K partials exists.
__device__ __forceinline__ bool partial_ok(const TcParams& p, const float* at) {
#if DG_DEBUG
    const int64_t k = at - p.partials;
    return DG_CHECK(k >= 0 && k < p.dbg_partials_elems, p.status, STATUS_CHECK_BOUNDS);
#else
    (void)p, (void)at;
    return true;
#endif
}

// Lane t's CH accumulator columns into row t of the staging tile (16-byte
// stores; the tile is 16-byte aligned and STAGE_LD a multiple of 4).
template <int CH>
__device__ __forceinline__ void stage_row(float* stage, int lane, const uint32_t (&r)[32]) {
    static_assert(CH % 4 == 0, "whole 16-byte stores");
    float4* dst = reinterpret_cast<float4*>(stage + lane * STAGE_LD);
#pragma unroll
    for (int c = 0; c < CH; c += 4)
        dst[c / 4] = make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                 __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
}

// Epilogue of one CH-column chunk of this warp's 32 rows.  On entry lane t
// holds row row_base + t, columns col0 .. col0+CH-1 (fp32 accumulators).
template <int CH>
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const Unit& w, int64_t row_base,
                                               int lane, int col0, const uint32_t (&r)[32],
                                               float* stage) {
    const Epilogue& e = p.epi;
    if (row_base >= p.M) return;
    if (p.partials) {
        // raw fp32 partial tile, stored densely in C's layout
        const int64_t slice = static_cast<int64_t>(w.split) * p.batch + w.b;
        float* P = p.partials + slice * static_cast<int64_t>(p.M) * p.N;
        if (!e.c_row_major) {
            const int64_t row = row_base + lane;
            if (row >= p.M) return;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                float* at = P + static_cast<int64_t>(col0 + c) * p.M + row;
                if (col0 + c < p.N && partial_ok(p, at)) *at = __uint_as_float(r[c]);
            }
            return;
        }
        stage_row<CH>(stage, lane, r);
        __syncwarp();
        const int col = col0 + lane;
        if (lane < CH && col < p.N) {
#pragma unroll 8
            for (int rr = 0; rr < 32; ++rr) {
                const int64_t row = row_base + rr;
                if (row < p.M && partial_ok(p, P + row * p.N + col))
                    P[row * p.N + col] = stage[rr * STAGE_LD + lane];
            }
        }
        __syncwarp();
        return;
    }
    if (!e.c_row_major) {
        if (e.c_dtype == DT_BF16)
            cols_out<CH, __nv_bfloat16>(e, w, p.M, p.N, row_base, lane, col0, r);
        else if (e.c_dtype == DT_F16)
            cols_out<CH, __half>(e, w, p.M, p.N, row_base, lane, col0, r);
        else
            cols_out<CH, float>(e, w, p.M, p.N, row_base, lane, col0, r);
        return;
    }
    // row-major output: transpose through shared memory so that each warp
    // store covers consecutive columns of one row.
    stage_row<CH>(stage, lane, r);
    __syncwarp();
    if (e.c_dtype == DT_BF16)
        rows_out<CH, __nv_bfloat16>(e, w, p.M, p.N, row_base, lane, col0, stage);
    else if (e.c_dtype == DT_F16)
        rows_out<CH, __half>(e, w, p.M, p.N, row_base, lane, col0, stage);
    else
        rows_out<CH, float>(e, w, p.M, p.N, row_base, lane, col0, stage);
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack2_out(int dt, float lo, float hi) {
    if (dt == DT_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack2_in(int dt, uint32_t u) {
    if (dt == DT_BF16) return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
}

// Stream-K fix-up: add the other cluster's fp32 partial of this warp's 32 rows
// into the accumulator in tensor memory, before the ordinary output pass.
// The partial is lane-interleaved (float4 k of lane l at k * 32 + l), so each
// load instruction of the warp reads 512 contiguous bytes; the loads of chunk
// c + 1 are in flight while chunk c is added.
template <int BN, int CHUNK>
__device__ __forceinline__ void add_partial_to_tmem(uint32_t tmem_row, const float* slab,
                                                    int lane) {
    constexpr int NV = CHUNK / 4;
    const float4* a4 = reinterpret_cast<const float4*>(slab) + lane;
    float4 cur[NV], nxt[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) cur[j] = __ldcg(a4 + j * 32);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += CHUNK) {
        if (c0 + CHUNK < BN) {
#pragma unroll
            for (int j = 0; j < NV; ++j) nxt[j] = __ldcg(a4 + ((c0 + CHUNK) / 4 + j) * 32);
        }
        uint32_t r[32];
        const uint32_t taddr = tmem_row + static_cast<uint32_t>(c0);
        if constexpr (CHUNK == 32)
            tmem_ld_x32(taddr, r);
        else
            tmem_ld_x16(taddr, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            r[4 * j + 0] = __float_as_uint(__uint_as_float(r[4 * j + 0]) + cur[j].x);
            r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + cur[j].y);
            r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + cur[j].z);
            r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + cur[j].w);
        }
        if constexpr (CHUNK == 32)
            tmem_st_x32(taddr, r);
        else
            tmem_st_x16(taddr, r);
#pragma unroll
        for (int j = 0; j < NV; ++j) cur[j] = nxt[j];
    }
    tmem_st_wait();
}

// Split form with a spread reduction: every piece of the tile has published
// its fp32 partial (lane-interleaved per warp, as above); piece j now sums
// share j of the tile's TILE4 float4 positions over the S partials and writes
// those outputs through the element-wise epilogue.  The share is one
// contiguous range of every partial, so:
//  1. one epilogue warp polls the flags of the publishing warps whose rows the
//     share covers (relaxed loads, each lane a set of flags, all in flight),
//     then fences (the acquire half of the publishers' release stores) and
//     issues one bulk copy per partial, each bringing that partial's share
//     into the stage memory the main loop has finished with;
//  2. the four epilogue warps wait for the copies on the gather barrier and
//     sum position by position in piece order (deterministic), then store
//     four outputs at a time.
// Returns false on a timeout (the status word is set).  The warp that issued
// the copies does not return before they have landed (a second bounded wait).
template <int BN, int CM>
__device__ __forceinline__ bool spread_reduce(const TcParams& p, int b, int pid_m, int pid_n,
                                           int slot0, int piece, int S, uint32_t rank, int q,
                                           int lane, volatile int* abort_flag, uint32_t gather,
                                           const float4* gather_ptr, uint32_t gather_cap,
                                           uint32_t gather_bar) {
    constexpr int QUARTER4 = 32 * BN / 4;  // float4 positions of one warp's 32 rows
    constexpr int TILE4 = 4 * QUARTER4;
    const int e0 = static_cast<int>(static_cast<int64_t>(piece) * TILE4 / S);
    const int e1 = static_cast<int>(static_cast<int64_t>(piece + 1) * TILE4 / S);
    const int npos = e1 - e0;
    if (npos <= 0) return true;
    const uint32_t bytes = static_cast<uint32_t>(npos) * 16u;
    if (static_cast<uint64_t>(bytes) * S > gather_cap) {
        // (cannot happen: every tile width's stage memory holds a whole tile
        // plus one float4 per piece)
        if (lane == 0 && p.status) DG_SET_TIMEOUT(p.status);
        return false;
    }
    bool issued = false;
    if (q == 0) {
        const int q0 = e0 / QUARTER4;
        const int nq = (e1 - 1) / QUARTER4 - q0 + 1;
        const unsigned long long* flags = p.sk_flags + (static_cast<int64_t>(slot0) * CM + rank) * 4;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
            // up to eight flags per lane are loaded before any is compared, so
            // that their loads are in flight together
            bool mine = true;
            for (int f0 = 0; f0 < S * nq; f0 += 256) {
                unsigned long long v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int f = f0 + 32 * u + lane;
                    const int s = f / nq;
                    const int qq = q0 + (f - s * nq);
                    v[u] = f < S * nq
                               ? ld_relaxed_u64(flags + static_cast<int64_t>(s) * CM * 4 + qq)
                               : p.sk_epoch;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) mine = mine && v[u] == p.sk_epoch;
            }
            if (__all_sync(0xffffffffu, mine)) break;
            int give_up = 0;
            if (lane == 0 && (it & 15u) == 0 &&
                (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns)) {
                *abort_flag = 1;
                if (p.status) DG_SET_TIMEOUT(p.status);
                give_up = 1;
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
        fence_acq_rel_gpu();
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(gather_bar, bytes * static_cast<uint32_t>(S));
        __syncwarp();
        const float4* src = reinterpret_cast<const float4*>(p.sk_partials) +
                            (static_cast<int64_t>(slot0) * CM + rank) * TILE4 + e0;
        const int64_t sstride = static_cast<int64_t>(CM) * TILE4;  // float4 from one piece's slot to the next
        for (int s = lane; s < S; s += 32)
            bulk_load(gather + static_cast<uint32_t>(s) * bytes, src + s * sstride, bytes, gather_bar);
        issued = true;
    }
    bool ok = mbar_wait(gather_bar, 0u, abort_flag, p.status, p.timeout_ns);
    if (issued && !ok) {
        // the copies read valid memory and finish on their own: wait (bounded
        // again) until they have landed before this CTA may leave
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(gather_bar, 0u) && globaltimer_ns() - t0 < p.timeout_ns) {
        }
    }
    if (!__all_sync(0xffffffffu, ok)) return false;
#pragma unroll 1
    for (int k = q * 32 + lane; k < npos; k += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int s = 0; s < S; ++s) {
            const float4 v = gather_ptr[s * npos + k];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        // position e: row (e / QUARTER4) * 32 + e % 32, columns 4 * ((e % QUARTER4) / 32) + 0..3
        const int e = e0 + k;
        const int qq = e / QUARTER4;
        const int f = e - qq * QUARTER4;
        const int64_t i = static_cast<int64_t>(pid_m) * TC_BLOCK_M + qq * 32 + (f & 31);
        const int64_t j = static_cast<int64_t>(pid_n) * BN + 4 * (f >> 5);
        if (i < p.M && j < p.N) epilogue_store4(p.epi, b, i, j, p.N, acc);
    }
    return true;
}

// Debug build: a TMA box store or load of the output starts at a column, row
// and depth inside it (the unit clips the far edges, but a store must never
// start at a negative coordinate).
__device__ __forceinline__ bool out_box_ok(const TcParams& p, int x, int y, int z) {
#if DG_DEBUG
    const int depth = p.partials ? p.splits * p.batch : p.batch;
    return DG_CHECK(x >= 0 && x < p.N && y >= 0 && z >= 0 && z < depth, p.status,
                    STATUS_CHECK_BOUNDS);
#else
    (void)p, (void)x, (void)y, (void)z;
    return true;
#endif
}

// Debug build, count-writes mode: the final values of row `row`, columns
// col0 .. col0 + ncols - 1 (those inside the output) were written.
__device__ __forceinline__ void count_row(const TcParams& p, int b, int64_t row, int col0,
                                          int ncols) {
#if DG_DEBUG
    if (p.epi.dbg_counts && !p.partials && row < p.M)
        for (int c = 0; c < ncols && col0 + c < p.N; ++c) count_write(p.epi, b, row, col0 + c);
#else
    (void)p, (void)b, (void)row, (void)col0, (void)ncols;
#endif
}

// TMA-store epilogue of one tile for this warp's 32 rows.  The tile is cut
// into chunks of 32 columns.  Per chunk, lane t turns row t's accumulators
// into output values (alpha, beta*C, bias, GELU, one rounding; or raw fp32
// for split-K partials) and writes them as row t of a 32-row box in shared
// memory, laid out as the tensor map's swizzle expects (rows of RB = 32*ES
// bytes; 128-byte swizzle for fp32, 64-byte swizzle for 16-bit outputs);
// lane 0 then stores the box with one TMA tensor store.  The TMA unit clips
// rows >= M and columns >= N.  Two boxes per warp alternate, so the math of
// a chunk overlaps the store of the previous one.
template <int BN, int ES>
__device__ __forceinline__ void tile_out_tma(const TcParams& p, const Unit& w, int q, int lane,
                                             uint32_t tmem_row, uint8_t* wbuf, uint32_t& nbox,
                                             uint64_t pol) {
    constexpr int EB = 32;             // columns per chunk
    constexpr int RB = EB * ES;        // bytes per box row: 128 (fp32) or 64 (16-bit)
    constexpr int NJ = RB / 16;        // 16-byte pieces per row
    constexpr int NW = RB / 4;         // 32-bit words per row
    const Epilogue& e = p.epi;
    const bool partial = p.partials != nullptr;
    const int dt = partial ? DT_F32 : e.c_dtype;
    const int row0 = w.pid_m * BM + q * 32;
    const int64_t row = static_cast<int64_t>(row0) + lane;
    const bool row_ok = row < p.M;
    const int zc = partial ? w.split * p.batch + w.b : w.b;
    // swizzle: piece j of row r sits at piece j ^ ((r * RB / 128) % NJ)
    const int swz = ((lane * RB) >> 7) & (NJ - 1);
    const bool need_c = !partial && e.beta != 0.0f && row_ok;
    const char* crow =
        need_c ? static_cast<const char*>(e.C) + (static_cast<int64_t>(w.b) * e.stride_c + row * e.ldc) * ES
               : nullptr;
    // beta*C of this thread's row segment for one chunk, as raw output words
    auto load_c = [&](int col0, uint32_t (&craw)[NW]) {
        const int64_t off = static_cast<int64_t>(w.b) * e.stride_c + row * e.ldc + col0;
        const int n = p.N - col0 < EB ? p.N - col0 : EB;
        if (!c_span_ok(e, off, n) ||
            !DG_CHECK(col0 + EB > p.N || (reinterpret_cast<uintptr_t>(crow + col0 * ES) & 15) == 0,
                      e.dbg_status, STATUS_CHECK_ALIGN)) {
#pragma unroll
            for (int i = 0; i < NW; ++i) craw[i] = 0u;
            return;
        }
        if (col0 + EB <= p.N) {
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const uint4 t = reinterpret_cast<const uint4*>(crow + static_cast<int64_t>(col0) * ES)[j];
                craw[4 * j + 0] = t.x;
                craw[4 * j + 1] = t.y;
                craw[4 * j + 2] = t.z;
                craw[4 * j + 3] = t.w;
            }
        } else {
            const char* src = crow + static_cast<int64_t>(col0) * ES;
            const int nvalid = p.N - col0;
#pragma unroll
            for (int i = 0; i < NW; ++i) craw[i] = 0u;
#pragma unroll
            for (int i = 0; i < EB; ++i) {
                if (i < nvalid) {
                    if (ES == 4) {
                        craw[i] = reinterpret_cast<const uint32_t*>(src)[i];
                    } else {
                        const uint32_t h = reinterpret_cast<const uint16_t*>(src)[i];
                        craw[i >> 1] |= (i & 1) ? (h << 16) : h;
                    }
                }
            }
        }
    };
    // the loads for chunk c+1 are issued before chunk c is computed
    uint32_t craw[NW], craw_next[NW];
    if (need_c) load_c(w.pid_n * BN, craw_next);

#pragma unroll 1
    for (int c = 0; c < BN / EB; ++c) {
        const int col0 = w.pid_n * BN + c * EB;
        if (col0 >= p.N) break;
        const bool full = col0 + EB <= p.N;
        if (need_c) {
#pragma unroll
            for (int i = 0; i < NW; ++i) craw[i] = craw_next[i];
            if (c + 1 < BN / EB && col0 + EB < p.N) load_c(col0 + EB, craw_next);
        }
        // accumulators: 32 consecutive TMEM columns of this lane's row
        uint32_t r[32];
        tmem_ld_x32(tmem_row + static_cast<uint32_t>(c * EB), r);
        tmem_ld_wait(r);
        float v[EB];
#pragma unroll
        for (int i = 0; i < EB; ++i) v[i] = __uint_as_float(r[i]);
        if (!partial) {
            // one pass per epilogue term, each branch taken once per chunk
            if (e.alpha != 1.0f) {
#pragma unroll
                for (int i = 0; i < EB; ++i) v[i] *= e.alpha;
            }
            if (need_c) {
#pragma unroll
                for (int i = 0; i < EB; ++i) {
                    float cval;
                    if (ES == 4) {
                        cval = __uint_as_float(craw[i]);
                    } else {
                        const float2 f = unpack2_in(dt, craw[i >> 1]);
                        cval = (i & 1) ? f.y : f.x;
                    }
                    v[i] = fmaf(e.beta, cval, v[i]);
                }
            }
            if (e.bias) {
                if (e.bias_on_rows) {
                    const float bias_row = row_ok && bias_ok(e, row) ? e.bias[row] : 0.0f;
#pragma unroll
                    for (int i = 0; i < EB; ++i) v[i] += bias_row;
                } else if (full) {
                    if (bias_ok(e, col0 + EB - 1)) {
#pragma unroll
                        for (int i = 0; i < EB; ++i) v[i] += __ldg(e.bias + col0 + i);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < EB; ++i)
                        if (col0 + i < p.N && bias_ok(e, col0 + i)) v[i] += __ldg(e.bias + col0 + i);
                }
            }
            act_inplace<EB>(v, e.act);
        }
        // the box written two chunks ago must have been read by its TMA store
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* box = wbuf + (nbox & 1u) * EPI_BOX_BYTES;
        uint8_t* line = box + lane * RB;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            uint4 t;
            if (ES == 4) {
                t = make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                               __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
            } else {
                t.x = pack2_out(dt, v[8 * j + 0], v[8 * j + 1]);
                t.y = pack2_out(dt, v[8 * j + 2], v[8 * j + 3]);
                t.z = pack2_out(dt, v[8 * j + 4], v[8 * j + 5]);
                t.w = pack2_out(dt, v[8 * j + 6], v[8 * j + 7]);
            }
            *reinterpret_cast<uint4*>(line + ((j ^ swz) << 4)) = t;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (out_box_ok(p, col0, row0, zc)) {
                if (p.c_tma_3d)
                    tma_store_3d(&p.tmap_c, smem_u32(box), col0, row0, zc, pol);
                else
                    tma_store_2d(&p.tmap_c, smem_u32(box), col0, row0, pol);
            }
            bulk_commit_group();
        }
        count_row(p, w.b, row, col0, EB);
        ++nbox;
    }
}

// The C ring of one epilogue warp (epilogue form 2): two 4 KB boxes that TMA
// loads fill with 32 rows x 64 columns of a 16-bit C (the output's own tensor
// map and swizzle), each completing on its own mbarrier.  Every lane keeps the
// counts of boxes requested and consumed; lane 0 issues the loads.  A tile's
// first two boxes are requested before its accumulator is waited for, each
// later one when the box two steps before it has been read.
struct CRing {
    uint8_t* box;     // this warp's first box
    uint32_t bar;     // this warp's first barrier
    uint32_t issued;  // boxes requested
    uint32_t used;    // boxes consumed
};

// Requests the C box of 64-column step c of unit w, for this warp's 32 rows.
template <int BN>
__device__ __forceinline__ void c_ring_issue(const TcParams& p, const Unit& w, int q, int lane,
                                             CRing& cr, int c) {
    const uint32_t slot = cr.issued & 1u;
    if (lane == 0) {
        const uint32_t dst = smem_u32(cr.box + slot * EPI_BOX_BYTES);
        const uint32_t bar = cr.bar + 8u * slot;
        const int x = w.pid_n * BN + c * 64;
        const int y = w.pid_m * BM + q * 32;
        // the box's previous contents were read by this warp (generic proxy)
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, EPI_BOX_BYTES);
        if (p.c_tma_3d)
            tma_load_3d(dst, &p.tmap_c, bar, x, y, w.b, l2_policy_evict_first());
        else
            tma_load_2d(dst, &p.tmap_c, bar, x, y, l2_policy_evict_first());
    }
    ++cr.issued;
}

// 64-column steps of unit w that lie (at least partly) inside N.
template <int BN>
__device__ __forceinline__ int fast_steps(const TcParams& p, const Unit& w) {
    const int left = p.N - w.pid_n * BN;
    const int n = (left + 63) / 64;
    return n < BN / 64 ? n : BN / 64;
}

// Waits (bounded, ignoring an abort) until every requested C box has landed,
// so that no TMA load is still writing this CTA's shared memory when it exits.
__device__ __forceinline__ void c_ring_drain(CRing& cr, int lane, uint64_t timeout_ns) {
    if (lane == 0) {
        for (; cr.used < cr.issued; ++cr.used) {
            const uint32_t slot = cr.used & 1u;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(cr.bar + 8u * slot, (cr.used >> 1) & 1u) &&
                   globaltimer_ns() - t0 < timeout_ns) {
            }
        }
    }
    __syncwarp();
}

// Atomic split-K: this CTA's share of C's memory rows (rows of a row-major C,
// columns of a column-major one; all batch entries as one range) set to
// beta * C + bias by its four epilogue warps (warp q takes every fourth memory
// row, lanes 16-byte groups along it), then the share's flag is published with
// the launch's epoch.  In the debug build's count-writes mode this is the one
// counted write of each element.
__device__ __forceinline__ void atomic_init_c(const TcParams& p, int cta, int ncta, int q,
                                              int lane) {
    const Epilogue& e = p.epi;
    const bool cm = !e.c_row_major;
    const int64_t outer = cm ? p.N : p.M;  // memory rows
    const int inner = cm ? p.M : p.N;      // elements along one
    // the bias runs along a memory row, or is one value per memory row
    const bool bias_inner = e.bias && (cm ? e.bias_on_rows : !e.bias_on_rows);
    const int64_t rows = static_cast<int64_t>(p.batch) * outer;
    const int64_t r0 = rows * cta / ncta, r1 = rows * (cta + 1) / ncta;
    const int n4 = inner / 4;
    for (int64_t r = r0 + q; r < r1; r += 4) {
        const int64_t b = r / outer, o = r - b * outer;
        float* row = static_cast<float*>(e.C) + b * e.stride_c + o * e.ldc;
        const float brow = e.bias && !bias_inner && bias_ok(e, o) ? e.bias[o] : 0.0f;
        for (int j4 = lane; j4 < n4; j4 += 32) {
            if (!c_span_ok(e, b * e.stride_c + o * e.ldc + 4 * j4, 4)) continue;
            float4 v = make_float4(brow, brow, brow, brow);
            if (e.beta != 0.0f) {
                const float4 c = reinterpret_cast<const float4*>(row)[j4];
                v.x = fmaf(e.beta, c.x, v.x), v.y = fmaf(e.beta, c.y, v.y);
                v.z = fmaf(e.beta, c.z, v.z), v.w = fmaf(e.beta, c.w, v.w);
            }
            if (bias_inner && bias_ok(e, 4 * j4 + 3)) {
                v.x += e.bias[4 * j4], v.y += e.bias[4 * j4 + 1];
                v.z += e.bias[4 * j4 + 2], v.w += e.bias[4 * j4 + 3];
            }
            reinterpret_cast<float4*>(row)[j4] = v;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                count_write(e, b, cm ? 4 * j4 + k : o, cm ? o : 4 * j4 + k);
        }
        for (int j = 4 * n4 + lane; j < inner; j += 32) {
            if (!c_span_ok(e, b * e.stride_c + o * e.ldc + j)) continue;
            float v = brow;
            if (e.beta != 0.0f) v = fmaf(e.beta, row[j], v);
            if (bias_inner && bias_ok(e, j)) v += e.bias[j];
            row[j] = v;
            count_write(e, b, cm ? j : o, cm ? o : j);
        }
    }
    // every epilogue thread's stores, then one release of the share's flag
    __threadfence();
    asm volatile("bar.sync 1, %0;" ::"n"(TC_EPI_THREADS) : "memory");
    if (q == 0 && lane == 0) st_release_u64(p.sk_flags + cta, p.sk_epoch);
}

// Atomic split-K: waits (bounded) until every CTA has published its share of
// C's initial values; then TMA reduce-adds of this warp may follow.  Returns
// false on a timeout (the status word is set).
__device__ __forceinline__ bool atomic_wait_init(const TcParams& p, int ncta, int lane,
                                                 volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        // every flag load of the lane in flight at once (no short-circuit)
        bool mine = true;
        for (int c = lane; c < ncta; c += 32) mine &= ld_relaxed_u64(p.sk_flags + c) == p.sk_epoch;
        if (__all_sync(0xffffffffu, mine)) break;
        int give_up = 0;
        if (lane == 0 && (it & 15u) == 0 && (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns)) {
            *abort_flag = 1;
            if (p.status) DG_SET_TIMEOUT(p.status);
            give_up = 1;
        }
        if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
    // the relaxed loads saw the released flags: acquire, then order the other
    // CTAs' generic stores before this warp's async-proxy reduce-adds
    fence_acq_rel_gpu();
    fence_proxy_async_global();
    __syncwarp();
    return true;
}

// Atomic split-K with a column-major C (a swapped skinny product): the warp's
// 32 rows x BN columns of alpha * accumulator go into one box laid out as C is
// (BN columns of 32 contiguous rows, 128 bytes each), which one TMA reduce-add
// adds into C through the output map (boxes of 32 rows x BN columns; the TMA
// unit skips rows and columns outside C).
template <int BN>
__device__ __forceinline__ void tile_reduce_cols(const TcParams& p, const Unit& w, int q, int lane,
                                                 uint32_t tmem_row, uint8_t* wbuf) {
    static_assert(BN <= 64, "a box of 32 x BN floats fits the warp's 8 KB");
    constexpr int CH = BN < 32 ? BN : 32;
    const int row0 = w.pid_m * BM + q * 32;
    float* box = reinterpret_cast<float*>(wbuf);
    // this warp's previous reduce-add has read the box
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
#pragma unroll
    for (int c0 = 0; c0 < BN; c0 += CH) {
        uint32_t r[32];
        if constexpr (CH == 32)
            tmem_ld_x32(tmem_row + static_cast<uint32_t>(c0), r);
        else
            tmem_ld_x16(tmem_row + static_cast<uint32_t>(c0), r);
        tmem_ld_wait(r);
#pragma unroll
        for (int c = 0; c < CH; ++c) box[(c0 + c) * 32 + lane] = p.epi.alpha * __uint_as_float(r[c]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < p.M &&
        DG_CHECK(w.pid_n * BN < p.N && p.batch == 1, p.status, STATUS_CHECK_BOUNDS)) {
        tma_reduce_add_2d(&p.tmap_c, smem_u32(box), row0, w.pid_n * BN);
        bulk_commit_group();
    }
}

// Output of one warp's 32 rows for the common case (C written by TMA store,
// beta == 0 or a split-K partial): 64 columns per step, two tcgen05.ld in
// flight, one fence / warp sync / store issue per step.  Each step fills 128
// bytes of every row: one 64-column box for a 16-bit C, two 32-column boxes
// for fp32, 128-byte swizzled like the operand tiles (16-byte piece j of row
// r at j ^ (r % 8); the boxes are 1024-byte aligned).  With BETA (epilogue
// form 2, 16-bit C) each step also adds beta * C from the warp's C ring, whose
// boxes have the same swizzle.  Returns false when a C box never arrived.
//
// [c_lo, c_hi): the 64-column steps of the tile this warp writes (all of them,
// or one half when two warps share a lane quarter).  SINGLE (16-bit C): one
// output box per warp instead of two alternating ones.
template <int BN, int ES, bool BETA = false, bool SINGLE = false>
__device__ __forceinline__ bool tile_out_fast(const TcParams& p, const Unit& w, int q, int lane,
                                              uint32_t tmem_row, uint8_t* wbuf, uint32_t& nbox,
                                              uint64_t pol, CRing* cr = nullptr,
                                              volatile int* abort_flag = nullptr, int c_lo = 0,
                                              int c_hi = BN / 64) {
    static_assert(!SINGLE || ES == 2, "one box per step: 16-bit C");
    static_assert(BN % 64 == 0, "64-column steps");
    static_assert(!BETA || ES == 2, "beta * C by TMA loads for 16-bit outputs");
    constexpr int NB = ES == 4 ? 2 : 1;  // boxes per step
    constexpr int BOXC = 128 / ES;       // columns per box
    const Epilogue& e = p.epi;
    const bool partial = p.partials != nullptr;
    const int dt = partial ? DT_F32 : e.c_dtype;
    const int row0 = w.pid_m * BM + q * 32;
    const int64_t row = static_cast<int64_t>(row0) + lane;
    const bool row_ok = row < p.M;
    const int zc = partial ? w.split * p.batch + w.b : w.b;
    const int swz = lane & 7;
    const bool need_c = BETA && !partial && e.beta != 0.0f;
    // atomic split-K: add alpha * acc into C (initialised to beta * C + bias)
    const bool reduce = !BETA && ES == 4 && p.sk_atomic != 0;
    const int nsteps = fast_steps<BN>(p, w);
    const int c_end = nsteps < c_hi ? nsteps : c_hi;
#pragma unroll 1
    for (int c = c_lo; c < c_hi; ++c) {
        const int col0 = w.pid_n * BN + c * 64;
        if (col0 >= p.N) break;
        const bool full = col0 + 64 <= p.N;
        uint32_t ra[32], rb[32];
        tmem_ld_x32(tmem_row + static_cast<uint32_t>(c * 64), ra);
        tmem_ld_x32(tmem_row + static_cast<uint32_t>(c * 64 + 32), rb);
        tmem_ld_wait2(ra, rb);
        float v[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] = __uint_as_float(ra[i]);
            v[32 + i] = __uint_as_float(rb[i]);
        }
        if (reduce) {
            if (e.alpha != 1.0f) {
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] *= e.alpha;
            }
        } else if (!partial) {
            if (e.alpha != 1.0f) {
#pragma unroll
                for (int i = 0; i < 64; ++i) v[i] *= e.alpha;
            }
            if constexpr (BETA) {
                if (need_c) {
                    // this step's C box, requested two steps (or a tile) earlier
                    const uint32_t slot = cr->used & 1u;
                    int ok = 1;
                    if (lane == 0)
                        ok = mbar_wait(cr->bar + 8u * slot, (cr->used >> 1) & 1u, abort_flag,
                                       p.status, p.timeout_ns)
                                 ? 1
                                 : 0;
                    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
                    __syncwarp();
                    const uint8_t* cl = cr->box + slot * EPI_BOX_BYTES + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 t = *reinterpret_cast<const uint4*>(cl + ((j ^ swz) << 4));
                        const uint32_t wd[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = unpack2_in(dt, wd[k]);
                            v[8 * j + 2 * k] = fmaf(e.beta, f.x, v[8 * j + 2 * k]);
                            v[8 * j + 2 * k + 1] = fmaf(e.beta, f.y, v[8 * j + 2 * k + 1]);
                        }
                    }
                    ++cr->used;
                    __syncwarp();  // every lane has read the box before it is refilled
                    if (c + 2 < c_end) c_ring_issue<BN>(p, w, q, lane, *cr, c + 2);
                }
            }
            if (e.bias) {
                if (e.bias_on_rows) {
                    const float bias_row = row_ok && bias_ok(e, row) ? e.bias[row] : 0.0f;
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] += bias_row;
                } else if (full) {
                    if (bias_ok(e, col0 + 64 - 1)) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] += __ldg(e.bias + col0 + i);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (col0 + i < p.N && bias_ok(e, col0 + i)) v[i] += __ldg(e.bias + col0 + i);
                }
            }
            act_inplace<64>(v, e.act);
        }
        // the box(es) written before must have been read by their TMA stores:
        // 16-bit C alternates two boxes, fp32 fills both every step
        if (lane == 0) {
            if constexpr (NB == 2 || SINGLE)
                bulk_wait_group_read<0>();
            else
                bulk_wait_group_read<1>();
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            uint8_t* box = wbuf + (NB == 2 ? k : (SINGLE ? 0u : (nbox & 1u))) * EPI_BOX_BYTES;
            uint8_t* line = box + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                uint4 t;
                if constexpr (ES == 4) {
                    const float* f = v + k * 32 + 4 * j;
                    t = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                   __float_as_uint(f[2]), __float_as_uint(f[3]));
                } else {
                    const float* f = v + 8 * j;
                    t.x = pack2_out(dt, f[0], f[1]);
                    t.y = pack2_out(dt, f[2], f[3]);
                    t.z = pack2_out(dt, f[4], f[5]);
                    t.w = pack2_out(dt, f[6], f[7]);
                }
                *reinterpret_cast<uint4*>(line + ((j ^ swz) << 4)) = t;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const int bc = col0 + k * BOXC;
                if (bc >= p.N) break;
                const uint32_t box =
                    smem_u32(wbuf + (NB == 2 ? k : (SINGLE ? 0u : (nbox & 1u))) * EPI_BOX_BYTES);
                if (!out_box_ok(p, bc, row0, zc)) continue;
                if (reduce) {
                    if (p.c_tma_3d)
                        tma_reduce_add_3d(&p.tmap_c, box, bc, row0, zc);
                    else
                        tma_reduce_add_2d(&p.tmap_c, box, bc, row0);
                } else if (p.c_tma_3d) {
                    tma_store_3d(&p.tmap_c, box, bc, row0, zc, pol);
                } else {
                    tma_store_2d(&p.tmap_c, box, bc, row0, pol);
                }
            }
            bulk_commit_group();
        }
        if (!reduce) count_row(p, w.b, row, col0, 64);
        ++nbox;
    }
    return true;
}

// Pull this warp's rows of the C tile into L2 before the accumulator is ready
// (beta != 0 only), so that the epilogue's reads of C hit L2.
template <int BN>
__device__ __forceinline__ void prefetch_c_tile(const TcParams& p, const Unit& w, int64_t row) {
    const Epilogue& e = p.epi;
    if (e.beta == 0.0f || p.partials || !e.c_row_major || row >= p.M) return;
    const int col0 = w.pid_n * BN;
    const int ncols = p.N - col0 < BN ? p.N - col0 : BN;
    const int es = dt_size(e.c_dtype);
    const char* base = static_cast<const char*>(e.C) +
                       (static_cast<int64_t>(w.b) * e.stride_c + row * e.ldc + col0) * es;
    for (int off = 0; off < ncols * es; off += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + off));
}

template <int BN, int MODE, int EPI, int KS = 1>
__global__ void __launch_bounds__(Cfg<BN, MODE, EPI, KS>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<BN, MODE, EPI, KS>;
    constexpr int CM = C::CM;
    constexpr int CG = C::CG;
    const uint32_t rank = CM > 1 ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int cta0 = static_cast<int>(blockIdx.x) / CM;  // cluster index
    const int ncta = static_cast<int>(gridDim.x) / CM;   // clusters in the grid
    constexpr uint16_t kPair = (1u << CM) - 1u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sA0 = smem_u32(smem);
    const uint32_t sB0 = sA0 + C::STAGES * C::A_BYTES;
    // layout: [A stages][B stages][epilogue boxes (1024-aligned)][C ring (kind 2)][barriers]
    uint8_t* epi_smem = smem + C::STAGES * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + C::EPI_SMEM);
    const uint32_t bar0 = smem_u32(bars);
    // barrier slots: full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2], drain,
    // gather (the spread reduction's copies), C boxes [epilogue warps][2]
    const uint32_t full0 = bar0;
    const uint32_t empty0 = bar0 + 8u * C::STAGES;
    const uint32_t tfull0 = bar0 + 16u * C::STAGES;
    const uint32_t tempty0 = tfull0 + 16u;
    const uint32_t drain_bar = tempty0 + 16u;
    const uint32_t gather_bar = drain_bar + 8u;
    const uint32_t cbar0 = gather_bar + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 6 + 2 * C::EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // An MN-contiguous operand arrives in 64-wide atom columns of 64 * KS K
    // rows (128 bytes each, 128-byte swizzled): one column takes 8 KB * KS.
    constexpr uint32_t kAtomCol = 8192u * KS;

    if constexpr (C::KIND == 2 || (C::KIND == 0 && BN > 64)) {
        // the atomic split-K runs with the TMA-store epilogue, or with the
        // general one for a column-major C and tiles up to 64 wide (the plan
        // never asks otherwise); report instead of skipping work
        if (p.sk_atomic) {
            if (threadIdx.x == 0 && p.status) DG_SET_TIMEOUT(p.status);
            return;
        }
    }
    if constexpr (EPI >= 3) {
        // forms 3 and 4 take whole tiles only, form 3 with plain stores and form
        // 4 with TMA stores (the plan never asks otherwise); report instead of
        // skipping work
        if (p.sk_atomic || p.sk_iters > 0 || p.sk_split > 0 || p.sk_spread || p.partials ||
            (EPI == 3 ? p.c_tma != 0 : p.c_tma == 0)) {
            if (threadIdx.x == 0 && p.status) DG_SET_TIMEOUT(p.status);
            return;
        }
    }

    // The launch parameters outside the tensor maps lie in four 64-byte lines.
    // A role's first reads of them miss the constant cache one after another
    // along its dependent chain of decisions; one read per line, from four warps
    // at once during the prologue, takes those misses together instead.
    if (lane == 0) {
        if (warp == 2) asm volatile("" ::"r"(p.M));
        if (warp == 3) asm volatile("" ::"f"(p.epi.alpha));
        if (warp == 4) asm volatile("" ::"r"(p.c_tma));
        if (warp == 5) asm volatile("" ::"l"(p.sk_epoch));
    }

    // Debug build: the stage ring sits on 1024-byte boundaries (the 128-byte
    // swizzle atoms) and the barriers on 8-byte ones (recorded only: the
    // layout is fixed at compile time).
    if (threadIdx.x == 0)
        (void)DG_CHECK((sA0 & 1023u) == 0 && (sB0 & 1023u) == 0 && (bar0 & 7u) == 0 &&
                           (smem_u32(epi_smem) & 1023u) == 0,
                       p.status, STATUS_CHECK_ALIGN);

    if (threadIdx.x == 0) {
        // MODE 2: the leader's stage barrier collects the bytes of both CTAs'
        // loads; its accumulator-release barrier counts the epilogue warps of
        // both CTAs.  Accumulator releases are one arrival per epilogue warp.
        const uint32_t full_count = 1u;
        const uint32_t empty_count = 1u;
        const uint32_t tempty_count = MODE == 2 ? 2u * C::EPI_WARPS : C::EPI_WARPS;
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full0 + 8u * s, full_count);
            mbar_init(empty0 + 8u * s, empty_count);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8u * b, 1);
            mbar_init(tempty0 + 8u * b, tempty_count);
        }
        mbar_init(drain_bar, 1);
        mbar_init(gather_bar, 1);
        for (int b = 0; b < 2 * C::EPI_WARPS; ++b) mbar_init(cbar0 + 8u * b, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&p.tmap_a);
        prefetch_tmap(&p.tmap_b);
        if (p.c_tma || p.sk_atomic) prefetch_tmap(&p.tmap_c);
    }
    if (warp == 1) {
        tmem_alloc_cg<CG>(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_cg<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CM > 1)
        cluster_sync();  // the peer's barriers are initialised before any cross-CTA signal
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            // L2 policies of the two operands ("Skill: Write a Triton GEMM Kernel",
            // Kernel design rules: keep the operand reused across the tile group)
            const uint64_t pol_normal = l2_policy_evict_normal();
            const uint64_t pol_first = l2_policy_evict_first();
            const uint64_t pol_last = l2_policy_evict_last();
            const uint64_t pol_a = p.l2_hints == 1 ? pol_first : (p.l2_hints == 2 ? pol_last : pol_normal);
            const uint64_t pol_b = p.l2_hints == 1 ? pol_last : (p.l2_hints == 2 ? pol_first : pol_normal);
            // an operand copied by the launch before this one: every CTA waits
            // for the copy to complete (so this grid never completes before it)
            if (p.pdl) griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0;
            bool ok = true;
            WorkIter wi = work_begin(p, cta0, ncta);
            Unit w;
            while (ok && work_next<CM, KS>(p, wi, ncta, rank, w)) {
                for (int kb = w.kb0; kb < w.kb1; kb += KS) {
                    if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.status,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    if (p.test_stall == 1 && armed == 0) {
                        // test only: leave this stage unfilled; the MMA warp's bounded
                        // wait on it must expire and report the timeout.
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full0 + 8u * stage;
                    // MODE 2: the leader's barrier takes the bytes of both CTAs;
                    // the peer's barrier is unused.
                    if (MODE != 2 || leader)
                        mbar_arrive_expect_tx(fb, MODE == 2 ? 2u * C::STAGE_BYTES : C::STAGE_BYTES);
                    const uint32_t a_dst = sA0 + stage * C::A_BYTES;
                    const uint32_t b_dst = sB0 + stage * C::B_BYTES;
                    const int k0 = kb * BK;
                    if constexpr (MODE == 2) {
                        // own A rows and own BN/2 B columns; bytes complete on the leader
                        const uint32_t lb = leader ? fb : mapa_shared(fb, 0u);
                        if (!p.a_mn) {
                            if constexpr (KS == 2)  // K blocks kb and kb + 1 (past the end: zeros)
                                tma_load_3d_pair(a_dst, &p.tmap_a, lb, 0, w.pid_m * BM, kb, pol_a);
                            else
                                load_pair(&p.tmap_a, a_dst, lb, k0, w.pid_m * BM, w.b, p.a_3d, pol_a);
                        } else {
                            // 64-wide atom columns of 64 * KS K rows (rows past K: zeros)
#pragma unroll
                            for (int h = 0; h < BM / 64; ++h)
                                load_pair(&p.tmap_a, a_dst + h * kAtomCol, lb, w.pid_m * BM + 64 * h,
                                          k0, w.b, p.a_3d, pol_a);
                        }
                        // per N = SUB_N MMA, this CTA's half of its columns
                        constexpr int HALF = C::SUB_N / 2;
                        static_assert(KS == 1 || C::NSUB == 1, "two K blocks per load: one sub-MMA");
#pragma unroll
                        for (int sn = 0; sn < C::NSUB; ++sn) {
                            const uint32_t bs = b_dst + sn * (HALF * 128u);
                            const int n0 = w.pid_n * BN + sn * C::SUB_N + static_cast<int>(rank) * HALF;
                            if (!p.b_mn) {
                                if constexpr (KS == 2)
                                    tma_load_3d_pair(bs, &p.tmap_b, lb, 0, n0, kb, pol_b);
                                else
                                    load_pair(&p.tmap_b, bs, lb, k0, n0, w.b, p.b_3d, pol_b);
                            } else {
#pragma unroll
                                for (int hh = 0; hh < HALF / 64; ++hh)
                                    load_pair(&p.tmap_b, bs + hh * kAtomCol, lb, n0 + 64 * hh, k0,
                                              w.b, p.b_3d, pol_b);
                            }
                        }
                    } else if (!p.a_mn) {
                        if constexpr (KS == 2)  // K blocks kb and kb + 1 (past the end: zeros)
                            tma_load_3d(a_dst, &p.tmap_a, fb, 0, w.pid_m * BM, kb, pol_a);
                        else
                            load_tile(&p.tmap_a, a_dst, fb, k0, w.pid_m * BM, w.b, p.a_3d, pol_a);
                    } else {
#pragma unroll
                        for (int h = 0; h < BM / 64; ++h)
                            load_tile(&p.tmap_a, a_dst + h * kAtomCol, fb, w.pid_m * BM + 64 * h, k0,
                                      w.b, p.a_3d, pol_a);
                    }
                    if constexpr (MODE == 0) {
                        if (!p.b_mn) {
                            if constexpr (KS == 2)
                                tma_load_3d(b_dst, &p.tmap_b, fb, 0, w.pid_n * BN, kb, pol_b);
                            else
                                load_tile(&p.tmap_b, b_dst, fb, k0, w.pid_n * BN, w.b, p.b_3d, pol_b);
                        } else {
                            if constexpr (BN >= 64) {
#pragma unroll
                                for (int h = 0; h < BN / 64; ++h)
                                    load_tile(&p.tmap_b, b_dst + h * kAtomCol, fb,
                                              w.pid_n * BN + 64 * h, k0, w.b, p.b_3d, pol_b);
                            }
                        }
                    }
                    ++armed;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every issued fill must land before the CTA may exit.  A MODE 2
            // peer's loads complete on the leader's barriers: after a normal
            // run the leader has consumed them all before the final cluster
            // barrier; after an abort the peer gives its copies a fixed bound.
            if (MODE == 2 && !leader) {
                if (!ok) {
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 200000ull) {
                    }
                }
            } else {
                for (int s = 0; s < C::STAGES && static_cast<uint32_t>(s) < armed; ++s) {
                    const uint32_t fills = (armed - 1u - s) / C::STAGES + 1u;
                    wait_drain(full0 + 8u * s, (fills - 1u) & 1u, p.timeout_ns);
                }
            }
        }
    } else if (warp == 1) {
        if (MODE == 2 && !leader) {
            // MODE 2 peer: the leader's thread issues the MMAs for both CTAs
        } else if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int abuf = 0;
            uint32_t aphase = 0;
            bool issued = false;
            bool ok = true;
            // K step k (16 deep) of a stage.  K-major: 32 bytes per step inside
            // the 128-byte swizzle row, and with KS = 2 the second K block BM
            // (or B_ROWS) rows of 128 bytes after the first.  MN-major: two
            // 8-row (1024-byte) groups per step down one atom column of 64 * KS
            // K rows; the descriptor's leading byte offset is the distance
            // between atom columns.
            auto k_off = [](bool mn, int k, uint32_t rows) -> uint32_t {
                return mn ? static_cast<uint32_t>(k) * 2048u
                          : static_cast<uint32_t>(k / 4) * (rows * 128u) + static_cast<uint32_t>(k % 4) * 32u;
            };
            const bool a_mn = p.a_mn != 0, b_mn = p.b_mn != 0;
            const uint32_t a_lbo = a_mn ? kAtomCol : 16u;
            const uint32_t b_lbo = b_mn ? kAtomCol : 16u;
            WorkIter wi = work_begin(p, cta0, ncta);
            Unit w;
            while (ok && work_next<CM, KS>(p, wi, ncta, rank, w)) {
                if (!mbar_wait(tempty0 + 8u * abuf, aphase ^ 1u, abort_flag, p.status,
                               p.timeout_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(abuf * BN);
                for (int kb = w.kb0; kb < w.kb1; kb += KS) {
                    if (!mbar_wait(full0 + 8u * stage, phase, abort_flag, p.status,
                                   p.timeout_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_base = sA0 + stage * C::A_BYTES;
                    const uint32_t b_base = sB0 + stage * C::B_BYTES;
#pragma unroll
                    for (int k = 0; k < KS * BK / 16; ++k) {
                        const uint64_t ad =
                            smem_desc_sw128(a_base + k_off(a_mn, k, BM), a_lbo, 1024u);
#pragma unroll
                        for (int sn = 0; sn < C::NSUB; ++sn) {
                            // sub-tile sn: its B rows from (SUB_N / 2) * 128 bytes on, its
                            // accumulator SUB_N columns on (one 64-wide atom column is 8 KB
                            // for MN-major B, the same offset)
                            const uint32_t bsub = b_base + sn * (C::SUB_N / 2) * 128u;
                            const uint64_t bd =
                                smem_desc_sw128(bsub + k_off(b_mn, k, C::B_ROWS), b_lbo, 1024u);
                            umma_f16_cg<CG>(d_tmem + sn * C::SUB_N, ad, bd, p.idesc,
                                            (kb > w.kb0 || k > 0) ? 1u : 0u);
                        }
                    }
                    issued = true;
                    if constexpr (CM > 1)
                        umma_commit_mc_cg<CG>(empty0 + 8u * stage, kPair);
                    else
                        umma_commit_cg<CG>(empty0 + 8u * stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (MODE == 2)
                    umma_commit_mc_cg<CG>(tfull0 + 8u * abuf, kPair);  // both CTAs' accumulators
                else
                    umma_commit_cg<CG>(tfull0 + 8u * abuf);
                if (++abuf == C::ACC_BUFS) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            if (issued) {
                // all MMAs complete before tensor memory is released
                umma_commit_cg<CG>(drain_bar);
                wait_drain(drain_bar, 0u, p.timeout_ns);
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, or 2..9)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_field = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* wbuf = epi_smem + (warp - 2) * C::EPI_WARP;
        // forms 3, 4: the column half of each tile this warp writes; its
        // 64-column steps [step_lo, step_hi)
        const int col_half = (warp - 2) >> 2;
        const int step_lo = C::EPI_WARPS == 8 ? col_half * (BN / 128) : 0;
        const int step_hi = C::EPI_WARPS == 8 ? step_lo + BN / 128 : BN / 64;
        float* stage = reinterpret_cast<float*>(wbuf);
        uint32_t nbox = 0;
        // outputs leave L2 first; split-K partials stay for the reduction that follows
        const uint64_t store_pol = p.partials ? l2_policy_evict_last() : l2_policy_evict_first();
        int abuf = 0;
        uint32_t aphase = 0;
        // epilogue form 2: this warp's ring of C boxes and their barriers
        CRing cring{epi_smem + C::EPI_WARPS * C::EPI_WARP + (warp - 2) * C_RING_WARP_BYTES,
                    cbar0 + 16u * static_cast<uint32_t>(warp - 2), 0u, 0u};
        WorkIter wi = work_begin(p, cta0, ncta);
        Unit w;
        bool first = true;
        // atomic split-K: this CTA's share of C's initial values first (shares
        // and flags per CTA of the grid, pairs or not).  The wait for every
        // other CTA's share comes with the first accumulator: polling the flags
        // while the main loop runs (every CTA's epilogue warps on the same few
        // lines) measured 2 us slower on 256 x 256 x 65536.
        bool init_seen = false;
        if constexpr (EPI == 1 || (EPI == 0 && BN <= 64)) {
            if (p.sk_atomic)
                atomic_init_c(p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), q, lane);
        }
        while (work_next<CM, KS>(p, wi, ncta, rank, w)) {
            if constexpr (C::KIND == 2) {
                // the first two C boxes of a tile this warp will write, requested
                // before its accumulator is waited for
                if (p.epi.beta != 0.0f && (w.kind == UNIT_FULL || w.kind == UNIT_HEAD)) {
                    const int n = fast_steps<BN>(p, w);
                    const int end = n < step_hi ? n : step_hi;
                    for (int c = step_lo; c < step_lo + 2 && c < end; ++c)
                        c_ring_issue<BN>(p, w, q, lane, cring, c);
                }
            }
            if constexpr (C::KIND == 0 || C::KIND == 2) {
                // C tile of the next item into L2 (and of this one, the first time)
                if (first)
                    prefetch_c_tile<BN>(p, w, static_cast<int64_t>(w.pid_m) * BM + q * 32 + lane);
                first = false;
                WorkIter peek = wi;
                Unit wn;
                if (work_next<CM, KS>(p, peek, ncta, rank, wn))
                    prefetch_c_tile<BN>(p, wn, static_cast<int64_t>(wn.pid_m) * BM + q * 32 + lane);
            }
            int ok = 1;
            if (lane == 0)
                ok = mbar_wait(tfull0 + 8u * abuf, aphase, abort_flag, p.status, p.timeout_ns) ? 1
                                                                                               : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const int64_t row_base = static_cast<int64_t>(w.pid_m) * BM + q * 32;
            const int col_base = w.pid_n * BN;
            const uint32_t tmem_row = tmem_base + lane_field + static_cast<uint32_t>(abuf * BN);
            if constexpr (EPI == 3) {
                // form 3: whole tiles, plain stores; this warp's half of the
                // columns, 32 at a time
#pragma unroll 1
                for (int c0 = col_half * (BN / 2); c0 < (col_half + 1) * (BN / 2); c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_x32(tmem_row + static_cast<uint32_t>(c0), r);
                    tmem_ld_wait(r);
                    epilogue_chunk<32>(p, w, row_base, lane, col_base + c0, r, stage);
                }
            } else if (p.sk_atomic) {
                // atomic split-K (fp32 C, TMA reduce-adds): every piece adds
                // its share, once C's initial values are all in place
                if constexpr (EPI == 1 || (EPI == 0 && BN <= 64)) {
                    if (!init_seen) {
                        if (!atomic_wait_init(p, static_cast<int>(gridDim.x), lane, abort_flag))
                            break;
                        init_seen = true;
                    }
                    if constexpr (EPI == 1)
                        tile_out_fast<BN, 4>(p, w, q, lane, tmem_row, wbuf, nbox, store_pol);
                    else
                        tile_reduce_cols<BN>(p, w, q, lane, tmem_row, wbuf);
                }
            } else if (w.kind == UNIT_TAIL || w.kind == UNIT_SPREAD) {
                // stream-K tail or spread piece: publish this CTA's raw fp32 partial
                // for the cluster(s) that finish the tile
                const int64_t slot = static_cast<int64_t>(w.slot) * CM + rank;
                float4* dst = reinterpret_cast<float4*>(p.sk_partials + (slot * BM + q * 32) * BN) + lane;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += C::CHUNK) {
                    uint32_t r[32];
                    const uint32_t taddr = tmem_row + static_cast<uint32_t>(c0);
                    if constexpr (C::CHUNK == 32)
                        tmem_ld_x32(taddr, r);
                    else
                        tmem_ld_x16(taddr, r);
                    tmem_ld_wait(r);
#pragma unroll
                    for (int i = 0; i < C::CHUNK / 4; ++i)
                        __stcg(dst + (c0 / 4 + i) * 32,
                               make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                           __uint_as_float(r[4 * i + 2]),
                                           __uint_as_float(r[4 * i + 3])));
                }
                // the warp sync orders every lane's stores before lane 0's release
                // store of the flag, which makes them visible (cumulatively) to a
                // reader that acquires the flag
                __syncwarp();
                // (test only: with test_stall 2 the first CTA never publishes, so
                // the waits for its partial must expire and report a timeout)
                if (lane == 0 && !(p.test_stall == 2 && blockIdx.x == 0))
                    st_release_u64(p.sk_flags + slot * 4 + q, p.sk_epoch);
            } else {
                // stream-K head: wait (bounded) for each other piece's partial of
                // this tile and add it to the accumulator
                int got = 1;
                for (int ps = 0; w.kind == UNIT_HEAD && ps < w.nslots; ++ps) {
                    const int64_t slot = static_cast<int64_t>(w.slot + ps) * CM + rank;
                    if (lane == 0) {
                        const unsigned long long* flag = p.sk_flags + slot * 4 + q;
                        if (ld_acquire_u64(flag) != p.sk_epoch) {
                            const uint64_t t0 = globaltimer_ns();
                            for (uint32_t it = 1;; ++it) {
                                if (ld_acquire_u64(flag) == p.sk_epoch) break;
                                if ((it & 15u) == 0) {
                                    if (*abort_flag || globaltimer_ns() - t0 > p.timeout_ns) {
                                        *abort_flag = 1;
                                        if (p.status) DG_SET_TIMEOUT(p.status);
                                        got = 0;
                                        break;
                                    }
                                }
                            }
                        }
                    }
                    got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) break;
                    __syncwarp();  // lane 0's acquire orders the whole warp's reads below
                    add_partial_to_tmem<BN, C::CHUNK>(tmem_row, p.sk_partials + (slot * BM + q * 32) * BN,
                                                      lane);
                }
                if (!got) break;
                if constexpr (EPI == 1) {
                    if (p.partials != nullptr || p.epi.c_dtype == DT_F32)
                        tile_out_fast<BN, 4>(p, w, q, lane, tmem_row, wbuf, nbox, store_pol);
                    else
                        tile_out_fast<BN, 2>(p, w, q, lane, tmem_row, wbuf, nbox, store_pol);
                } else if constexpr (C::KIND == 2) {
                    // the plan takes this form for a 16-bit C only
                    if (!tile_out_fast<BN, 2, true, EPI == 4>(p, w, q, lane, tmem_row, wbuf, nbox,
                                                              store_pol, &cring, abort_flag,
                                                              step_lo, step_hi))
                        break;
                } else if (p.c_tma) {
                    if constexpr (BN >= 32) {
                        if (p.partials != nullptr || p.epi.c_dtype == DT_F32)
                            tile_out_tma<BN, 4>(p, w, q, lane, tmem_row, wbuf, nbox, store_pol);
                        else
                            tile_out_tma<BN, 2>(p, w, q, lane, tmem_row, wbuf, nbox, store_pol);
                    }
                } else {
#pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += C::CHUNK) {
                        uint32_t r[32];
                        const uint32_t taddr = tmem_row + static_cast<uint32_t>(c0);
                        if constexpr (C::CHUNK == 32)
                            tmem_ld_x32(taddr, r);
                        else
                            tmem_ld_x16(taddr, r);
                        tmem_ld_wait(r);
                        epilogue_chunk<C::CHUNK>(p, w, row_base, lane, col_base + c0, r, stage);
                    }
                }
            }
            // every lane's tensor-memory reads are ordered before the warp's
            // single release of the accumulator buffer
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (MODE == 2 && !leader)
                    mbar_arrive_remote(mapa_shared(tempty0 + 8u * abuf, 0u));
                else
                    mbar_arrive(tempty0 + 8u * abuf);
            }
            if (++abuf == C::ACC_BUFS) {
                abuf = 0;
                aphase ^= 1u;
            }
        }
        // a spread piece is its cluster's last work item: once it has been
        // published and the accumulator released, the share is reduced (the
        // piece is found again from the cluster index, so nothing stays live
        // across the loop).  The plan runs the spread form with single-CTA
        // tiles only.
        if constexpr (MODE == 0 && EPI < 3) {
            if (p.sk_spread && !*abort_flag) {
                WorkIter sw = work_begin(p, cta0, ncta);
                sw.rr_left = 0;
                Unit u;
                if (sw.piece >= 0 && work_next<CM, KS>(p, sw, ncta, rank, u))
                    spread_reduce<BN, CM>(p, u.b, u.pid_m, u.pid_n, u.slot - u.piece, u.piece,
                                          u.nslots, rank, q, lane, abort_flag, sA0,
                                          reinterpret_cast<const float4*>(smem),
                                          C::STAGES * C::STAGE_BYTES, gather_bar);
            }
        }
        // the TMA stores must finish, and no C box may still be loading, before
        // the CTA exits
        if constexpr (C::KIND == 2) c_ring_drain(cring, lane, p.timeout_ns);
        if (lane == 0) bulk_wait_group_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if constexpr (CM > 1)
        cluster_sync();  // no CTA leaves while its peer may still touch its shared or tensor memory
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_cg<CG>(tmem_base, C::TMEM_COLS);
    }
}

// A launch in which CTAs wait for partials that other CTAs publish (every
// stream-K form: the finishing piece of a tile waits for the others; in the
// spread form every piece waits for every other one) is cooperative: the CUDA
// runtime then starts every CTA of the grid together, or refuses the launch,
// so a waiting CTA never holds an SM that one of its publishers needs, even
// when another kernel (a second GEMM on another stream) occupies the rest of
// the GPU.  The bounded waits remain as a second line of defence.
template <int BN, int MODE, int EPI, int KS = 1>
cudaError_t launch_bn(const TcParams& p, int grid, cudaStream_t stream) {
    constexpr int CM = Cfg<BN, MODE, EPI, KS>::CM;
    const bool waits = p.sk_spread || p.sk_split > 0 || p.sk_iters > 0 || p.sk_atomic;
    const bool pdl = p.pdl && !waits;
    if (CM == 1 && !waits && !pdl) {
        tc_gemm_kernel<BN, MODE, EPI, KS>
            <<<grid, Cfg<BN, MODE, EPI, KS>::THREADS, Cfg<BN, MODE, EPI, KS>::SMEM, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg<BN, MODE, EPI, KS>::THREADS);
    cfg.dynamicSmemBytes = Cfg<BN, MODE, EPI, KS>::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    unsigned n = 0;
    if (CM > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CM;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (waits) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<BN, MODE, EPI, KS>, p);
}

template <int BN, int MODE, int EPI, int KS = 1>
cudaError_t prepare_bn() {
    return cudaFuncSetAttribute(tc_gemm_kernel<BN, MODE, EPI, KS>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(Cfg<BN, MODE, EPI, KS>::SMEM));
}

// Two-CTA clusters that can be resident at once (0 on error).
template <int BN, int MODE, int EPI, int KS = 1>
int max_clusters_bn() {
    constexpr int CM = 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CM * 64);
    cfg.blockDim = dim3(Cfg<BN, MODE, EPI, KS>::THREADS);
    cfg.dynamicSmemBytes = Cfg<BN, MODE, EPI, KS>::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<BN, MODE, EPI, KS>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace
}  // namespace dg
