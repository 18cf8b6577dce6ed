// Host side of the C ABI declared in include/gemm.h: argument validation,
// planning (tile width, swap-AB, split-K, operand copies), TMA tensor-map
// encoding and kernel launches.  No device memory is allocated here; the
// only per-device state is a `__device__` error word and kernel attributes.
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "gemm.h"
#include "internal.h"
#include "ptx.cuh"
#include "span_check.h"
#include "tile_order.h"

namespace dg {

// Error word written by kernels whose bounded waits expire.
__device__ int g_status_word;

namespace {

std::atomic<int64_t> g_opt_group_m{8};
std::atomic<int64_t> g_opt_max_ctas{0};
std::atomic<int64_t> g_opt_timeout_us{1000000};
std::atomic<int64_t> g_opt_test_stall{0};
std::atomic<int64_t> g_opt_cta_pair{0};
std::atomic<int64_t> g_opt_swap_ab{0};
std::atomic<int64_t> g_opt_l2_hints{0};
std::atomic<int64_t> g_opt_overlap_copy{0};
std::atomic<int64_t> g_opt_epilogue_warps{0};
std::atomic<int64_t> g_opt_stream_k{0};
std::atomic<int64_t> g_opt_fast_epilogue{0};
std::atomic<int64_t> g_opt_sgemm_kernel{0};
std::atomic<int64_t> g_opt_wide_tile{0};
std::atomic<int64_t> g_opt_split_reduce{0};
std::atomic<int64_t> g_opt_block_n{0};
std::atomic<int64_t> g_opt_double_k{0};
std::atomic<int64_t> g_opt_test_sim_sms{0};
std::atomic<int64_t> g_opt_test_debug_bound{0};
// count-writes mode of the debug build: counter array and its length
std::atomic<uint32_t*> g_dbg_counts{nullptr};
std::atomic<int64_t> g_dbg_count_elems{0};
// stream-K flag values: one fresh 64-bit value per launch (stale or garbage
// workspace contents never equal it)
std::atomic<unsigned long long> g_sk_epoch{0x9E3779B97F4A7C15ull ^
                                           static_cast<unsigned long long>(
                                               reinterpret_cast<uintptr_t>(&g_opt_group_m))};

constexpr int kMaxDevices = 64;
constexpr int kBlockN[] = {16, 32, 64, 128, 256, 512};

struct DevState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sm_count = 0;
    int cc = 0;
    int* status = nullptr;
    int max_pairs[3][3] = {};  // co-resident two-CTA clusters [mode][BN 128, 256, 512] (mode 2)
};
DevState g_dev[kMaxDevices];

gemm_status_t device_state(DevState** out);

// The device a planning query plans for: the current one, or, with the
// test-only GEMM_OPT_TEST_SIM_SMS = n, an sm_103 device of n SMs whose CTA
// pairs of every tile width fit n / 2 at once (nothing is launched).
gemm_status_t planning_device(DevState& sim, DevState** out) {
    const int64_t n = g_opt_test_sim_sms.load();
    if (n <= 0) return device_state(out);
    sim.sm_count = static_cast<int>(n);
    sim.cc = 103;
    for (auto& mode : sim.max_pairs)
        for (int& v : mode) v = static_cast<int>(n / 2);
    *out = &sim;
    return GEMM_OK;
}

gemm_status_t device_state(DevState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    DevState& d = g_dev[dev];
    std::call_once(d.once, [&] {
        int sms = 0, major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        d.cc = major * 10 + minor;
        if (e == cudaSuccess && d.cc == 103) {
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
            for (int bn : kBlockN)
                if (e == cudaSuccess) e = tc_prepare(bn);
            if (e == cudaSuccess) e = sgemm_prepare();
            if (e == cudaSuccess) {
                d.max_pairs[2][0] = tc_max_pairs(128, 2);
                d.max_pairs[2][1] = tc_max_pairs(256, 2);
                d.max_pairs[2][2] = tc_max_pairs(512, 2);
            }
        }
        d.sm_count = sms;
        d.err = e;
        if (e != cudaSuccess) cudaGetLastError();
    });
    if (d.err != cudaSuccess) return GEMM_ERR_CUDA;
    if (d.cc != 103) return GEMM_ERR_NO_DEVICE;
    *out = &d;
    return GEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }
inline int dt_bytes(int dt) { return dt == DT_F32 ? 4 : 2; }

// gemm_epilogue_t fields: bit 0 bias, bits 1-2 activation, bit 3 bias along rows
inline bool epi_valid(int epi) { return epi >= 0 && epi <= 15 && !((epi & 8) && !(epi & 1)); }
inline bool epi_bias(int epi) { return (epi & 1) != 0; }
inline bool epi_row_bias(int epi) { return (epi & 8) != 0; }
inline int epi_act(int epi) {
    switch ((epi >> 1) & 3) {
        case 1: return ACT_GELU_TANH;
        case 2: return ACT_RELU;
        case 3: return ACT_GELU_ERF;
    }
    return ACT_NONE;
}
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Call {
    int ab;
    int64_t batch, M, N, K;
    const void* A;
    int64_t lda;
    int la;
    int64_t sa;
    const void* B;
    int64_t ldb;
    int lb;
    int64_t sb;
    void* C;
    int64_t ldc;
    int lc;
    int64_t sc;
    int cdt;
    float alpha, beta;
    const float* bias;
    int epi;
    int split_k;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

// One operand in the role it plays in the computed problem.
struct Operand {
    const void* ptr;
    int64_t ld, stride;
    bool mn;          // stored MN-contiguous
    int64_t mn_ext;   // extent along M (A role) or N (B role)
    int64_t k_ext;
    bool pack = false;
    int64_t pack_ld = 0;
    int64_t pack_batch = 0;
    size_t pack_off = 0;
    size_t pack_bytes = 0;
    int64_t inner() const { return mn ? mn_ext : k_ext; }
    int64_t outer() const { return mn ? k_ext : mn_ext; }
};

struct Plan {
    int kernel = 0;  // 0 none, 1 tensor core, 2 CUDA-core fp32, 3 epilogue only
    bool swap = false;
    int64_t Mc = 0, Nc = 0;
    int bn = 0, stages = 0, splits = 1, group_m = 8, grid = 0, launches = 0, cm = 1, mode = 0;
    bool fast_epi = false;  // TMA-store-only epilogue form
    bool beta_epi = false;  // TMA-store epilogue that reads beta * C by TMA loads
    bool epi8 = false;      // epilogue on eight warps (forms 3 and 4)
    int ks = 1;             // 64-deep K blocks per stage and per operand load
    int sk = 0;  // stream-K: 0 off, 1 contiguous K ranges, 2 last wave split into equal pieces
    int inkernel_split = 0;  // automatic split-K done in one kernel by the split form
    bool spread = false;     // ... with every piece reducing a share of its tile
    bool atomic = false;     // ... with every piece adding its partial into C (TMA reduce-add)
    int dp_per_cluster = 0, sk_split = 0, sk_tiles = 0;
    int64_t dp_units = 0, sk_iters = 0;
    int64_t sk_units = 0;    // contiguous form: units cut along K (sk_iters counts their steps)
    size_t sk_off = 0, sk_bytes = 0, sk_flags_off = 0, sk_flags_bytes = 0;
    int64_t kblocks = 0, tiles = 0, units = 0;
    Operand a{}, b{};
    bool c_row_major_c = true;
    size_t part_off = 0, part_bytes = 0, ws_need = 0;
};

gemm_status_t validate(const Call& c) {
    if (c.ab != DT_BF16 && c.ab != DT_F16 && c.ab != DT_F32) return GEMM_ERR_INVALID_ARG;
    if (c.cdt != DT_BF16 && c.cdt != DT_F16 && c.cdt != DT_F32) return GEMM_ERR_INVALID_ARG;
    if (c.ab == DT_F32 && c.cdt != DT_F32) return GEMM_ERR_UNSUPPORTED;
    if (c.ab != DT_F32 && c.cdt != DT_F32 && c.cdt != c.ab) return GEMM_ERR_UNSUPPORTED;
    for (int l : {c.la, c.lb, c.lc})
        if (l != GEMM_ROW_MAJOR && l != GEMM_COL_MAJOR) return GEMM_ERR_INVALID_ARG;
    if (!epi_valid(c.epi)) return GEMM_ERR_INVALID_ARG;
    if (c.batch < 0 || c.M < 0 || c.N < 0 || c.K < 0 || c.split_k < 0) return GEMM_ERR_INVALID_ARG;
    const int64_t lim = 0x7FFFFFFF;
    if (c.batch > lim || c.M > lim || c.N > lim || c.K > lim) return GEMM_ERR_INVALID_ARG;
    if (c.batch == 0 || c.M == 0 || c.N == 0) return GEMM_OK;
    if (!c.C) return GEMM_ERR_INVALID_ARG;
    if (!aligned(c.C, dt_bytes(c.cdt))) return GEMM_ERR_INVALID_ARG;
    const int64_t c_inner = c.lc == GEMM_ROW_MAJOR ? c.N : c.M;
    const int64_t c_outer = c.lc == GEMM_ROW_MAJOR ? c.M : c.N;
    if (c.ldc < c_inner) return GEMM_ERR_INVALID_ARG;
    if (!strided_span_ok(c_outer, c_inner, c.ldc, 1, c.batch, c.batch > 1 ? c.sc : 0) ||
        !count_ok(c.batch, c.M, c.N))
        return GEMM_ERR_INVALID_ARG;
    if (c.batch > 1) {
        // C[b] must not overlap
        if (c.sc < (c_outer - 1) * c.ldc + c_inner) return GEMM_ERR_INVALID_ARG;
    }
    if (epi_bias(c.epi) && (!c.bias || !aligned(c.bias, 4))) return GEMM_ERR_INVALID_ARG;
    if (c.K > 0 && c.alpha != 0.0f) {
        if (!c.A || !c.B) return GEMM_ERR_INVALID_ARG;
        if (!aligned(c.A, dt_bytes(c.ab)) || !aligned(c.B, dt_bytes(c.ab)))
            return GEMM_ERR_INVALID_ARG;
        const int64_t a_inner = c.la == GEMM_ROW_MAJOR ? c.K : c.M;
        const int64_t b_inner = c.lb == GEMM_ROW_MAJOR ? c.N : c.K;
        if (c.lda < a_inner || c.ldb < b_inner) return GEMM_ERR_INVALID_ARG;
        if (c.sa < 0 || c.sb < 0) return GEMM_ERR_INVALID_ARG;
        const int64_t a_outer = c.la == GEMM_ROW_MAJOR ? c.M : c.K;
        const int64_t b_outer = c.lb == GEMM_ROW_MAJOR ? c.K : c.N;
        if (!strided_span_ok(a_outer, a_inner, c.lda, 1, c.batch, c.batch > 1 ? c.sa : 0) ||
            !strided_span_ok(b_outer, b_inner, c.ldb, 1, c.batch, c.batch > 1 ? c.sb : 0) ||
            !count_ok(c.batch, c.M, c.K) || !count_ok(c.batch, c.K, c.N))
            return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

// Can TMA address this 16-bit operand in place?
bool tma_addressable(const Operand& o, int64_t batch) {
    if (!aligned(o.ptr, 16)) return false;
    if ((o.ld * 2) % 16 != 0) return false;
    if (batch > 1 && o.stride != 0) {
        if ((o.stride * 2) % 16 != 0) return false;
        if (o.stride < o.outer() * o.ld) return false;
    }
    return true;
}

// Split-K factor: minimises an estimate of the critical path, in units of one
// 64-wide K block of one tile: waves * (K blocks per slice + per-unit fixed
// cost) + (second launch + partial traffic) when split.
int auto_splits(int64_t units, int64_t kblocks, int ctas, int64_t batch, int64_t Mc, int64_t Nc,
                int bn) {
    if (units >= ctas || kblocks < 4) return 1;
    const double unit_cost = 4.0, launch_cost = 10.0;
    const double red_per_split =
        2.0 * batch * Mc * Nc * 4.0 / (static_cast<double>(ctas) * (128 + bn) * 128.0);
    int best = 1;
    double best_cost = static_cast<double>(cdiv(units, ctas)) * (kblocks + unit_cost);
    const int64_t smax = kblocks / 2 < 128 ? kblocks / 2 : 128;
    for (int64_t s = 2; s <= smax; ++s) {
        const double waves = static_cast<double>(cdiv(units * s, ctas));
        const double cost = waves * (static_cast<double>(kblocks) / s + unit_cost) + launch_cost +
                            s * red_per_split;
        if (cost < best_cost) {
            best_cost = cost;
            best = static_cast<int>(s);
        }
    }
    return best;
}

gemm_status_t make_plan(const Call& c, const DevState& d, Plan& pl) {
    const int sm_count = d.sm_count;
    pl = Plan{};
    pl.group_m = static_cast<int>(g_opt_group_m.load());
    int ctas = sm_count;
    const int64_t cap = g_opt_max_ctas.load();
    if (cap > 0 && cap < ctas) ctas = static_cast<int>(cap);
    if (c.batch == 0 || c.M == 0 || c.N == 0) return GEMM_OK;
    if (c.K == 0 || c.alpha == 0.0f) {
        pl.kernel = 3;
        pl.launches = 1;
        return GEMM_OK;
    }
    if (c.ab == DT_F32) {
        pl.kernel = 2;
        pl.launches = 1;
        pl.bn = 128;
        pl.grid = static_cast<int>(c.batch * cdiv(c.M, 128) * cdiv(c.N, 128));
        if (c.batch * cdiv(c.M, 128) * cdiv(c.N, 128) > 0x7FFFFFFF) return GEMM_ERR_UNSUPPORTED;
        return GEMM_OK;
    }
    pl.kernel = 1;
    const int64_t swap_opt = g_opt_swap_ab.load();
    pl.swap = swap_opt == 2 || (swap_opt == 0 && c.M <= 64 && c.N > c.M);
    const Operand opA{c.A, c.lda, c.sa, c.la == GEMM_COL_MAJOR, c.M, c.K};
    const Operand opB{c.B, c.ldb, c.sb, c.lb == GEMM_ROW_MAJOR, c.N, c.K};
    pl.a = pl.swap ? opB : opA;
    pl.b = pl.swap ? opA : opB;
    pl.Mc = pl.swap ? c.N : c.M;
    pl.Nc = pl.swap ? c.M : c.N;
    pl.c_row_major_c = pl.swap ? (c.lc == GEMM_COL_MAJOR) : (c.lc == GEMM_ROW_MAJOR);

    const int64_t tiles_m = cdiv(pl.Mc, TC_BLOCK_M);
    if (pl.Nc <= 16)
        pl.bn = 16;
    else if (pl.Nc <= 32)
        pl.bn = 32;
    else if (pl.Nc <= 64)
        pl.bn = 64;
    else
        pl.bn = (c.batch * tiles_m * cdiv(pl.Nc, 256) >= ctas) ? 256 : 128;
    if (g_opt_block_n.load() > 0) pl.bn = static_cast<int>(g_opt_block_n.load());
    if (pl.b.mn && pl.bn < 64) pl.bn = 64;  // MN-major B tiles come in 64-wide swizzle atoms
    pl.stages = tc_stages_for(pl.bn, 0);

    // operand copies for what TMA cannot address
    size_t off = 0;
    for (Operand* o : {&pl.a, &pl.b}) {
        o->pack = !tma_addressable(*o, c.batch);
        if (o->pack) {
            o->pack_ld = round_up(o->inner(), 8);
            o->pack_batch = (c.batch > 1 && o->stride != 0) ? c.batch : 1;
            o->pack_bytes = static_cast<size_t>(o->pack_batch * o->outer() * o->pack_ld * 2);
            o->pack_off = off;
            off += static_cast<size_t>(round_up(static_cast<int64_t>(o->pack_bytes), 256));
            pl.launches += 1;
        }
    }

    pl.kblocks = cdiv(c.K, TC_BLOCK_K);
    pl.tiles = tiles_m * cdiv(pl.Nc, pl.bn);
    pl.units = c.batch * pl.tiles;
    const size_t per_split = static_cast<size_t>(c.batch * pl.Mc * pl.Nc * 4);
    if (c.split_k >= 1) {
        pl.splits = static_cast<int>(c.split_k < pl.kblocks ? c.split_k : pl.kblocks);
    } else {
        const int s_auto = auto_splits(pl.units, pl.kblocks, ctas, c.batch, pl.Mc, pl.Nc, pl.bn);
        // The automatic split runs in one kernel, as the split form of stream-K
        // below: the S K pieces of each unit go to S CTAs that start together,
        // so there is no reduction pass and no second launch.  It needs a CTA
        // per piece.  Up to kMaxInKernel pieces, piece 0 adds the others' fp32
        // partials in tensor memory one by one before writing the output; with
        // more (or GEMM_OPT_SPLIT_REDUCE = 2) every piece publishes its partial
        // and then reduces one S-th of the tile (GEMM_OPT_SPLIT_REDUCE = 1 keeps
        // the two-pass form there instead).
        constexpr int kMaxInKernel = 4;
        int s_in = s_auto;
        if (pl.units > 0 && s_in > ctas / pl.units) s_in = static_cast<int>(ctas / pl.units);
        if (s_in > pl.kblocks / 4) s_in = static_cast<int>(pl.kblocks / 4);
        const int64_t want_spread = g_opt_split_reduce.load();
        const bool spread =
            want_spread == 2 ||
            ((want_spread == 0 || want_spread == 3 || want_spread == 4) && s_auto > kMaxInKernel);
        if (g_opt_stream_k.load() != 1 && s_auto >= 2 && s_in >= 2 &&
            (spread || s_auto <= kMaxInKernel)) {
            const size_t nslots = static_cast<size_t>(pl.units) * (spread ? s_in : s_in - 1);
            const size_t need = static_cast<size_t>(round_up(
                                    static_cast<int64_t>(nslots * TC_BLOCK_M * pl.bn * 4), 256)) +
                                static_cast<size_t>(round_up(static_cast<int64_t>(nslots * 4 * 8), 256));
            if (c.ws != nullptr && off + need <= c.ws_bytes) {
                pl.inkernel_split = s_in;
                pl.spread = spread;
            }
        }
        // The pages' atomic accumulation ("Skill: Write a Triton GEMM Kernel",
        // Kernel design rules), for an fp32 C that takes TMA stores and no
        // activation: every K piece adds alpha * its partial into C, which the
        // CTAs first set to beta * C + bias; no partial slots, no fix-up, no
        // waiting on pieces.  A column-major computed C (a swapped skinny
        // product, one matrix) takes it too, with tiles up to 64 wide and the
        // general epilogue's column-major boxes.  By default where more than
        // kMaxInKernel pieces would otherwise need the spread reduction
        // (measured 30.7 -> 24.6 us on 256 x 256 x 65536), and for a swapped
        // skinny product whatever its piece count (16 x 8192 x 8192: 32.8 ->
        // 30.7 us against the balanced form, whose last pieces wait for the
        // others' partials); GEMM_OPT_SPLIT_REDUCE = 4 whenever it applies, 1
        // and 2 never (their reductions keep a fixed order).
        const int64_t es4 = 4;
        const bool want_atomic =
            want_spread == 4 ||
            (want_spread == 0 && (s_auto > kMaxInKernel || !pl.c_row_major_c));
        if (want_atomic && g_opt_stream_k.load() != 1 && s_auto >= 2 && c.cdt == DT_F32 &&
            epi_act(c.epi) == ACT_NONE && aligned(c.C, 16) &&
            (c.ldc * es4) % 16 == 0 && (c.batch == 1 || (c.sc * es4) % 16 == 0) &&
            (pl.c_row_major_c ? tc_has_fast(pl.bn) : (c.batch == 1 && pl.bn <= 64)) &&
            c.ws != nullptr &&
            off + static_cast<size_t>(round_up(static_cast<int64_t>(ctas) * 8, 256)) <= c.ws_bytes) {
            pl.atomic = true;
            pl.inkernel_split = 0;
            pl.spread = false;
        }
        if (pl.atomic || pl.inkernel_split > 0) {
            pl.splits = 1;
        } else {
            pl.splits = s_auto;
            // never ask for more workspace than was given: the partials start at
            // `off` (256-aligned) and take per_split * splits rounded up to 256
            const size_t avail = c.ws_bytes > off ? c.ws_bytes - off : 0;
            auto need = [&](int s) {
                return static_cast<size_t>(round_up(static_cast<int64_t>(per_split) * s, 256));
            };
            while (pl.splits > 1 && need(pl.splits) > avail) --pl.splits;
            if (pl.splits < 2) pl.splits = 1;
        }
    }
    if (pl.splits > 1) {
        pl.part_off = off;
        pl.part_bytes = per_split * pl.splits;
        off += round_up(static_cast<int64_t>(pl.part_bytes), 256);
        pl.launches += 1;
    }
    pl.ws_need = off;
    // CTA pairs along M (GEMM_OPT_CTA_PAIR: 0 auto, 1 never, 3 pair MMA) for problems with at least a full wave of tile pairs and a
    // main loop of at least kPairMinKBlocks K blocks: with shorter ones the
    // pair's shared epilogue hand-off costs more than the halved B traffic
    // saves (measured: K <= 256 ran 10-25 % slower paired, K = 512 even,
    // K >= 1024 5-20 % faster).
    constexpr int64_t kPairMinKBlocks = 12;
    const int64_t want = g_opt_cta_pair.load();
    int mode = 0;
    if (want == 3 || want == 0) mode = 2;
    const int bn_idx = pl.bn == 256 ? 1 : 0;
    int max_pairs = mode > 0 && (pl.bn == 128 || pl.bn == 256) ? d.max_pairs[mode][bn_idx] : 0;
    const int64_t pair_units = c.batch * cdiv(pl.Mc, 2 * TC_BLOCK_M) * cdiv(pl.Nc, pl.bn);
    // The atomic split-K runs paired whenever two tile rows allow it: a pair
    // loads each operand element once per K piece instead of once per tile
    // row or column that uses it (measured on 256 x 256 x 65536).
    const bool pair_atomic = pl.atomic && (pl.bn == 128 || pl.bn == 256);
    if (mode > 0 && tc_has_mode(pl.bn, mode) && max_pairs > 0 && pl.splits == 1 && tiles_m >= 2 &&
        pl.inkernel_split == 0 &&
        (want == 3 || pair_atomic ||
         (!pl.atomic && pair_units >= max_pairs && pl.kblocks >= kPairMinKBlocks))) {
        pl.mode = mode;
        pl.cm = 2;
        pl.stages = tc_stages_for(pl.bn, mode);
        pl.tiles = cdiv(pl.Mc, 2 * TC_BLOCK_M) * cdiv(pl.Nc, pl.bn);
        pl.units = pair_units;
        // wide pair tile, 256 x 512 (GEMM_OPT_WIDE_TILE: 0 auto, 1 never, 2 whenever
        // the pair MMA runs with BN = 256 and N >= 512)
        const int64_t wide = g_opt_wide_tile.load();
        const int mp_wide = d.max_pairs[2][2];
        if (pl.mode == 2 && (pl.bn == 256 || (pl.bn == 128 && wide == 2)) && pl.Nc >= 512 &&
            mp_wide > 0 && wide == 2) {
            pl.bn = 512;
            pl.stages = tc_stages_for(512, 2);
            pl.tiles = cdiv(pl.Mc, 2 * TC_BLOCK_M) * cdiv(pl.Nc, 512);
            pl.units = c.batch * pl.tiles;
            max_pairs = mp_wide;
        }
    }
    const int64_t total_units = pl.units * pl.splits;
    if (total_units > 0x7FFFFFFF) return GEMM_ERR_UNSUPPORTED;
    if (pl.cm == 2) {
        int clusters = max_pairs;
        if (cap > 0 && cap / 2 < clusters) clusters = static_cast<int>(cap / 2 > 0 ? cap / 2 : 1);
        if (total_units < clusters) clusters = static_cast<int>(total_units);
        pl.grid = 2 * clusters;
    } else {
        pl.grid = static_cast<int>(total_units < ctas ? total_units : ctas);
    }
    // Stream-K ("2 . La GEMM, de zero a cuBLAS", section 2.10): when whole-unit
    // waves would leave clusters idle in the last one, the last units are cut
    // along K.  GEMM_OPT_STREAM_K: 0 auto, 1 never, 2 contiguous form, 3 split form
    // (both forced whenever a partial last wave follows at least one full wave).
    const int64_t want_sk = g_opt_stream_k.load();
    const int64_t P = pl.grid / pl.cm;
    auto sk_need = [&](size_t nslots) {
        return static_cast<size_t>(round_up(static_cast<int64_t>(nslots * TC_BLOCK_M * pl.bn * 4), 256)) +
               static_cast<size_t>(round_up(static_cast<int64_t>(nslots * 4 * 8), 256));
    };
    if (pl.atomic) {
        // atomic split-K: the contiguous form over every CTA, no whole units
        // first; the workspace holds only each CTA's flag for C's initial values
        const size_t flags = static_cast<size_t>(ctas) * 8;
        pl.sk = 1;
        pl.dp_per_cluster = 0;
        pl.dp_units = 0;
        pl.sk_units = pl.units;
        pl.sk_off = off;
        pl.sk_bytes = 0;
        pl.sk_flags_off = off;
        pl.sk_flags_bytes = flags;
        off += static_cast<size_t>(round_up(static_cast<int64_t>(flags), 256));
        pl.ws_need = off;
        if (pl.cm == 2) {
            // every cluster that fits takes a piece, whatever the unit count
            int clusters = max_pairs;
            if (cap > 0 && cap / 2 < clusters) clusters = static_cast<int>(cap / 2 > 0 ? cap / 2 : 1);
            pl.grid = 2 * clusters;
        } else {
            pl.grid = ctas;
        }
    } else if (pl.inkernel_split > 0 && !pl.spread && g_opt_split_reduce.load() != 3 && pl.units > 0 &&
        ctas / pl.units <= 4 && ctas > pl.units && off + sk_need(ctas) <= c.ws_bytes) {
        // the automatic split-K above, in one kernel, balanced over every CTA:
        // the contiguous form with no whole units first, each CTA taking an
        // equal range of the units' K steps.  A unit then spans a few CTAs
        // (at most ceil(ctas / units) + 1); the one holding its first step adds
        // the others' partials.  (GEMM_OPT_SPLIT_REDUCE = 3 keeps equal
        // pieces, one CTA each, on inkernel_split * units CTAs instead.)
        const size_t nslots = static_cast<size_t>(ctas);
        const size_t slots = nslots * TC_BLOCK_M * pl.bn * 4;
        const size_t flags = nslots * 4 * 8;
        pl.sk = 1;
        pl.inkernel_split = 0;
        pl.dp_per_cluster = 0;
        pl.dp_units = 0;
        pl.sk_units = pl.units;
        pl.sk_off = off;
        pl.sk_bytes = slots;
        pl.sk_flags_off = off + static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256));
        pl.sk_flags_bytes = flags;
        off += static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256)) +
               static_cast<size_t>(round_up(static_cast<int64_t>(flags), 256));
        pl.ws_need = off;
        pl.grid = ctas;
    } else if (pl.inkernel_split > 0) {
        // the automatic split-K above, in one kernel: no whole units first, every
        // unit cut into inkernel_split pieces, one CTA each
        const int64_t S = pl.inkernel_split, r = pl.units;
        const size_t nslots = static_cast<size_t>(r * (pl.spread ? S : S - 1));
        const size_t slots = nslots * TC_BLOCK_M * pl.bn * 4;
        const size_t flags = nslots * 4 * 8;
        pl.sk = 2;
        pl.dp_per_cluster = 0;
        pl.dp_units = 0;
        pl.sk_split = static_cast<int>(S);
        pl.sk_tiles = static_cast<int>(r);
        pl.sk_off = off;
        pl.sk_bytes = slots;
        pl.sk_flags_off = off + static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256));
        pl.sk_flags_bytes = flags;
        off += static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256)) +
               static_cast<size_t>(round_up(static_cast<int64_t>(flags), 256));
        pl.ws_need = off;
        pl.grid = static_cast<int>(S * r);
    } else if (want_sk != 1 && c.split_k != 1 && pl.splits == 1 && P > 0 && pl.units > P &&
               pl.units % P != 0 && pl.kblocks >= 2 && pl.bn <= 256) {
        // (split_k == 1 asks for no split of K at all: every tile is summed over
        // the whole K in one accumulator, so no stream-K pieces either)
        const int64_t W = pl.units / P, r = pl.units % P;
        // split form: each of the r last units becomes S pieces of at least
        // kMinPiece K blocks, one per cluster, all starting together so that
        // concurrent clusters keep reading the same K slices of A and B; the
        // piece that finishes a unit adds the others' partials one by one, so
        // S stays small
        constexpr int64_t kMinPiece = 4, kMaxSplit = 4;
        int64_t S = P / r;
        if (S > kMaxSplit) S = kMaxSplit;
        if (S > pl.kblocks / kMinPiece) S = pl.kblocks / kMinPiece;
        int form = 0;
        if (want_sk == 2) {
            form = 1;
        } else if (want_sk == 3) {
            form = S >= 2 ? 2 : 0;
        } else if (S >= 2) {
            // Cost model in K-block times: the last wave shrinks from kblocks to
            // kblocks / S; each cut unit costs one extra epilogue for the partial
            // and half of one per partial added.  An epilogue is about 10 K
            // blocks of main loop with 128 x 256 tiles; kEpi = 20 also covers
            // what the measured gains fell short of that (a partial last wave
            // of whole tiles runs faster than a full one), so that auto picks
            // the split form only where it measured a gain (K >= 4096).
            constexpr double kEpi = 20.0;
            const double gain = static_cast<double>(pl.kblocks) * (1.0 - 1.0 / S);
            const double cost = kEpi * (1.0 + 0.5 * static_cast<double>(S - 1));
            if (gain > cost) form = 2;
        }
        if (form != 0) {
            const int64_t nslots = form == 1 ? P : r * (S - 1);
            const size_t slots = static_cast<size_t>(nslots) * pl.cm * TC_BLOCK_M * pl.bn * 4;
            const size_t flags = static_cast<size_t>(nslots) * pl.cm * 4 * 8;
            const size_t need = static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256)) +
                                static_cast<size_t>(round_up(static_cast<int64_t>(flags), 256));
            if (c.ws != nullptr && off + need <= c.ws_bytes) {
                pl.sk = form;
                if (form == 1) {
                    pl.dp_per_cluster = static_cast<int>(W - 1);
                    pl.dp_units = (W - 1) * P;
                    pl.sk_units = pl.units - pl.dp_units;
                } else {
                    pl.dp_per_cluster = static_cast<int>(W);
                    pl.dp_units = W * P;
                    pl.sk_split = static_cast<int>(S);
                    pl.sk_tiles = static_cast<int>(r);
                }
                pl.sk_off = off;
                pl.sk_bytes = slots;
                pl.sk_flags_off = off + static_cast<size_t>(round_up(static_cast<int64_t>(slots), 256));
                pl.sk_flags_bytes = flags;
                off += need;
                pl.ws_need = off;
            }
        }
    }
    pl.launches += 1;
    // epilogue form: the TMA-store-only one when the output (C, or the split-K
    // partials) takes TMA stores and no beta * C has to be read
    if (pl.atomic) {
        // checked above: fp32 C that takes TMA stores (row-major: the TMA-store
        // epilogue; column-major: the general one's column boxes)
        pl.fast_epi = pl.c_row_major_c;
    } else if (g_opt_fast_epilogue.load() == 0 && tc_has_fast(pl.bn) && pl.c_row_major_c) {
        if (pl.splits > 1) {
            pl.fast_epi = (pl.Nc * 4) % 16 == 0;
        } else if (c.beta == 0.0f) {
            const int64_t es = dt_bytes(c.cdt);
            pl.fast_epi = aligned(c.C, 16) && (c.ldc * es) % 16 == 0 &&
                          (c.batch == 1 || (c.sc * es) % 16 == 0);
        } else if (c.cdt != DT_F32 && tc_has_beta_form(pl.bn, pl.mode)) {
            // beta * C read by TMA loads through the output's tensor map
            pl.beta_epi = aligned(c.C, 16) && (c.ldc * 2) % 16 == 0 &&
                          (c.batch == 1 || (c.sc * 2) % 16 == 0);
            if (pl.beta_epi) pl.stages = tc_stages_beta(pl.bn, pl.mode);
        }
    }
    // Two K blocks per TMA load (KS = 2) wherever the kernel is compiled that
    // way (tc_has_ks2: CTA pairs with the TMA-store-only epilogue; single CTAs
    // with it or with the general epilogue, for at least 8 K blocks): whole
    // units and stream-K pieces alike, whose boundaries then fall on whole
    // two-block steps; explicit split-K slices are not cut that way.
    // A K-major operand is seen as (64 K, rows, K blocks), so K must be a whole
    // number of 64-deep blocks (an odd count reads its last block's partner
    // past the end: zeros) and the operand one matrix (one batch entry, or a
    // broadcast).  An MN-major operand keeps its own map with boxes of 128 K
    // rows instead of 64 (rows past K: zeros), batched or not.  (A K-major
    // operand with a K that ends inside a block could load its last step
    // through the ordinary map; measured on K = 1000 that was 1-2 us slower
    // than one block per load, so such a K keeps one block per load.)
    auto ks2_ok = [&](const Operand& o) {
        return o.mn || (c.K % TC_BLOCK_K == 0 && (c.batch == 1 || o.stride == 0));
    };
    const int epi_form = pl.beta_epi ? 2 : (pl.fast_epi ? 1 : 0);
    if (g_opt_double_k.load() == 0 && pl.kernel == 1 && pl.splits == 1 &&
        tc_has_ks2(pl.bn, pl.mode, epi_form) && (pl.mode == 2 || pl.kblocks >= 8) &&
        ks2_ok(pl.a) && ks2_ok(pl.b)) {
        pl.ks = 2;
        pl.stages = tc_stages_ks2(pl.bn, pl.mode, epi_form);
    }
    // Forms 3 and 4: the epilogue of whole 256-wide pair tiles runs on eight
    // warps, two per tensor-memory lane quarter, each writing half the
    // columns.  Form 3 takes a general (plain-store) epilogue, for an output
    // TMA cannot store (a row-major C whose base, rows or batch stride are not
    // 16-byte aligned; a column-major one): its chain of shared-memory
    // transposes and plain stores is latency-bound, and short-K tiles wait for
    // it through the two accumulators.  Form 4 takes the epilogue that reads
    // beta * C by TMA loads, for short-K tiles (at most 32 K blocks), with one
    // output box per warp so that the pipeline keeps four stages.
    // GEMM_OPT_EPILOGUE_WARPS = 4 keeps four warps.
    {
        const int64_t es = dt_bytes(c.cdt);
        const bool c_tma_able = pl.c_row_major_c && aligned(c.C, 16) && (c.ldc * es) % 16 == 0 &&
                                (c.batch == 1 || (c.sc * es) % 16 == 0);
        const bool whole = pl.kernel == 1 && pl.ks == 1 && pl.splits == 1 && pl.sk == 0 &&
                           !pl.atomic && !pl.spread && pl.inkernel_split == 0 &&
                           g_opt_epilogue_warps.load() == 0;
        const int form = (epi_form == 0 && !c_tma_able) ? 3
                         : (epi_form == 2 && pl.kblocks <= 32) ? 4
                                                                : 0;
        if (whole && form != 0 && tc_has_epi8(pl.bn, pl.mode, form)) {
            pl.epi8 = true;
            pl.stages = tc_stages_epi8(pl.bn, pl.mode, form);
        }
    }
    // the contiguous form's iterations are steps of ks K blocks
    if (pl.sk == 1) pl.sk_iters = pl.sk_units * cdiv(pl.kblocks, pl.ks);
    // the tensor-core kernel counts work units and tiles in 32-bit integers
    if (pl.kernel == 1 && (pl.units > 0x7FFFFFFF / (pl.splits > 0 ? pl.splits : 1) ||
                           pl.tiles > 0x7FFFFFFF))
        return GEMM_ERR_UNSUPPORTED;
    if (pl.ws_need > 0 && (c.ws == nullptr || c.ws_bytes < pl.ws_need)) return GEMM_ERR_WORKSPACE;
    if (pl.ws_need > 0 && !aligned(c.ws, 256)) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// bias_on_rows: the computed problem is the caller's transposed (swap-AB).
Epilogue make_epilogue(const Call& c, bool row_major, bool bias_on_rows) {
    Epilogue e{};
    e.C = c.C;
    e.ldc = c.ldc;
    e.stride_c = c.batch > 1 ? c.sc : 0;
    e.c_row_major = row_major ? 1 : 0;
    e.c_dtype = c.cdt;
    const int es = dt_bytes(c.cdt);
    e.c_vec_ok = (row_major && aligned(c.C, 16) && (c.ldc * es) % 16 == 0 &&
                  (e.stride_c * es) % 16 == 0)
                     ? 1
                     : 0;
    e.alpha = c.alpha;
    e.beta = c.beta;
    e.bias = epi_bias(c.epi) ? c.bias : nullptr;
    // a row bias of the caller's problem runs along the columns of a swapped one
    e.bias_on_rows = (bias_on_rows != epi_row_bias(c.epi)) ? 1 : 0;
    e.act = epi_act(c.epi);
    return e;
}

// Debug build: the bounds the device-side checks use for the output side of
// a call (C's span, the bias length, the count-writes array), and whether the
// count array is large enough.  A no-op returning GEMM_OK in the product build.
gemm_status_t debug_epilogue(Epilogue& e, const Call& c, bool swap, int* status) {
#if DG_DEBUG
    const int64_t inner = c.lc == GEMM_ROW_MAJOR ? c.N : c.M;
    const int64_t outer = c.lc == GEMM_ROW_MAJOR ? c.M : c.N;
    e.dbg_status = status;
    e.dbg_c_elems = (c.batch > 1 ? (c.batch - 1) * c.sc : 0) + (outer - 1) * c.ldc + inner;
    e.dbg_bias_len = epi_bias(c.epi) ? (epi_row_bias(c.epi) ? c.M : c.N) : 0;
    e.dbg_counts = g_dbg_counts.load();
    e.dbg_m = c.M;
    e.dbg_n = c.N;
    e.dbg_swap = swap ? 1 : 0;
    if (e.dbg_counts && c.batch * c.M * c.N > g_dbg_count_elems.load())
        return GEMM_ERR_INVALID_ARG;
#else
    (void)e, (void)c, (void)swap, (void)status;
#endif
    return GEMM_OK;
}

gemm_status_t encode_operand(CUtensorMap* map, int ab, const Operand& o, const void* ptr,
                             int64_t ld, int64_t stride, int64_t batch, uint32_t box_k_major_rows,
                             bool two_k_blocks, bool* is3d) {
    auto fn = encode_fn();
    if (!fn) return GEMM_ERR_CUDA;
    const CUtensorMapDataType type =
        ab == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (two_k_blocks && !o.mn) {
        // K-major, K a multiple of 64: (64 K, rows, K blocks), two K blocks a box
        if (o.k_ext % 64 != 0) return GEMM_ERR_UNSUPPORTED;
        cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(o.outer()),
                              static_cast<cuuint64_t>(o.k_ext / 64)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), 128u};
        cuuint32_t box[3] = {64u, box_k_major_rows, 2u};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        const CUresult r = fn(map, type, 3u, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
        *is3d = true;
        return GEMM_OK;
    }
    const bool three = batch > 1 && stride != 0;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(o.inner()), static_cast<cuuint64_t>(o.outer()),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * 2), static_cast<cuuint64_t>(stride * 2)};
    // K-major: box = 64 K x rows-of-tile; MN-major: box = 64 MN x 64 K (one swizzle atom
    // column), or 64 MN x 128 K when one load brings two K blocks (rows past K: zeros)
    cuuint32_t box[3] = {64u, o.mn ? (two_k_blocks ? 128u : 64u) : box_k_major_rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(map, type, three ? 3u : 2u, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
    *is3d = three;
    return GEMM_OK;
}

// Tensor map of the epilogue's output boxes (32 columns x 32 rows): C itself
// when TMA can address it, or the dense fp32 split-K partials.  Returns false
// when the row-major TMA epilogue does not apply (the kernel then falls back
// to st.global stores).
// Output map of the tensor-core epilogue: boxes of 32 rows by 32 columns, or,
// with `wide`, by 128 bytes of columns (64 for a 16-bit C), 128-byte swizzled
// when a box row is 128 bytes and 64-byte swizzled otherwise.
bool encode_output_map(CUtensorMap* map, int dt, void* ptr, int64_t N, int64_t M, int64_t ld,
                       int64_t depth, int64_t stride, bool wide, bool* is3d) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int es = dt_bytes(dt);
    if (!aligned(ptr, 16) || (ld * es) % 16 != 0) return false;
    const bool three = depth > 1;
    if (three && (stride * es) % 16 != 0) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                          static_cast<cuuint64_t>(depth)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es), static_cast<cuuint64_t>(stride * es)};
    const cuuint32_t box_cols = wide ? static_cast<cuuint32_t>(128 / es) : 32u;
    cuuint32_t box[3] = {box_cols, 32u, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUtensorMapDataType t = dt == DT_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dt == DT_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const CUresult r =
        fn(map, t, three ? 3u : 2u, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           box_cols * es == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    *is3d = three;
    return true;
}

// Output map of a column-major fp32 C (one matrix) for the atomic split-K:
// rows contiguous, boxes of 32 rows by `cols` columns, no swizzle.
bool encode_output_cols_map(CUtensorMap* map, void* ptr, int64_t rows, int64_t cols_total,
                            int64_t ld, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (!aligned(ptr, 16) || (ld * 4) % 16 != 0) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols_total)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 4)};
    cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(cols)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2u, ptr, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gemm_status_t run(const Call& c) {
    gemm_status_t st = validate(c);
    if (st != GEMM_OK) return st;
    if (c.batch == 0 || c.M == 0 || c.N == 0) return GEMM_OK;
    DevState* d = nullptr;
    st = device_state(&d);
    if (st != GEMM_OK) return st;
    Plan pl;
    st = make_plan(c, *d, pl);
    if (st != GEMM_OK) return st;

    if (pl.kernel == 3) {
        Epilogue e = make_epilogue(c, c.lc == GEMM_ROW_MAJOR, false);
        st = debug_epilogue(e, c, false, d->status);
        if (st != GEMM_OK) return st;
        return splitk_epilogue_launch(nullptr, 0, c.batch, c.M, c.N, e, c.stream) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    }
    if (pl.kernel == 2) {
        SgemmParams p{};
        p.A = static_cast<const float*>(c.A);
        p.lda = c.lda;
        p.stride_a = c.batch > 1 ? c.sa : 0;
        p.a_row = c.la == GEMM_ROW_MAJOR;
        p.B = static_cast<const float*>(c.B);
        p.ldb = c.ldb;
        p.stride_b = c.batch > 1 ? c.sb : 0;
        p.b_row = c.lb == GEMM_ROW_MAJOR;
        p.M = static_cast<int32_t>(c.M);
        p.N = static_cast<int32_t>(c.N);
        p.K = static_cast<int32_t>(c.K);
        p.batch = static_cast<int32_t>(c.batch);
        p.a_vec_ok = aligned(c.A, 16) && c.lda % 4 == 0 && p.stride_a % 4 == 0;
        p.b_vec_ok = aligned(c.B, 16) && c.ldb % 4 == 0 && p.stride_b % 4 == 0;
        // the cp.async kernel (128 x 64 tiles) for row-major, 16-byte aligned A
        // and B; the register-staged one (128 x 128 tiles) for everything else
        p.kernel = g_opt_sgemm_kernel.load() == 0 && p.a_row && p.b_row && p.a_vec_ok &&
                           p.b_vec_ok
                       ? 0
                       : 1;
        p.num_pid_m = static_cast<int32_t>(cdiv(c.M, 128));
        p.num_pid_n = static_cast<int32_t>(cdiv(c.N, p.kernel == 0 ? 64 : 128));
        p.group_m = pl.group_m;
        p.epi = make_epilogue(c, c.lc == GEMM_ROW_MAJOR, false);
        st = debug_epilogue(p.epi, c, false, d->status);
        if (st != GEMM_OK) return st;
        return sgemm_launch(p, c.stream) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }

    // tensor-core path
    char* ws = static_cast<char*>(c.ws);
    const void* a_ptr = pl.a.ptr;
    const void* b_ptr = pl.b.ptr;
    int64_t a_ld = pl.a.ld, b_ld = pl.b.ld;
    int64_t a_stride = c.batch > 1 ? pl.a.stride : 0, b_stride = c.batch > 1 ? pl.b.stride : 0;
    if (pl.a.pack) {
        if (pack16_launch(pl.a.ptr, pl.a.ld, a_stride, pl.a.outer(), pl.a.inner(), pl.a.pack_batch,
                          ws + pl.a.pack_off, pl.a.pack_ld, c.stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        a_ptr = ws + pl.a.pack_off;
        a_ld = pl.a.pack_ld;
        a_stride = pl.a.pack_batch > 1 ? pl.a.outer() * pl.a.pack_ld : 0;
    }
    if (pl.b.pack) {
        if (pack16_launch(pl.b.ptr, pl.b.ld, b_stride, pl.b.outer(), pl.b.inner(), pl.b.pack_batch,
                          ws + pl.b.pack_off, pl.b.pack_ld, c.stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        b_ptr = ws + pl.b.pack_off;
        b_ld = pl.b.pack_ld;
        b_stride = pl.b.pack_batch > 1 ? pl.b.outer() * pl.b.pack_ld : 0;
    }

    TcParams p;
    std::memset(&p, 0, sizeof(p));
    bool a3 = false, b3 = false;
    st = encode_operand(&p.tmap_a, c.ab, pl.a, a_ptr, a_ld, a_stride, c.batch, TC_BLOCK_M,
                        pl.ks == 2, &a3);
    if (st != GEMM_OK) return st;
    // B box: the rows (N) one load brings, half of an N <= 256 MMA per CTA of a pair
    const int sub_n = pl.bn < 256 ? pl.bn : 256;
    st = encode_operand(&p.tmap_b, c.ab, pl.b, b_ptr, b_ld, b_stride, c.batch,
                        static_cast<uint32_t>(pl.cm == 2 ? sub_n / 2 : pl.bn), pl.ks == 2, &b3);
    if (st != GEMM_OK) return st;
    p.M = static_cast<int32_t>(pl.Mc);
    p.N = static_cast<int32_t>(pl.Nc);
    p.K = static_cast<int32_t>(c.K);
    p.batch = static_cast<int32_t>(c.batch);
    p.num_pid_m = static_cast<int32_t>(cdiv(pl.Mc, TC_BLOCK_M * pl.cm));
    p.num_pid_n = static_cast<int32_t>(cdiv(pl.Nc, pl.bn));
    p.tiles_per_batch = static_cast<int32_t>(pl.tiles);
    p.splits = pl.splits;
    p.kblocks = static_cast<int32_t>(pl.kblocks);
    p.group_m = pl.group_m;
    p.total_units = static_cast<int32_t>(pl.units * pl.splits);
    p.a_mn = pl.a.mn ? 1 : 0;
    p.b_mn = pl.b.mn ? 1 : 0;
    p.a_3d = a3 ? 1 : 0;
    p.b_3d = b3 ? 1 : 0;
    p.idesc = make_idesc_f16(c.ab == DT_BF16, pl.a.mn, pl.b.mn, pl.mode == 2 ? 2 * TC_BLOCK_M : TC_BLOCK_M,
                             sub_n);
    p.epi = make_epilogue(c, pl.c_row_major_c, pl.swap);
    st = debug_epilogue(p.epi, c, pl.swap, d->status);
    if (st != GEMM_OK) return st;
    p.partials = pl.splits > 1 ? reinterpret_cast<float*>(ws + pl.part_off) : nullptr;
    const bool want_fast = pl.fast_epi || pl.beta_epi;  // 128-byte boxes
    int epi_form = 0;
    if (pl.c_row_major_c && pl.bn >= 32) {
        bool c3 = false;
        bool ok;
        if (p.partials)
            ok = encode_output_map(&p.tmap_c, DT_F32, p.partials, pl.Nc, pl.Mc, pl.Nc,
                                   static_cast<int64_t>(pl.splits) * c.batch, pl.Mc * pl.Nc,
                                   want_fast, &c3);
        else
            ok = encode_output_map(&p.tmap_c, c.cdt, c.C, pl.Nc, pl.Mc, c.ldc, c.batch, c.sc,
                                   want_fast, &c3);
        p.c_tma = ok ? 1 : 0;
        p.c_tma_3d = c3 ? 1 : 0;
        epi_form = ok && pl.beta_epi ? 2 : (ok && pl.fast_epi ? 1 : 0);
        if (pl.epi8) {
            // the plan took C as TMA-storable exactly for form 4
            if (ok != pl.beta_epi) return GEMM_ERR_UNSUPPORTED;
            epi_form = pl.beta_epi ? 4 : 3;
        }
    } else if (pl.atomic) {
        // column-major computed C, one matrix: boxes of 32 contiguous rows by
        // the tile's columns, for the TMA reduce-adds
        if (!encode_output_cols_map(&p.tmap_c, c.C, pl.Mc, pl.Nc, c.ldc, pl.bn))
            return GEMM_ERR_CUDA;
    }
    p.status = d->status;
    p.timeout_ns = static_cast<uint64_t>(g_opt_timeout_us.load()) * 1000ull;
    p.test_stall = static_cast<int32_t>(g_opt_test_stall.exchange(0));
    p.l2_hints = static_cast<int32_t>(g_opt_l2_hints.load());
    // the launch right before this one is an operand copy: let the GEMM in early
    p.pdl = (pl.a.pack || pl.b.pack) && g_opt_overlap_copy.load() == 0 ? 1 : 0;
    if (pl.sk) {
        p.dp_per_cluster = pl.dp_per_cluster;
        p.dp_units = static_cast<int32_t>(pl.dp_units);
        p.sk_iters = pl.sk_iters;
        p.sk_split = pl.sk_split;
        p.sk_tiles = pl.sk_tiles;
        p.sk_spread = pl.spread ? 1 : 0;
        p.sk_atomic = pl.atomic ? 1 : 0;
        p.sk_partials = reinterpret_cast<float*>(ws + pl.sk_off);
        p.sk_flags = reinterpret_cast<unsigned long long*>(ws + pl.sk_flags_off);
        do {
            p.sk_epoch = g_sk_epoch.fetch_add(1) + 1;
        } while (p.sk_epoch == 0);  // cleared flags (0) must never read as published
        // A launch captured into a CUDA graph is replayed with this same epoch,
        // so the flags an earlier replay published would already read as
        // published to the next one.  When capturing, clear them in the graph,
        // right before the kernel, so that every replay starts from zero.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(c.stream, &cap) != cudaSuccess) {
            cudaGetLastError();
            cap = cudaStreamCaptureStatusNone;
        }
        if (cap == cudaStreamCaptureStatusActive &&
            cudaMemsetAsync(p.sk_flags, 0, pl.sk_flags_bytes, c.stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
#if DG_DEBUG
    p.dbg_sk_slots = pl.sk ? static_cast<int64_t>(pl.sk_bytes / (TC_BLOCK_M * pl.bn * 4)) : 0;
    p.dbg_partials_elems = pl.splits > 1 ? static_cast<int64_t>(pl.part_bytes / 4) : 0;
    p.dbg_num_pid_n = p.num_pid_n;
    // test only: one bound set too small, so that a check fails (buffers untouched)
    const int64_t plant = g_opt_test_debug_bound.exchange(0);
    if (plant == 1) p.epi.dbg_c_elems /= 2;
    if (plant == 2) p.dbg_num_pid_n -= 1;
#endif
    if (tc_launch(pl.bn, pl.mode, epi_form, pl.ks, p, pl.grid, c.stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (pl.splits > 1) {
        if (splitk_epilogue_launch(p.partials, pl.splits, c.batch, pl.Mc, pl.Nc, p.epi,
                                   c.stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

Call make_call(int ab, int64_t batch, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
               gemm_layout_t la, int64_t sa, const void* B, int64_t ldb, gemm_layout_t lb,
               int64_t sb, void* C, int64_t ldc, gemm_layout_t lc, int64_t sc, int cdt,
               float alpha, float beta, const float* bias, gemm_epilogue_t epi, int split_k,
               void* ws, size_t ws_bytes, gemm_stream_t stream) {
    Call c;
    c.ab = ab;
    c.batch = batch;
    c.M = M;
    c.N = N;
    c.K = K;
    c.A = A;
    c.lda = lda;
    c.la = la;
    c.sa = sa;
    c.B = B;
    c.ldb = ldb;
    c.lb = lb;
    c.sb = sb;
    c.C = C;
    c.ldc = ldc;
    c.lc = lc;
    c.sc = sc;
    c.cdt = cdt;
    c.alpha = alpha;
    c.beta = beta;
    c.bias = bias;
    c.epi = epi;
    c.split_k = split_k;
    c.ws = ws;
    c.ws_bytes = ws_bytes;
    c.stream = static_cast<cudaStream_t>(stream);
    return c;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                        gemm_layout_t la, const void* B, int64_t ldb, gemm_layout_t lb, void* C,
                        int64_t ldc, gemm_layout_t lc, gemm_dtype_t c_dtype, float alpha,
                        float beta, const float* bias, gemm_epilogue_t epi, int split_k,
                        void* workspace, size_t workspace_bytes, gemm_stream_t stream) {
    if (c_dtype == GEMM_DT_F16) return GEMM_ERR_UNSUPPORTED;
    return run(make_call(DT_BF16, 1, M, N, K, A, lda, la, 0, B, ldb, lb, 0, C, ldc, lc, 0, c_dtype,
                         alpha, beta, bias, epi, split_k, workspace, workspace_bytes, stream));
}

gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                       gemm_layout_t la, const void* B, int64_t ldb, gemm_layout_t lb, void* C,
                       int64_t ldc, gemm_layout_t lc, gemm_dtype_t c_dtype, float alpha,
                       float beta, const float* bias, gemm_epilogue_t epi, int split_k,
                       void* workspace, size_t workspace_bytes, gemm_stream_t stream) {
    if (c_dtype == GEMM_DT_BF16) return GEMM_ERR_UNSUPPORTED;
    return run(make_call(DT_F16, 1, M, N, K, A, lda, la, 0, B, ldb, lb, 0, C, ldc, lc, 0, c_dtype,
                         alpha, beta, bias, epi, split_k, workspace, workspace_bytes, stream));
}

gemm_status_t sgemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                        gemm_layout_t la, const float* B, int64_t ldb, gemm_layout_t lb, float* C,
                        int64_t ldc, gemm_layout_t lc, float alpha, float beta, const float* bias,
                        gemm_epilogue_t epi, gemm_stream_t stream) {
    return run(make_call(DT_F32, 1, M, N, K, A, lda, la, 0, B, ldb, lb, 0, C, ldc, lc, 0, DT_F32,
                         alpha, beta, bias, epi, 1, nullptr, 0, stream));
}

gemm_status_t gemm_batched(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N, int64_t K,
                           const void* A, int64_t lda, gemm_layout_t la, int64_t stride_a,
                           const void* B, int64_t ldb, gemm_layout_t lb, int64_t stride_b,
                           void* C, int64_t ldc, gemm_layout_t lc, int64_t stride_c,
                           gemm_dtype_t c_dtype, float alpha, float beta, const float* bias,
                           gemm_epilogue_t epi, int split_k, void* workspace,
                           size_t workspace_bytes, gemm_stream_t stream) {
    return run(make_call(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb, stride_b, C,
                         ldc, lc, stride_c, c_dtype, alpha, beta, bias, epi, split_k, workspace,
                         workspace_bytes, stream));
}

size_t gemm_workspace_size(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N, int64_t K,
                           int split_k) {
    if (ab_dtype != GEMM_DT_BF16 && ab_dtype != GEMM_DT_F16) return 0;
    if (batch <= 0 || M <= 0 || N <= 0 || K <= 0 || split_k < 0) return 0;
    if (batch > 0x7FFFFFFF || M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return 0;
    // the counts every call with these sizes must pass (padding rows to 8 included)
    if (!count_ok(batch, M, N) || !count_ok(batch, M + 8, K + 8) || !count_ok(batch, K + 8, N + 8))
        return 0;
    DevState sim;
    DevState* d = nullptr;
    if (planning_device(sim, &d) != GEMM_OK) return 0;
    const int64_t pa = batch * (M * round_up(K, 8) > K * round_up(M, 8) ? M * round_up(K, 8)
                                                                         : K * round_up(M, 8));
    const int64_t pb = batch * (N * round_up(K, 8) > K * round_up(N, 8) ? N * round_up(K, 8)
                                                                         : K * round_up(N, 8));
    size_t worst_part = 0;
    static const char dummy[16] __attribute__((aligned(256))) = {0};
    for (int la = 0; la < 2; ++la)
        for (int lb = 0; lb < 2; ++lb)
            for (int lc = 0; lc < 2; ++lc) {
                // aligned, unpacked operands with unlimited workspace: the largest split
                const int64_t lda = la == 0 ? round_up(K, 8) : round_up(M, 8);
                const int64_t ldb = lb == 0 ? round_up(N, 8) : round_up(K, 8);
                const int64_t ldc = lc == 0 ? N : M;
                const int64_t sa = la == 0 ? M * lda : K * lda;
                const int64_t sb = lb == 0 ? K * ldb : N * ldb;
                const int64_t sc = lc == 0 ? M * ldc : N * ldc;
                Call c = make_call(ab_dtype, batch, M, N, K, dummy, lda,
                                   static_cast<gemm_layout_t>(la), sa, dummy, ldb,
                                   static_cast<gemm_layout_t>(lb), sb, const_cast<char*>(dummy),
                                   ldc, static_cast<gemm_layout_t>(lc), sc, GEMM_DT_F32, 1.0f,
                                   0.0f, nullptr, GEMM_EPI_NONE, split_k,
                                   const_cast<char*>(dummy), SIZE_MAX / 2, nullptr);
                Plan pl;
                if (make_plan(c, *d, pl) == GEMM_OK && pl.part_bytes > worst_part)
                    worst_part = pl.part_bytes;
            }
    // stream-K slots and flags: one 128 x 256 fp32 tile per CTA of the grid, plus flags
    const int64_t sk = round_up(static_cast<int64_t>(d->sm_count) * TC_BLOCK_M * 256 * 4, 256) +
                       round_up(static_cast<int64_t>(d->sm_count) * 4 * 8, 256);
    return static_cast<size_t>(round_up(pa * 2, 256) + round_up(pb * 2, 256)) +
           static_cast<size_t>(round_up(static_cast<int64_t>(worst_part), 256)) +
           static_cast<size_t>(sk);
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
        case GEMM_ERR_WORKSPACE: return "GEMM_ERR_WORKSPACE";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE";
        case GEMM_ERR_DEVICE_CHECK: return "GEMM_ERR_DEVICE_CHECK";
    }
    return "GEMM_ERR_UNKNOWN";
}

gemm_status_t gemm_check_device_status(gemm_stream_t stream) {
    DevState* d = nullptr;
    const gemm_status_t st = device_state(&d);
    if (st != GEMM_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    int v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return GEMM_ERR_CUDA;
        // bits 8 and up: a failed device-side check (debug build); bit 0: a wait expired
        return (v & ~0xFF) ? GEMM_ERR_DEVICE_CHECK : GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

int32_t gemm_build_flags(void) { return DG_DEBUG ? 1 : 0; }

gemm_status_t gemm_debug_count_writes(uint32_t* counts, int64_t count_elems) {
#if DG_DEBUG
    if (counts != nullptr && count_elems <= 0) return GEMM_ERR_INVALID_ARG;
    g_dbg_count_elems.store(counts ? count_elems : 0);
    g_dbg_counts.store(counts);
    return GEMM_OK;
#else
    (void)counts, (void)count_elems;
    return GEMM_ERR_UNSUPPORTED;
#endif
}

gemm_status_t gemm_plan_query(gemm_dtype_t ab_dtype, int64_t batch, int64_t M, int64_t N,
                              int64_t K, const void* A, int64_t lda, gemm_layout_t la,
                              int64_t stride_a, const void* B, int64_t ldb, gemm_layout_t lb,
                              int64_t stride_b, void* C, int64_t ldc, gemm_layout_t lc,
                              int64_t stride_c, gemm_dtype_t c_dtype, float alpha, float beta,
                              const float* bias, gemm_epilogue_t epi, int split_k,
                              size_t workspace_bytes, gemm_plan_t* plan) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    std::memset(plan, 0, sizeof(*plan));
    // a non-null stand-in so that the plan can be made without a real workspace
    static const char probe[16] __attribute__((aligned(256))) = {0};
    const Call c = make_call(ab_dtype, batch, M, N, K, A, lda, la, stride_a, B, ldb, lb, stride_b,
                             C, ldc, lc, stride_c, c_dtype, alpha, beta, bias, epi, split_k,
                             const_cast<char*>(probe), workspace_bytes, nullptr);
    gemm_status_t st = validate(c);
    if (st != GEMM_OK) return st;
    DevState sim;
    DevState* d = nullptr;
    st = planning_device(sim, &d);
    if (st != GEMM_OK) return st;
    Plan pl;
    st = make_plan(c, *d, pl);
    plan->kernel = pl.kernel;
    plan->block_m = pl.kernel == 1 ? TC_BLOCK_M : (pl.kernel == 2 ? 128 : 0);
    plan->block_n = pl.bn;
    plan->block_k = pl.kernel == 1 ? TC_BLOCK_K * pl.ks : (pl.kernel == 2 ? 8 : 0);
    plan->stages = pl.stages;
    plan->split_k = pl.splits;
    plan->swap_ab = pl.swap ? 1 : 0;
    plan->pack_a = pl.a.pack ? 1 : 0;
    plan->pack_b = pl.b.pack ? 1 : 0;
    plan->grid = pl.grid;
    plan->group_m = pl.group_m;
    plan->launches = pl.launches;
    plan->workspace_bytes = static_cast<int64_t>(pl.ws_need);
    plan->cta_pair = pl.mode;
    plan->fast_epilogue = pl.epi8 ? (pl.beta_epi ? 4 : 3) : (pl.beta_epi ? 2 : (pl.fast_epi ? 1 : 0));
    plan->stream_k = pl.atomic ? 4 : (pl.spread ? 3 : pl.sk);
    return st;
}

gemm_status_t gemm_set_option(gemm_option_t option, int64_t value) {
    switch (option) {
        case GEMM_OPT_GROUP_M:
            if (value < 1 || value > 64) return GEMM_ERR_INVALID_ARG;
            g_opt_group_m.store(value);
            return GEMM_OK;
        case GEMM_OPT_MAX_CTAS:
            if (value < 0 || value > 0x7FFFFFFF) return GEMM_ERR_INVALID_ARG;
            g_opt_max_ctas.store(value);
            return GEMM_OK;
        case GEMM_OPT_TIMEOUT_US:
            if (value < 1 || value > 60ll * 1000 * 1000) return GEMM_ERR_INVALID_ARG;
            g_opt_timeout_us.store(value);
            return GEMM_OK;
        case GEMM_OPT_TEST_STALL:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_opt_test_stall.store(value);
            return GEMM_OK;
        case GEMM_OPT_CTA_PAIR:
            // (2 named pairs that shared B through multicast loads; that form
            // is gone and the value is refused)
            if (value < 0 || value > 3 || value == 2) return GEMM_ERR_INVALID_ARG;
            g_opt_cta_pair.store(value);
            return GEMM_OK;
        case GEMM_OPT_SWAP_AB:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_opt_swap_ab.store(value);
            return GEMM_OK;
        case GEMM_OPT_L2_HINTS:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_opt_l2_hints.store(value);
            return GEMM_OK;
        case GEMM_OPT_STREAM_K:
            if (value < 0 || value > 3) return GEMM_ERR_INVALID_ARG;
            g_opt_stream_k.store(value);
            return GEMM_OK;
        case GEMM_OPT_FAST_EPILOGUE:
            if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
            g_opt_fast_epilogue.store(value);
            return GEMM_OK;
        case GEMM_OPT_SGEMM_KERNEL:
            if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
            g_opt_sgemm_kernel.store(value);
            return GEMM_OK;
        case GEMM_OPT_WIDE_TILE:
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_opt_wide_tile.store(value);
            return GEMM_OK;
        case GEMM_OPT_SPLIT_REDUCE:
            if (value < 0 || value > 4) return GEMM_ERR_INVALID_ARG;
            g_opt_split_reduce.store(value);
            return GEMM_OK;
        case GEMM_OPT_BLOCK_N:
            if (value != 0 && value != 16 && value != 32 && value != 64 && value != 128 &&
                value != 256)
                return GEMM_ERR_INVALID_ARG;
            g_opt_block_n.store(value);
            return GEMM_OK;
        case GEMM_OPT_DOUBLE_K:
            if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
            g_opt_double_k.store(value);
            return GEMM_OK;
        case GEMM_OPT_TEST_SIM_SMS:
            if (value < 0 || value > 4096) return GEMM_ERR_INVALID_ARG;
            g_opt_test_sim_sms.store(value);
            return GEMM_OK;
        case GEMM_OPT_TEST_DEBUG_BOUND:
            if (!DG_DEBUG) return GEMM_ERR_UNSUPPORTED;
            if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
            g_opt_test_debug_bound.store(value);
            return GEMM_OK;
        case GEMM_OPT_OVERLAP_COPY:
            if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
            g_opt_overlap_copy.store(value);
            return GEMM_OK;
        case GEMM_OPT_EPILOGUE_WARPS:
            if (value != 0 && value != 4) return GEMM_ERR_INVALID_ARG;
            g_opt_epilogue_warps.store(value);
            return GEMM_OK;
    }
    return GEMM_ERR_INVALID_ARG;
}

int64_t gemm_get_option(gemm_option_t option) {
    switch (option) {
        case GEMM_OPT_GROUP_M: return g_opt_group_m.load();
        case GEMM_OPT_MAX_CTAS: return g_opt_max_ctas.load();
        case GEMM_OPT_TIMEOUT_US: return g_opt_timeout_us.load();
        case GEMM_OPT_TEST_STALL: return g_opt_test_stall.load();
        case GEMM_OPT_CTA_PAIR: return g_opt_cta_pair.load();
        case GEMM_OPT_SWAP_AB: return g_opt_swap_ab.load();
        case GEMM_OPT_L2_HINTS: return g_opt_l2_hints.load();
        case GEMM_OPT_STREAM_K: return g_opt_stream_k.load();
        case GEMM_OPT_FAST_EPILOGUE: return g_opt_fast_epilogue.load();
        case GEMM_OPT_SGEMM_KERNEL: return g_opt_sgemm_kernel.load();
        case GEMM_OPT_WIDE_TILE: return g_opt_wide_tile.load();
        case GEMM_OPT_SPLIT_REDUCE: return g_opt_split_reduce.load();
        case GEMM_OPT_BLOCK_N: return g_opt_block_n.load();
        case GEMM_OPT_DOUBLE_K: return g_opt_double_k.load();
        case GEMM_OPT_TEST_SIM_SMS: return g_opt_test_sim_sms.load();
        case GEMM_OPT_TEST_DEBUG_BOUND: return g_opt_test_debug_bound.load();
        case GEMM_OPT_OVERLAP_COPY: return g_opt_overlap_copy.load();
        case GEMM_OPT_EPILOGUE_WARPS: return g_opt_epilogue_warps.load();
    }
    return -1;
}

void gemm_tile_order(int num_pid_m, int num_pid_n, int group_m, int* pid_m, int* pid_n) {
    if (num_pid_m <= 0 || num_pid_n <= 0 || group_m <= 0 || !pid_m || !pid_n) return;
    const int64_t n = static_cast<int64_t>(num_pid_m) * num_pid_n;
    for (int64_t t = 0; t < n; ++t)
        tile_coord(static_cast<int>(t), num_pid_m, num_pid_n, group_m, pid_m[t], pid_n[t]);
}

}  // extern "C"
