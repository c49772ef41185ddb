// Host side of the block-scaled FP8 GEMM: launch plan (tile shape, split-K),
// TMA tensor maps, the split-K workspace and the device status word.  The
// kernel itself is in gemm_kernel.cuh; gemm_b*.cu instantiate it per recipe.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "gemm_dual.cuh"
#include "gemm_kernel.cuh"

namespace sgq {

__device__ uint32_t g_gemm_status;
#ifdef SGQ_TRACE
__device__ unsigned long long g_gemm_trace[1024 * gemm::kTraceSlots];
#endif

namespace gemm {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

sgq_status get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode ? SGQ_OK : SGQ_ERR_CUDA;
}

// 2-D map over a [rows, K] uint8 matrix, box = 128 K-bytes x box_rows rows,
// 128-byte swizzle (the UMMA K-major SW128 layout).
sgq_status make_tmap(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, int box_rows) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGQ_OK : SGQ_ERR_CUDA;
}

// 2-D map over a [rows, ks] fp32 scale matrix; box = box_cols columns (a
// multiple of 4, i.e. of 16 bytes) x box_rows rows, no swizzle.  Rows and
// columns past the matrix read as zero.
sgq_status make_scale_map(CUtensorMap* m, const float* ptr, int64_t rows, int64_t ks, int box_rows,
                          int box_cols) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(ks), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ks) * sizeof(float)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGQ_OK : SGQ_ERR_CUDA;
}

// Split-K workspace, one per device, created on first need.  The last
// kDualCounters arrival counts belong to the two-accumulator tiles (their
// counts are never reset, only kept at multiples of 16).
constexpr size_t kWsBytes = size_t(64) << 20;
constexpr int kMaxCounters = 1 << 16;
constexpr int kDualCounters = 1024;
struct DevWs {
    float* partial = nullptr;
    uint32_t* counters = nullptr;
};
DevWs g_ws[64];
std::mutex g_ws_mu;

sgq_status get_workspace(cudaStream_t st, DevWs* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (!g_ws[dev].partial) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return SGQ_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return SGQ_ERR_UNSUPPORTED;
        void* p = nullptr;
        void* c = nullptr;
        if (cudaMalloc(&p, kWsBytes) != cudaSuccess) return SGQ_ERR_CUDA;
        if (cudaMalloc(&c, kMaxCounters * sizeof(uint32_t)) != cudaSuccess) {
            cudaFree(p);
            return SGQ_ERR_CUDA;
        }
        if (cudaMemset(c, 0, kMaxCounters * sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaFree(p);
            cudaFree(c);
            return SGQ_ERR_CUDA;
        }
        g_ws[dev].partial = static_cast<float*>(p);
        g_ws[dev].counters = static_cast<uint32_t*>(c);
    }
    *out = g_ws[dev];
    return SGQ_OK;
}

struct Plan {
    bool swap;
    bool pair;   // CTA pairs on 256 x 256 tiles (cluster of two, cta_group::2)
    bool alt;    // 128 x 256 tiles with two alternating MMA issuers
    bool ck;     // swap-AB with two K splits exchanged inside a cluster of two
    int bn, tiles_r, tiles_c, kb_total, kb_per_split, splits, items, grid;
};

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

// Split-K scratch a plan may use: bytes of fp32 partial tiles and arrival
// counters (one per tile).  The default entry point's workspace, or the
// allocation-free entry point's fixed array.
struct ScratchLimit {
    size_t partial_bytes;
    size_t counters;
};
constexpr ScratchLimit kWsLimit{kWsBytes, size_t(kMaxCounters - kDualCounters)};

// wide_only: keep the 128 x 256 tiles for M > 64 (the issue-mode testing
// flags compare the wide tiles' two issue modes).  lim: the split-K scratch
// available; split counts whose partials or counters exceed it are skipped.
Plan make_plan(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, bool wide_only = false,
               ScratchLimit lim = kWsLimit) {
    Plan p{};
    static const int grid_max = env_int("SGQ_GRID_MAX", 0);
    if (grid_max > 0 && grid_max < sm_count) sm_count = grid_max;
    static const int swap_max = env_int("SGQ_SWAP_MAX", 64);
    static const int mid_swap = env_int("SGQ_MIDSWAP", 1);
    static const int ovh = env_int("SGQ_SPLIT_OVERHEAD", 2);
    static const int forced = env_int("SGQ_SPLITS", 0);
    p.kb_total = static_cast<int>((K + kBK - 1) / kBK);
    const int max_s = p.kb_total < 32 ? p.kb_total : 32;
    auto tiles_of = [&](bool swap, int bn) {
        const int64_t rows = swap ? N : M, cols = swap ? M : N;
        return ((rows + kBM - 1) / kBM) * ((cols + bn - 1) / bn);
    };
    // Best split count of a tile shape, and its cost in K stages of that shape.
    // Wide tiles keep one split: their single accumulator buffer serialises a
    // split's epilogue with the next item's MMAs, and the measured split-K
    // runs were slower (2048 x 1536 x 7168: 44.6 us unsplit, 88.8 us in three;
    // 128 x 1536 x 7168: 35 us unsplit, 64 us in four).
    auto best_split = [&](bool swap, int bn, double* cost_out) {
        const int64_t tiles = tiles_of(swap, bn);
        const int max_split = (swap || forced > 0) ? max_s : 1;   // SGQ_SPLITS may still force one
        int best_s = 1;
        double best = 1e300;
        for (int s = 1; s <= max_split; ++s) {
            const int kbp = (p.kb_total + s - 1) / s;
            if ((p.kb_total + kbp - 1) / kbp != s) continue;   // every split non-empty
            const int64_t items = tiles * s;
            if (s > 1 && (size_t(tiles) > lim.counters ||
                          size_t(items) * kBM * bn * sizeof(float) > lim.partial_bytes))
                continue;
            const int64_t waves = (items + sm_count - 1) / sm_count;
            const double cost = double(waves) * (kbp + ovh) + (s > 1 ? 0.5 : 0.0);
            if (forced > 0 ? s == forced : cost < best) {
                best = cost;
                best_s = s;
            }
        }
        if (cost_out) *cost_out = best;
        return best_s;
    };
    p.swap = M <= swap_max;
    p.bn = p.swap ? (M <= 16 ? 16 : (M <= 32 ? 32 : 64)) : 256;
    // Mid M with few wide tiles (128 x 1536 x 7168: 6 tiles for 152 SMs):
    // swap-AB tiles of 64 tokens can split K where the wide tiles cannot.  A
    // 128 x 64 K stage (four N=64 MMAs, bound by their issue) takes about
    // 1/1.8 of a 128 x 256 one, 1/1.5 where the wide tiles run two alternating
    // issuers ([*,128], long K); the cheaper plan wins.
    if (!p.swap && !wide_only && mid_swap != 0 && M <= 1024) {
        double c_wide = 0.0, c_swap = 0.0;
        best_split(false, 256, &c_wide);
        best_split(true, 64, &c_swap);
        const double wide_stage = (blk_k == 128 && p.kb_total >= 32) ? 1.5 : 1.8;
        if (c_swap < wide_stage * c_wide) {
            p.swap = true;
            p.bn = 64;
        }
    }
    p.tiles_r = static_cast<int>(((p.swap ? N : M) + kBM - 1) / kBM);
    p.tiles_c = static_cast<int>(((p.swap ? M : N) + p.bn - 1) / p.bn);
    const int64_t tiles = int64_t(p.tiles_r) * p.tiles_c;
    const int best_s = best_split(p.swap, p.bn, nullptr);
    p.splits = best_s;
    p.kb_per_split = (p.kb_total + best_s - 1) / best_s;
    p.items = static_cast<int>(tiles * best_s);
    p.grid = p.items < sm_count ? p.items : sm_count;
    // Large M: pairs of CTAs can share 256 x 256 tiles, each loading half of
    // the weight tile, which cuts the operand bytes every SM pulls per FLOP by
    // a third.  Needs one split and TMA-loadable scale rows.  Off unless
    // SGQ_PAIR=1: with per-stage scale boxes the pair's stages are bound by
    // TMA operations per SM, not by bytes, and the single-CTA tiles are faster.
    static const int pair_on = env_int("SGQ_PAIR", 0);
    const int64_t ks = K / blk_k;
    p.pair = pair_on != 0 && !p.swap && p.splits == 1 && M > kBM && (ks % 4) == 0 &&
             ks >= (blk_k == 128 ? 8 : 16);   // the kernel's TMA scale-group path
    // Two alternating MMA issuers (one scale warp): measured faster for the
    // [*,128] recipe with long K (4096 x 7168 x 7168: 207 -> 185 us), slower for
    // [*,32] (the single scale warp's conversion then bounds the stage) and for
    // short K (per-tile costs dominate).  SGQ_ALT=0/1 forces it off/on.
    // Two K splits of a swap-AB tile can run as a cluster of two that sums
    // the partials in shared memory instead of through the global workspace.
    // Measured faster when a CTA takes several items (24576 x 1536 at M = 16:
    // 15.8 -> 13.2 us), level or slower with one item per CTA (7168 x 2048 at
    // M = 32: 9.85 -> 10.24 us).  SGQ_CK=0/1 forces it off/on.
    static const int ck_env = env_int("SGQ_CK", -1);
    const bool ck_ok = p.swap && p.splits == 2 && p.bn <= 32;
    p.ck = ck_ok && (ck_env < 0 ? p.items > p.grid : ck_env != 0);
    static const int alt_env = env_int("SGQ_ALT", -1);
    const bool alt_auto = blk_k == 128 && p.kb_total >= 32;
    p.alt = !p.swap && !p.pair && (alt_env < 0 ? alt_auto : alt_env != 0);
    if (p.pair) {
        p.tiles_r = static_cast<int>((M + 2 * kBM - 1) / (2 * kBM));
        p.items = p.tiles_r * p.tiles_c;
        const int pairs = p.items < sm_count / 2 ? p.items : sm_count / 2;
        p.grid = 2 * pairs;
    }
    return p;
}

// Address of the device status word on the current device.
uint32_t* g_status_ptr[64] = {};
std::mutex g_status_mu;

}  // namespace

sgq_status status_word(uint32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_status) != cudaSuccess) return SGQ_ERR_CUDA;
        g_status_ptr[dev] = static_cast<uint32_t*>(p);
    }
    *out = g_status_ptr[dev];
    return SGQ_OK;
}
}  // namespace gemm

namespace gemm {
namespace {

// Split-K scratch of the allocation-free entry point: a fixed file-scope
// array instead of the workspace that sgq_fp8_block_gemm allocates on first
// use.  Some callers cannot let a library allocate device memory (a serving
// engine that reserves nearly all of HBM for its own pool up front, or a host
// whose allocator must account for every byte).  The array is part of the
// module image, so every GPU that loads the library holds it until the
// process exits.
constexpr size_t kNoAllocCounterBytes = 16384 * sizeof(uint32_t);      // 64 KiB of counters
constexpr size_t kNoAllocPartialBytes = size_t(16) << 20;               // 16 MiB of partials
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocCounterBytes + kNoAllocPartialBytes];
unsigned char* g_noalloc_ptr[64] = {};
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device.  The host-side
// name is only a stand-in; the address is looked up once per device, with
// that device current.
sgq_status noalloc_scratch(unsigned char** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SGQ_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return SGQ_OK;
}

// Fused quantisation request: bf16 activations, the UE8M0 choice and the
// optional code / scale outputs.
struct Fuse {
    const void* x;
    int ue8m0;
    void* xq;
    float* xs;
};

// Per-channel scaling request (fp8_scaled_mm).
struct Chan {
    const float* sa;
    int64_t sa_n;
    const float* sb;
    int64_t sb_n;
    const void* bias;
};

// Tile width of the two-accumulator GEMM: 224 or 192 weight rows.  A K stage
// of either is bound by its operand bytes in flight (256 + BN rows of 128
// bytes), so the cost of a width is its rounds of tiles over the grid times
// that: 4096 x 7168 takes 192 (608 tiles: exactly 4 rounds of 152 SMs, where
// 224 makes 512 tiles, 3.4 rounds, so 4 of the longer stage; 168.6 vs 174.2
// us), 8192 x 24576 takes 224 (24 rounds against 27; 280 vs 294 us).
// pair: tiles of 512 rows over the SM pairs, each CTA holding 256 rows and BN / 2.
int dual_width(int64_t M, int64_t N, int sm_count, bool pair = false) {
    // SGQ_DUAL_BN=192/224 forces a width
    static const int forced = env_int("SGQ_DUAL_BN", 0);
    if (forced == dual::kBNNarrow || forced == dual::kBNWide) return forced;
    const int rows = pair ? 2 * dual::kRowsA : dual::kRowsA;
    const int units = pair ? sm_count / 2 : sm_count;
    const int64_t tr = (M + rows - 1) / rows;
    auto cost = [&](int bn) {
        const int64_t tiles = tr * ((N + bn - 1) / bn);
        return ((tiles + units - 1) / units) * (rows + bn);
    };
    return cost(dual::kBNNarrow) < cost(dual::kBNWide) ? dual::kBNNarrow : dual::kBNWide;
}

// K splits of the two-accumulator tiles.  Where the tiles alone leave SMs
// idle, each tile's K stages are dealt out to several CTAs of one wave (one
// item per CTA: the kernel stages the partials in its idle operand ring),
// which then sum their fp32 partials in split order (deterministic).  Cost of s
// splits, in K-stage times: ceil(kst / s) stages plus, for s > 1, the partial
// exchange (each CTA stores a 256 x BN fp32 tile and reads as much back,
// about four stages' time); the smallest s with the least cost is taken.
// SGQ_DUAL_SPLITS forces a count.
int dual_splits(int64_t tiles, int kst, int sm_count, int bn, ScratchLimit lim) {
    static const int forced = env_int("SGQ_DUAL_SPLITS", 0);
    auto fits = [&](int sp) {
        const size_t per = 8u * size_t((bn / 4 + sp - 1) / sp);
        return size_t(tiles) * size_t(sp) * size_t(sp) * per * 512u <= lim.partial_bytes &&
               tiles <= kDualCounters && sp <= 16 && dual::red_need(bn, sp) <= dual::kRedArea;
    };
    int best = 1;
    if (forced > 0) {
        best = forced < kst ? forced : kst;
        while (best > 1 && tiles * best > sm_count) --best;   // one item per CTA (the kernel's rule)
    } else {
        int64_t best_cost = kst;
        for (int sp = 2; sp <= 16 && sp <= kst && tiles * sp <= sm_count; ++sp) {
            if (!fits(sp)) continue;
            const int64_t cost = (kst + sp - 1) / sp + 4;
            if (cost < best_cost) {
                best_cost = cost;
                best = sp;
            }
        }
    }
    // within the scratch and shared memory, every split non-empty:
    // (splits - 1) * ceil(kst / splits) < kst
    while (best > 1 && (!fits(best) || int64_t(best - 1) * ((kst + best - 1) / best) >= kst)) --best;
    return best;
}

// Launch plan of the two-accumulator prefill GEMM (power-of-two scales):
// tiles of 256 activation rows (512 on CTA pairs) x BN weight rows over a
// persistent grid of at most one CTA per SM (pair), with K split over several
// CTAs where the tiles are fewer than the SMs (allow_split: the split-K
// workspace may be used; single CTAs only).
struct DualPlan {
    int bn, rows, tiles_r, tiles_c, kst, tiles, splits, kps, items, per, grid;
};
DualPlan plan_dual(int64_t M, int64_t N, int64_t K, int sm_count, bool allow_split, bool pair, ScratchLimit lim) {
    DualPlan q{};
    q.bn = dual_width(M, N, sm_count, pair);
    q.rows = pair ? 2 * dual::kRowsA : dual::kRowsA;
    q.tiles_r = static_cast<int>((M + q.rows - 1) / q.rows);
    q.tiles_c = static_cast<int>((N + q.bn - 1) / q.bn);
    q.kst = static_cast<int>(K / kBK);
    q.tiles = q.tiles_r * q.tiles_c;
    const int units = pair ? sm_count / 2 : sm_count;
    q.splits = allow_split && !pair ? dual_splits(q.tiles, q.kst, sm_count, q.bn, lim) : 1;
    q.kps = (q.kst + q.splits - 1) / q.splits;
    q.items = q.tiles * q.splits;
    q.per = 8 * ((q.bn / 4 + q.splits - 1) / q.splits);
    q.grid = (q.items < units ? q.items : units) * (pair ? 2 : 1);
    return q;
}

// Launches the two-accumulator prefill GEMM on plan_dual's plan.
// Ae/We: UE8M0 scale bytes in place of As/Ws (both given or both null).
sgq_status launch_dual(const void* Aq, const float* As, const void* Wq, const float* Ws, void* D, int64_t M,
                       int64_t N, int64_t K, int blk_n, int blk_k, int sm_count, bool allow_split, bool pair,
                       ScratchLimit lim, cudaStream_t st, const uint8_t* Ae = nullptr, const uint8_t* We = nullptr) {
    const DualPlan q = plan_dual(M, N, K, sm_count, allow_split, pair, lim);
    const int bn = q.bn;
    dual::DualArgs a{};
    a.As = As;
    a.Ws = Ws;
    a.Ae = Ae;
    a.We = We;
    const bool e8 = Ae != nullptr;
    a.D = static_cast<__nv_bfloat16*>(D);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.ks = static_cast<int>(K / blk_k);
    a.tiles_r = q.tiles_r;
    a.tiles_c = q.tiles_c;
    a.kst = q.kst;
    a.tiles = q.tiles;
    a.group_r = a.tiles_r < 16 ? a.tiles_r : 16;
    a.splits = q.splits;
    a.kps = q.kps;
    a.items = q.items;
    a.per = q.per;
    sgq_status rc = status_word(&a.status);
    if (rc != SGQ_OK) return rc;
    if (a.splits > 1) {
        DevWs ws;
        rc = get_workspace(st, &ws);
        if (rc != SGQ_OK) return rc;
        a.partial = ws.partial;
        a.counters = ws.counters + (kMaxCounters - kDualCounters);
    }
    CUtensorMap maps[2];
    if (make_tmap(&maps[0], Aq, M, K, dual::kRowsA) != SGQ_OK ||
        make_tmap(&maps[1], Wq, N, K, pair ? bn / 2 : bn) != SGQ_OK)
        return SGQ_ERR_CUDA;
    if (pair) return dual::dispatch(bn, dual::kPairs, e8, blk_n, blk_k, maps[0], maps[1], a, q.grid, st);
    return dual::dispatch(bn, a.splits > 1 ? dual::kSplitK : dual::kPlain, e8, blk_n, blk_k, maps[0], maps[1], a,
                          q.grid, st);
}

// Whether a GEMM with the power-of-two promise runs on the two-accumulator
// tiles: 0 no, 1 yes with one K split, 2 yes with the K splits dual_splits
// chooses.  Rules, from timings on GB300 (CUDA graphs of 20 calls, weights
// from HBM; SGQ_DUAL=0/1 forces the choice):
// - a wave of 256 x 224 tiles or more (and not a swap-AB plan): always
//   (4096 x 7168 x 7168: 168.6 vs 174.2 us on the 128 x 256 tiles);
// - M >= 128 and at least 0.6 of a wave: one split (700 x 7168 x 2048:
//   19.7 vs 28.2 us; 128 x 24576 x 1536: 14.7 vs 16.9 us);
// - M >= 768 with fewer tiles: K splits, where the split plan's estimate,
//   0.8 us per K stage of a split plus ~2.5 us of pipeline fill plus ~9 us of
//   partial exchange, is under 1/1.3 of the 128 x 256 tiles' estimate, rounds
//   x (0.5 us per K stage + 3 us) (1024 x 1536 x 7168: 25.3 vs 36.7 us; at
//   2048 x 1536 x 7168 and at M <= 512 the split plans measured no faster).
int dual_mode(int64_t M, int64_t N, int64_t K, int blk_k, uint32_t flags, const Plan& p, int sm_count,
              ScratchLimit lim, bool e8 = false) {
    static const int dual_env = env_int("SGQ_DUAL", -1);
    if (!(flags & SGQ_GEMM_SCALES_POW2) || K % kBK != 0 || M <= 64 ||
        (flags & (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE)) != 0)
        return 0;
    // SGQ_DUAL_PAIR=0/1 forces CTA pairs off/on for the wave-sized plans
    static const int pair_env = env_int("SGQ_DUAL_PAIR", -1);
    if (dual_env >= 0) return dual_env == 0 ? 0 : (pair_env > 0 ? 3 : 2);
    const int64_t tr = (M + dual::kRowsA - 1) / dual::kRowsA;
    const int64_t dual_tiles = tr * ((N + dual::kBNWide - 1) / dual::kBNWide);
    // A wave of tiles: CTA pairs with long K where a stage's scale work is
    // light -- fp32 scales with the [*,128] recipe (4096 x 7168 x 7168: 159.3
    // vs 167.9 us) and UE8M0 bytes with either recipe (4096 x 4096 x 7168
    // [*,32]: 85.0 vs 89.5 us; 4096 x 7168 x 7168 [*,128]: 155.0 vs 160.8 us).
    // The pair's longer per-stage handshake loses on short K (8192 x 24576 x
    // 1536 [*,32]: 333 vs 308 us) and with fp32 [*,32] scales (4096 x 4096 x
    // 7168: 105 vs 100 us).
    if (!p.swap && dual_tiles >= sm_count) {
        const bool pair_auto = K >= 4096 && (e8 || blk_k == 128);
        return pair_env > 0 || (pair_env < 0 && pair_auto) ? 3 : 1;
    }
    if (M >= 128 && dual_tiles * 5 >= int64_t(sm_count) * 3) return 1;
    if (M < 768) return 0;
    const int bn = dual_width(M, N, sm_count);
    const int64_t tiles = tr * ((N + bn - 1) / bn);
    const int kst = static_cast<int>(K / kBK);
    const int sp = dual_splits(tiles, kst, sm_count, bn, lim);
    if (sp < 2) return 0;
    const double est_dual = 0.8 * ((kst + sp - 1) / sp) + 2.5 + 9.0;
    const int64_t t128 = ((M + kBM - 1) / kBM) * ((N + 255) / 256);
    const double est_wide = double((t128 + sm_count - 1) / sm_count) * (0.5 * kst + 3.0);
    return est_wide > 1.3 * est_dual ? 2 : 0;
}

// Plans and launches one GEMM.  noalloc: split-K scratch from the fixed array
// (its counters cleared by an asynchronous memset), else the per-device
// workspace.  fuse (Aq/As unused): the activations are quantised inside the
// GEMM when the plan is a swap-AB one with TMA-loadable weight scales, else
// SGQ_ERR_UNSUPPORTED is returned before anything is launched.
sgq_status launch(const void* Aq, const float* As, const void* Wq, const float* Ws, void* D, int64_t M,
                  int64_t N, int64_t K, int blk_n, int blk_k, uint32_t flags, bool noalloc, const Fuse* fuse,
                  cudaStream_t st, const Chan* chan = nullptr) {
    if (get_encoder() != SGQ_OK) return SGQ_ERR_CUDA;
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    if (di.cc_major != 10 || di.cc_minor != 3) return SGQ_ERR_UNSUPPORTED;
    // The allocation-free entry point plans within its fixed array: split
    // counts whose partials or counters would not fit are skipped, so such a
    // shape runs with fewer K splits (or, at mid M, on the 128 x 256 tiles
    // that need no split-K) instead of being refused.
    const ScratchLimit lim =
        noalloc ? ScratchLimit{kNoAllocPartialBytes, kNoAllocCounterBytes / sizeof(uint32_t)} : kWsLimit;
    Plan p = make_plan(M, N, K, blk_k, di.sm_count, (flags & (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE)) != 0,
                       lim);
    // Power-of-two scales promised by the caller: the two-accumulator tiles
    // (gemm_dual.cuh, K in whole stages, M > 64) where they are measured
    // faster than this plan.
    if (int mode = dual_mode(M, N, K, blk_k, flags, p, di.sm_count, lim);
        mode != 0 && !fuse && !chan)
        return launch_dual(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, di.sm_count, mode == 2 && !noalloc, mode == 3,
                           lim, st);
    if (flags & SGQ_GEMM_ISSUE_ALT) p.alt = !p.swap && !p.pair;
    if (flags & SGQ_GEMM_ISSUE_SINGLE) p.alt = false;
    if (chan) {   // plain tiles: no scale boxes, one issuer
        p.alt = false;
        p.pair = false;
    }
    const int64_t ks_all = K / blk_k;
    const bool scale_tma_ok = (ks_all % 4) == 0 && ks_all >= (blk_k == 128 ? 8 : 16);
    // fused quantisation: swap-AB tiles of at most 64 tokens (the documented domain)
    if (fuse && !(p.swap && M <= 64 && scale_tma_ok)) return SGQ_ERR_UNSUPPORTED;
    GemmArgs a{};
    a.As = As;
    a.Ws = Ws;
    a.D = static_cast<__nv_bfloat16*>(D);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.ks = static_cast<int>(K / blk_k);
    a.rows = static_cast<int>(p.swap ? N : M);
    a.cols = static_cast<int>(p.swap ? M : N);
    a.tiles_r = p.tiles_r;
    a.tiles_c = p.tiles_c;
    a.kb_total = p.kb_total;
    a.kb_per_split = p.kb_per_split;
    a.splits = p.splits;
    a.items = p.items;
    a.group_r = 16;
    static const int prefetch = env_int("SGQ_PREFETCH", -1);
    a.prefetch = prefetch;
    a.force_promote = (flags & SGQ_GEMM_FORCE_PROMOTE) ? 1 : 0;
    ExtArgs fz{};
    fz.stall_job = (flags & SGQ_GEMM_TEST_TIMEOUT) ? 5 : -1;
    if (chan) {
        fz.sa = chan->sa;
        fz.sb = chan->sb;
        fz.sa_n = static_cast<int>(chan->sa_n);
        fz.sb_n = static_cast<int>(chan->sb_n);
        fz.bias = static_cast<const uint16_t*>(chan->bias);
    }
    if (fuse) {
        fz.x = static_cast<const uint16_t*>(fuse->x);
        fz.ue8m0 = fuse->ue8m0;
        fz.xq_out = static_cast<uint8_t*>(fuse->xq);
        fz.xs_out = fuse->xs;
    }
    rc = status_word(&a.status);
    if (rc != SGQ_OK) return rc;
#ifdef SGQ_TRACE
    {
        void* tp = nullptr;
        if (cudaGetSymbolAddress(&tp, g_gemm_trace) != cudaSuccess) return SGQ_ERR_CUDA;
        a.trace = static_cast<unsigned long long*>(tp);
    }
#endif
    if (p.splits > 1) {
        if (noalloc) {
            const size_t tiles = size_t(p.tiles_r) * size_t(p.tiles_c);
            const size_t part_bytes = size_t(p.items) * kBM * size_t(p.bn) * sizeof(float);
            if (tiles * sizeof(uint32_t) > kNoAllocCounterBytes || part_bytes > kNoAllocPartialBytes)
                return SGQ_ERR_UNSUPPORTED;   // needs more scratch than the fixed array holds
            unsigned char* base = nullptr;
            rc = noalloc_scratch(&base);
            if (rc != SGQ_OK) return rc;
            a.counters = reinterpret_cast<uint32_t*>(base);
            a.partial = reinterpret_cast<float*>(base + kNoAllocCounterBytes);
            // The array keeps the previous call's contents; the counters must
            // start at zero (a call that ended early may have left some set).
            if (cudaMemsetAsync(a.counters, 0, tiles * sizeof(uint32_t), st) != cudaSuccess) return SGQ_ERR_CUDA;
        } else {
            DevWs ws;
            rc = get_workspace(st, &ws);
            if (rc != SGQ_OK) return rc;
            a.partial = ws.partial;
            a.counters = ws.counters;
        }
    }
    // maps: A operand, B operand, A-operand scales, B-operand scales
    CUtensorMap maps[4];
    const void* opA = p.swap ? Wq : Aq;
    const void* opB = p.swap ? Aq : Wq;
    if (make_tmap(&maps[0], opA, a.rows, K, kBM) != SGQ_OK) return SGQ_ERR_CUDA;
    if (fuse) {
        maps[1] = maps[0];   // the activations are read by the kernel's threads, not by TMA
    } else if (make_tmap(&maps[1], opB, a.cols, K, p.pair ? p.bn / 2 : p.bn) != SGQ_OK) {
        return SGQ_ERR_CUDA;
    }
    // Scale rows are TMA-loadable when their pitch is a multiple of 16 bytes
    // and they are at least one box (one group of K stages) wide: a box wider
    // than the matrix's rows is not used.
    static const int scale_tma_on = env_int("SGQ_SCALE_TMA", 1);
    const int gcols = blk_k == 128 ? 8 : 16;
    const bool scale_tma = !chan && (scale_tma_on != 0 || fuse) && (a.ks % 4) == 0 && a.ks >= gcols;
    maps[2] = maps[0];
    maps[3] = maps[1];
    if (scale_tma) {
        const int64_t nb = (N + blk_n - 1) / blk_n;
        // one box = the scales of a group of four K stages (see the kernel)
        if (make_scale_map(&maps[2], p.swap ? Ws : As, p.swap ? nb : M, a.ks, p.swap ? kBM / blk_n : kBM,
                           gcols) != SGQ_OK ||
            (!fuse && make_scale_map(&maps[3], p.swap ? As : Ws, p.swap ? M : nb, a.ks,
                                     p.swap ? p.bn : p.bn / blk_n, gcols) != SGQ_OK))
            return SGQ_ERR_CUDA;
    }
    const Variant v{p.swap, p.pair, p.alt, scale_tma, fuse != nullptr, chan != nullptr,
                    p.ck && !fuse && !chan, p.bn};
    if (chan) return dispatch_chan(v, maps, a, fz, p.grid, st);
    if (blk_n == 32 && blk_k == 32) return dispatch_32_32(v, maps, a, fz, p.grid, st);
    if (blk_n == 32 && blk_k == 128) return dispatch_32_128(v, maps, a, fz, p.grid, st);
    if (blk_n == 128 && blk_k == 32) return dispatch_128_32(v, maps, a, fz, p.grid, st);
    return dispatch_128_128(v, maps, a, fz, p.grid, st);
}

// Widened fp32 copies of UE8M0 scale bytes, for the plans that read fp32
// scales (one buffer per device, grown on demand outside stream capture).
struct WideScales {
    float* p = nullptr;
    size_t bytes = 0;
};
WideScales g_wide[64];
std::mutex g_wide_mu;

sgq_status wide_scales(size_t bytes, cudaStream_t st, float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_wide_mu);
    WideScales& w = g_wide[dev];
    if (w.bytes < bytes) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return SGQ_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return SGQ_ERR_UNSUPPORTED;
        size_t cap = size_t(1) << 20;
        while (cap < bytes) cap <<= 1;
        if (w.p) {
            if (cudaDeviceSynchronize() != cudaSuccess) return SGQ_ERR_CUDA;   // no launch still reads it
            cudaFree(w.p);
            w.p = nullptr;
            w.bytes = 0;
        }
        void* p = nullptr;
        if (cudaMalloc(&p, cap) != cudaSuccess) return SGQ_ERR_CUDA;
        w.p = static_cast<float*>(p);
        w.bytes = cap;
    }
    *out = w.p;
    return SGQ_OK;
}

// UE8M0 scale bytes: the two-accumulator tiles read them as they are where
// their rules take the shape; other plans get fp32 copies (2^(e - 127)) in a
// library buffer first, then run as sgq_fp8_block_gemm_ex with the
// power-of-two promise.
sgq_status launch_ue8m0(const void* Aq, const uint8_t* Ae, const void* Wq, const uint8_t* We,
                                       void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                       uint32_t flags, cudaStream_t st) {
    if (M == 0) return SGQ_OK;
    if (get_encoder() != SGQ_OK) return SGQ_ERR_CUDA;
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    if (di.cc_major != 10 || di.cc_minor != 3) return SGQ_ERR_UNSUPPORTED;
    flags |= SGQ_GEMM_SCALES_POW2;
    const Plan p = make_plan(M, N, K, blk_k, di.sm_count, (flags & (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE)) != 0);
    const int mode = dual_mode(M, N, K, blk_k, flags, p, di.sm_count, kWsLimit, true);
    if (mode != 0 && (flags & SGQ_GEMM_FORCE_PROMOTE) == 0)
        return launch_dual(Aq, nullptr, Wq, nullptr, D, M, N, K, blk_n, blk_k, di.sm_count, mode == 2, mode == 3,
                           kWsLimit, st, Ae, We);
    const int64_t ks = K / blk_k, nb = (N + blk_n - 1) / blk_n;
    const size_t na = size_t(M) * size_t(ks), nw = size_t(nb) * size_t(ks);
    float* wide = nullptr;
    rc = wide_scales((na + nw) * sizeof(float), st, &wide);
    if (rc != SGQ_OK) return rc;
    rc = launch_ue8m0_to_scales(Ae, int64_t(na), wide, st);
    if (rc == SGQ_OK) rc = launch_ue8m0_to_scales(We, int64_t(nw), wide + na, st);
    if (rc != SGQ_OK) return rc;
    return launch(Aq, wide, Wq, wide + na, D, M, N, K, blk_n, blk_k, flags, false, nullptr, st);
}

}  // namespace
}  // namespace gemm

sgq_status launch_fp8_block_gemm(const void* Aq, const float* As, const void* Wq, const float* Ws,
                                 void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                 uint32_t flags, cudaStream_t st) {
    return gemm::launch(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, flags, false, nullptr, st);
}

sgq_status launch_fp8_block_gemm_ue8m0(const void* Aq, const uint8_t* Ae, const void* Wq, const uint8_t* We,
                                       void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                       uint32_t flags, cudaStream_t st) {
    return gemm::launch_ue8m0(Aq, Ae, Wq, We, D, M, N, K, blk_n, blk_k, flags, st);
}

// The launch plan of launch_fp8_block_gemm, except where that plan's split-K
// partials would not fit the fixed array: then fewer K splits (or the 128 x
// 256 tiles) are used, and D agrees with the default entry point's within the
// GEMM tolerance rather than bit for bit.
sgq_status launch_fp8_block_gemm_noalloc(const void* Aq, const float* As, const void* Wq, const float* Ws,
                                         void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                         cudaStream_t st) {
    return gemm::launch(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, SGQ_GEMM_DEFAULT, true, nullptr, st);
}

// fp8_scaled_mm: D = (Aq Wq^T) * sa * sb + bias.  The plan is the block GEMM's
// for blk_k = 128 (the scale arguments of the block path stay unused).
sgq_status gemm_plan_query(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int32_t* out) {
    const gemm::Plan p = gemm::make_plan(M, N, K, blk_k, sm_count);
    const int32_t v[8] = {p.swap ? 1 : 0, p.bn, p.splits, p.items, p.grid, p.alt ? 1 : 0, p.ck ? 1 : 0,
                          p.pair ? 1 : 0};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
    return SGQ_OK;
}

sgq_status gemm_plan_pow2_query(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int e8, int32_t* out) {
    const gemm::Plan p = gemm::make_plan(M, N, K, blk_k, sm_count);
    const int mode = gemm::dual_mode(M, N, K, blk_k, SGQ_GEMM_SCALES_POW2, p, sm_count, gemm::kWsLimit, e8 != 0);
    for (int i = 0; i < 8; ++i) out[i] = 0;
    out[0] = mode;
    if (mode == 0) return SGQ_OK;
    const gemm::DualPlan q = gemm::plan_dual(M, N, K, sm_count, mode == 2, mode == 3, gemm::kWsLimit);
    const int32_t v[6] = {q.bn, q.splits, q.items, q.grid, q.tiles, q.kps};
    for (int i = 0; i < 6; ++i) out[i + 1] = v[i];
    return SGQ_OK;
}

sgq_status launch_fp8_scaled_mm(const void* Aq, const float* sa, int64_t sa_n, const void* Wq, const float* sb,
                                int64_t sb_n, const void* bias, void* D, int64_t M, int64_t N, int64_t K,
                                cudaStream_t st) {
    const gemm::Chan c{sa, sa_n, sb, sb_n, bias};
    return gemm::launch(Aq, nullptr, Wq, nullptr, D, M, N, K, 128, 128, SGQ_GEMM_DEFAULT, false, nullptr, st, &c);
}

// Quantise-and-multiply.  With xq/xs given: the quantisation kernel into
// them, then the GEMM (the faster path: every weight-tile CTA of the single
// kernel re-quantises its share of the activations; measured at N=7168,
// K=2048: 10.7 vs 9.7 us per linear at M=16, 18.5 vs 12.5 us at M=64).
// Without them, decode-sized M (swap-AB plans with TMA-loadable weight
// scales) runs one kernel that quantises its activation tiles itself; any
// other shape is unsupported.
sgq_status launch_fp8_block_linear(const void* x, int ue8m0, const void* Wq, const float* Ws, void* D, int64_t M,
                                   int64_t N, int64_t K, int blk_n, int blk_k, void* xq, float* xs,
                                   cudaStream_t st) {
    const bool prefer_pair = xq && xs;
    const gemm::Fuse f{x, ue8m0, xq, xs};
    const sgq_status rc =
        prefer_pair ? SGQ_ERR_UNSUPPORTED
                    : gemm::launch(nullptr, nullptr, Wq, Ws, D, M, N, K, blk_n, blk_k, SGQ_GEMM_DEFAULT, false, &f, st);
    if (rc != SGQ_ERR_UNSUPPORTED) return rc;
    if (!xq || !xs) return SGQ_ERR_UNSUPPORTED;
    const sgq_status q = launch_quant_token_group(x, M, K, blk_k, ue8m0, xq, xs, st);
    if (q != SGQ_OK) return q;
    return launch_fp8_block_gemm(xq, xs, Wq, Ws, D, M, N, K, blk_n, blk_k, SGQ_GEMM_DEFAULT, st);
}

uint64_t allocated_bytes() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    uint64_t b = 0;
    {
        std::lock_guard<std::mutex> lk(gemm::g_ws_mu);
        if (gemm::g_ws[dev].partial) b += uint64_t(gemm::kWsBytes) + gemm::kMaxCounters * sizeof(uint32_t);
    }
    std::lock_guard<std::mutex> lk(gemm::g_wide_mu);
    return b + gemm::g_wide[dev].bytes;
}

sgq_status read_and_clear_device_status(cudaStream_t st) {
    if (cudaStreamSynchronize(st) != cudaSuccess) return SGQ_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(v)) != cudaSuccess) return SGQ_ERR_CUDA;
    if (v == 0) return SGQ_OK;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(zero)) != cudaSuccess) return SGQ_ERR_CUDA;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && gemm::g_ws[dev].counters) {
        // an aborted split-K launch may have left arrival counts behind
        if (cudaMemset(gemm::g_ws[dev].counters, 0, gemm::kMaxCounters * sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return SGQ_ERR_CUDA;
    }
    if (v & gemm::kStatusTimeout) return SGQ_ERR_TIMEOUT;
    return (v & dual::kStatusBadScale) ? SGQ_ERR_INVALID_ARG : SGQ_ERR_CUDA;
}

}  // namespace sgq

#ifdef SGQ_TRACE
// Development builds only: copies the per-CTA event trace of the last GEMM.
extern "C" int sgq_trace_read(void* host, uint64_t bytes) {
    if (bytes > sizeof(unsigned long long) * 1024 * sgq::gemm::kTraceSlots) return 1;
    return cudaMemcpyFromSymbol(host, sgq::g_gemm_trace, bytes) == cudaSuccess ? 0 : 4;
}
extern "C" int sgq_trace_clear(void) {
    static unsigned long long zeros[1024 * sgq::gemm::kTraceSlots];
    return cudaMemcpyToSymbol(sgq::g_gemm_trace, zeros, sizeof(zeros)) == cudaSuccess ? 0 : 4;
}
#endif
