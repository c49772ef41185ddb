// Prefill-sized block-scaled FP8 GEMM for sm_103a with power-of-two (UE8M0)
// scales: D = (Aq * As)(Wq * Ws)^T, fp32 accumulation, bf16 out.
//
// The operation is the one of gemm_kernel.cuh (vLLM "scaled_mm" API page,
// AiterInt8ScaledMMLinearKernel.apply_weights docstring, in the "NT" layout of
// sglang PR #42604, Modifications: fp8_gemm_nt((Aq, As), (Wq, Ws), D,
// recipe=(1, blk_n, blk_k))), for the case the PR's path uses -- every scale a
// power of two -- so that all scales go through the block-scaled MMA
// (kind::mxf8f6f4, one UE8M0 factor per row per 32-wide K chunk).
//
// Why a tile of 256 activation rows x BN weight rows with two accumulators:
// one 128 x 256 x 32 MMA keeps an SM's tensor core busy ~70 ns, so a 128-row
// tile needs its 48 KB per 128-wide K stage every ~280 ns -- more than the
// ~120 GB/s an SM pulls from L2.  Two 128-row halves sharing one weight tile
// need 60 KB per ~520 ns of MMA work (BN = 224), under that rate, and each
// half has its own issuing warp and TMEM accumulator (2 x BN columns, plus the
// scale factors: TMEM's 512 columns hold no second buffer, so a tile's
// epilogue does not overlap the next tile's first MMAs).
//
// Warps: 0 producer (TMA: the 256 x 128 activation box and the BN x 128 weight
// box per K stage, 3-stage ring), 1 and 2 MMA issuers (half 0 / half 1),
// 3 and 12 scale warps (UE8M0 words of half h's activation rows and of half
// of the weight rows, loaded ahead with plain loads), 4-11 epilogue (two warps
// per TMEM lane quadrant, half of the columns each).  Every wait is bounded;
// on time-out the CTA records a status word and leaves through the normal
// teardown.  A scale that is not a power of two sets a status bit instead of
// being applied (the caller promised power-of-two scales).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"
#include "sgq_internal.h"

namespace sgq {
namespace dual {

constexpr int kHalf = 128;                 // activation rows per half (MMA M)
constexpr int kRowsA = 2 * kHalf;          // activation rows per tile
constexpr int kBK = 128;                   // K bytes per stage
constexpr int kStages = 3;
constexpr int kWarps = 13;
constexpr int kThreads = 32 * kWarps;
constexpr int kEpi0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 1ull << 30;
constexpr uint64_t kAbortPollNs = 20000;
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusBadScale = 2u;

struct DualArgs {
    const float* As;        // fp32 [M, K / blk_k]
    const float* Ws;        // fp32 [ceil(N / blk_n), K / blk_k]
    const uint8_t* Ae;      // kE8: UE8M0 bytes [M, K / blk_k] (in place of As)
    const uint8_t* We;      // kE8: UE8M0 bytes [ceil(N / blk_n), K / blk_k] (in place of Ws)
    __nv_bfloat16* D;       // bf16 [M, N]
    uint32_t* status;       // device status word
    float* partial;         // splits > 1: one fp32 partial tile per item (splits * per * 128 floats)
    uint32_t* counters;     // splits > 1: one arrival count per tile, a multiple of 16 between launches
    int M, N, K, ks;        // ks = K / blk_k
    int tiles_r, tiles_c, kst, tiles, group_r;
    int splits, kps, items; // K splits per tile (<= 16), K stages per split (every split non-empty), tiles x splits
    int per;                // splits > 1: warp units (32 x 4 floats) per slice stride, 8 * ceil(BN / 4 / splits)
};

// Split-K exchange: shared memory for the slices a CTA receives from the
// other splits plus its staged slice of D.  The host takes only split counts
// whose (splits - 1) * 8 * ceil(BN / 4 / splits) units of 512 bytes and
// 256 rows of 8 * ceil(BN / 4 / splits) + 8 bytes fit in it.
constexpr int kRedArea = 212 * 1024;
constexpr int red_need(int bn, int splits) {
    const int ngmax = (bn / 4 + splits - 1) / splits;
    return (splits - 1) * 8 * ngmax * 512 + 256 * (8 * ngmax + 8);
}

// UE8M0 words (tcgen05.cp order) of one stage: half h's 128 activation rows,
// and the weight rows (two 128-row copies).
struct alignas(128) Slot {
    uint32_t sfa[2][128];
    uint32_t sfb[256];
};

template <int BN, bool kSplit, bool kPair = false>
struct Cfg {
    // kPair: a cluster of two CTAs shares a tile of 512 activation rows (256
    // per CTA, as two 128-row halves) x BN weight rows (BN / 2 per CTA); the
    // leader issues M = 256 MMAs over both CTAs' halves (.cta_group::2).
    static constexpr int kSt = kPair ? 4 : kStages;           // ring stages
    static constexpr int kABytes = kRowsA * kBK;
    static constexpr int kBBytes = (kPair ? BN / 2 : BN) * kBK;
    static constexpr size_t kOffA = 0;
    static constexpr size_t kOffB = kOffA + size_t(kSt) * kABytes;
    static constexpr int kRingBytes = kSt * (kABytes + kBBytes);
    // Split-K launches also hold the exchange area: the other splits' slices
    // of the partial tile land over the operand ring (idle once a CTA's only
    // item is accumulated) and past it.  Other launches stop at the ring, so
    // the SM keeps more of its L1 (the scale warps read through it).
    static constexpr size_t kAreaEnd = size_t(kSplit && kRedArea > kRingBytes ? kRedArea : kRingBytes);
    static constexpr size_t kOffSlot = kAreaEnd;
    // barriers: full[kSt], empty[kSt], accf[2], acce[2], drain[2], red
    static constexpr size_t kOffBar = kOffSlot + size_t(kSt) * sizeof(Slot);
    static constexpr int kNumBars = 2 * kSt + 7;
    static constexpr size_t kOffMisc = kOffBar + 8 * kNumBars;
    // pair: 16-byte signal buffers of the peer's two scale warps
    static constexpr size_t kOffXfer = (kOffMisc + 64 + 15) & ~size_t(15);
    // misc: 8 words (and, split-K, the 17 slice bounds), then alignment slack
    static constexpr size_t kSmem = (kPair ? kOffXfer + 32 : kOffMisc + (kSplit ? 128 : 64)) + 1024;
    // TMEM: accumulator h at columns [h*BN, (h+1)*BN), then two scale slots
    // of 16 columns per issuer (A words at +0, B words at +4 .. +11)
    static constexpr uint32_t kSfCol = 2u * BN;
    static_assert(BN % 16 == 0 && BN <= 256 && BN > 128, "MMA N (two B scale copies)");
    static_assert(kSfCol + 64u <= kTmemCols, "TMEM: two accumulators and the scale slots");
    static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0, "128-byte swizzle atoms");
    static_assert(kOffSlot % 128 == 0, "scale slots aligned");
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(!(kSplit && kPair), "split-K runs on single-CTA tiles");
    static constexpr int kColsPerWarp = BN / 2;       // epilogue: two warps per lane quadrant
    static_assert(kColsPerWarp % 16 == 0, "16-column epilogue chunks");
};

struct Sync {
    volatile uint32_t* abort_flag;
    uint32_t* status;
};

// kCl: the barrier also receives arrivals from the other CTA of a pair
// (acquire at cluster scope).
template <bool kCl = false>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    if constexpr (kCl) return ptx::mbar_try_wait_cluster(bar, parity);
    else return ptx::mbar_try_wait(bar, parity);
}
template <bool kCl = false>
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (try_wait_scoped<kCl>(bar, parity)) return true;
        if ((++spins & 15u) == 0) {
            const uint64_t dt = ptx::globaltimer() - t0;
            if (dt > kAbortPollNs && *s.abort_flag) return false;
            if (dt > kTimeoutNs) {
                *s.abort_flag = 1u;
                atomicOr(s.status, kStatusTimeout | (where << 8));
                return false;
            }
        }
        if (spins > 8) __nanosleep(32);
    }
}
template <bool kCl = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    uint32_t ok = 1;
    if ((threadIdx.x & 31) == 0 && !try_wait_scoped<kCl>(bar, parity))
        ok = wait_slow<kCl>(bar, parity, s, where) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// UE8M0 word of one scale row: byte q = exponent field of chunk q's scale
// (one scale per stage: repeated); `bad` collects scales that are not
// positive normal powers of two.
__device__ __forceinline__ uint32_t zero_byte(uint32_t w) { return (w - 0x01010101u) & ~w & 0x80808080u; }
template <int kSps>
__device__ __forceinline__ uint32_t sf_word(const float4& v, uint32_t& bad) {
    if constexpr (kSps == 1) {
        const uint32_t b = __float_as_uint(v.x);
        const uint32_t w = __byte_perm(b << 1, 0u, 0x3333);
        bad |= (b & 0x807FFFFFu) | zero_byte(w) | zero_byte(~w);
        return w;
    } else {
        const uint32_t x = __float_as_uint(v.x), y = __float_as_uint(v.y), z = __float_as_uint(v.z),
                       q = __float_as_uint(v.w);
        const uint32_t lo = __byte_perm(x << 1, y << 1, 0x0073);
        const uint32_t hi = __byte_perm(z << 1, q << 1, 0x0073);
        const uint32_t w = __byte_perm(lo, hi, 0x5410);
        bad |= ((x | y | z | q) & 0x807FFFFFu) | zero_byte(w) | zero_byte(~w);
        return w;
    }
}
template <int kSps>
__device__ __forceinline__ float4 load_scales(const float* p) {
    if constexpr (kSps == 4) return __ldg(reinterpret_cast<const float4*>(p));
    else return make_float4(__ldg(p), 0.0f, 0.0f, 0.0f);
}

// Tile t -> (row tile, column tile): column-major inside groups of group_r
// row tiles, so the CTAs of one wave share weight tiles and activation rows.
__device__ __forceinline__ void tile_coords(const DualArgs& a, int t, int& tr, int& tc) {
    const int per_group = a.group_r * a.tiles_c;
    const int g = t / per_group;
    const int first = g * a.group_r;
    const int gm = min(a.tiles_r - first, a.group_r);
    const int in = t - g * per_group;
    tr = first + in % gm;
    tc = in / gm;
}

// Work item i = (tile i / splits, K split i % splits): K stages [kb0, kb1).
// The splits of a tile are consecutive items, so with one item per CTA they
// run at the same time on neighbouring CTAs.
struct Item {
    int t, sp, tr, tc, kb0, kb1;
};
// (The scale warps ask once per K stage: nothing to compute without split-K.)
template <bool kSplit>
__device__ __forceinline__ int item_tile(const DualArgs& a, int i) {
    if constexpr (kSplit) return i / a.splits;
    else return i;
}
template <bool kSplit>
__device__ __forceinline__ int item_kb0(const DualArgs& a, int i) {
    if constexpr (kSplit) return (i % a.splits) * a.kps;
    else return 0;
}
template <bool kSplit>
__device__ __forceinline__ int item_kb1(const DualArgs& a, int i) {
    if constexpr (kSplit) return min(a.kst, item_kb0<true>(a, i) + a.kps);
    else return a.kst;
}
template <bool kSplit>
__device__ __forceinline__ Item item_at(const DualArgs& a, int i) {
    Item it;
    it.t = item_tile<kSplit>(a, i);
    it.sp = i - it.t * a.splits;
    tile_coords(a, it.t, it.tr, it.tc);
    it.kb0 = item_kb0<kSplit>(a, i);
    it.kb1 = item_kb1<kSplit>(a, i);
    return it;
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(8 * 32) : "memory"); }

// kSplit: K split over several CTAs per tile (splits > 1), with the partial
// exchange in the epilogue; a separate instantiation, so that the plain
// kernel's registers are allocated without it.
// kE8: the scales arrive as UE8M0 bytes (a 128-wide stage's four bytes of a
// row are its scale word as they are), not as fp32 values to convert.
template <int BN, int kBlkN, int kBlkK, bool kSplit, bool kPair, bool kE8>
__global__ void __launch_bounds__(kThreads, 1)
    dual_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const DualArgs a) {
    using C = Cfg<BN, kSplit, kPair>;
    constexpr int kCG = kPair ? 2 : 1;
    constexpr int kTileRows = kRowsA * kCG;    // activation rows per tile (both CTAs of a pair)
    constexpr int kSps = kBK / kBlkK;      // scale columns per stage (1 or 4)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    Slot* slot = reinterpret_cast<Slot*>(smem + C::kOffSlot);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    // misc: [0] TMEM base, [1] abort flag, [2] split-K go, [3] an epilogue warp gave up;
    // misc[8 + s], s = 0 .. splits: first column group of slice s (split-K)

    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::kSt + s); };
    auto accf_bar = [&](int h) { return bar0 + 8u * (2 * C::kSt + h); };
    auto acce_bar = [&](int h) { return bar0 + 8u * (2 * C::kSt + 2 + h); };
    auto drain_bar = [&](int h) { return bar0 + 8u * (2 * C::kSt + 4 + h); };
    const uint32_t red_bar = bar0 + 8u * (2 * C::kSt + 6);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Sync sync{reinterpret_cast<volatile uint32_t*>(misc + 1), a.status};
    // pair: rank 0 leads (issues every tcgen05 op of the pair); a pair walks
    // the items with index blockIdx.x / 2
    const uint32_t rank = kPair ? ptx::cluster_rank() : 0u;
    const int first_item = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int item_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    auto at_leader = [&](uint32_t bar) { return kPair ? ptx::mapa(bar, 0u) : bar; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kSt; ++s) {
            ptx::mbar_init(full_bar(s), 3);    // producer expect_tx + the two scale warps
            ptx::mbar_init(empty_bar(s), 2);   // a commit of each issuer
        }
        for (int h = 0; h < 2; ++h) {
            ptx::mbar_init(accf_bar(h), 1);    // the issuer's commit after the tile's last stage
            ptx::mbar_init(acce_bar(h), 8 * kCG);   // one arrive per epilogue warp (pair leader: of both CTAs)
            ptx::mbar_init(drain_bar(h), 1);
        }
        if constexpr (kSplit) ptx::mbar_init(red_bar, 1);
        misc[1] = 0;
        if constexpr (kSplit) {
            misc[3] = 0;
            for (int sp = 0; sp <= a.splits && sp <= 16; ++sp) misc[8 + sp] = static_cast<uint32_t>(sp * (BN / 4) / a.splits);
        }
        ptx::fence_mbar_init();
    }
    // weight-row words past 224 (the second copy's tail) stay 2^0
    for (int i = threadIdx.x; i < C::kSt * 256; i += kThreads) slot[i / 256].sfb[i % 256] = 0x7F7F7F7Fu;
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        if constexpr (kPair) {
            ptx::tmem_alloc_g<2>(ptx::smem_u32(misc), kTmemCols);
            ptx::tmem_relinquish_g<2>();
        } else {
            ptx::tmem_alloc(ptx::smem_u32(misc), kTmemCols);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (kPair) ptx::cluster_sync();   // both CTAs' barriers exist before any remote operation
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    // The next kernel on the stream may launch now; it still waits for this
    // grid to finish before it touches anything this grid writes.
    if (threadIdx.x == 0) ptx::launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The weight boxes of the first stages go out before the wait for the
        // preceding grid (weights are static); the activation boxes after it.
        const uint32_t leader = lane == 0 ? 1u : 0u;
        const uint32_t a0 = ptx::smem_u32(sA), b0 = ptx::smem_u32(sB);
        int n = 0;   // stage jobs issued
        bool failed = false;
        bool waited = false;
        for (int i = first_item; i < a.items && !failed; i += item_step) {
            const Item it = item_at<kSplit>(a, i);
            for (int kb = it.kb0; kb < it.kb1; ++kb, ++n) {
                const int s = n % C::kSt, r = n / C::kSt;
                if (r > 0 && !wait_warp<kPair>(empty_bar(s), (r - 1) & 1, sync, 1)) {
                    failed = true;
                    break;
                }
                // pair: both CTAs' boxes (and the peer's two scale signals) land on the leader's barrier
                ptx::mbar_arrive_expect_tx_if(leader && rank == 0u, full_bar(s),
                                              kCG * (C::kABytes + C::kBBytes) + (kPair ? 32 : 0));
                const int brow = it.tc * BN + static_cast<int>(rank) * (BN / kCG);
                const int arow = it.tr * kTileRows + static_cast<int>(rank) * kRowsA;
                if constexpr (kPair)
                    ptx::tma_load_2d_pair_if(leader, b0 + s * C::kBBytes, &tmB, kb * kBK, brow, at_leader(full_bar(s)));
                else
                    ptx::tma_load_2d_if(leader, b0 + s * C::kBBytes, &tmB, kb * kBK, brow, full_bar(s));
                if (!waited) {
                    ptx::grid_dependency_wait();   // Aq may be the preceding kernel's output
                    waited = true;
                }
                if constexpr (kPair)
                    ptx::tma_load_2d_pair_if(leader, a0 + s * C::kABytes, &tmA, kb * kBK, arow, at_leader(full_bar(s)));
                else
                    ptx::tma_load_2d_if(leader, a0 + s * C::kABytes, &tmA, kb * kBK, arow, full_bar(s));
            }
        }
        if (!waited) ptx::grid_dependency_wait();
    } else if (warp == 3 || warp == 12) {
        // ------------------------------------------------------------ scale warps
        // Half h: the UE8M0 words of activation rows h*128 .. +127 and of
        // weight rows h*112 .. +111 of each stage, from scales loaded one stage
        // ahead (all of a lane's loads in flight together).
        const int h = warp == 3 ? 0 : 1;
        constexpr int kBRowsPerWarp = BN / 2;
        ptx::grid_dependency_wait();   // As may be the preceding kernel's output
        // Raw scales of the next two stages are in flight while a stage is
        // converted (registers p0 for stage n + 1, p1 for stage n + 2).
        struct RawF {
            float4 a[4], b[4];
        };
        struct RawE {
            uint32_t a[4], b[4];
        };
        using Raw = std::conditional_t<kE8, RawE, RawF>;
        // A row's bytes for one stage as loaded (four scale columns, or one
        // [*,128] byte); the word is formed only where it is used, so that
        // nothing waits on a load that is still in flight.
        auto load_word = [&](const uint8_t* p) -> uint32_t {
            if constexpr (kSps == 4) return __ldg(reinterpret_cast<const uint32_t*>(p));
            else return static_cast<uint32_t>(__ldg(p));
        };
        auto load = [&](Raw& v, int i, int kb) {
            if (i >= a.items) return;
            int tr, tc;
            tile_coords(a, item_tile<kSplit>(a, i), tr, tc);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = tr * kTileRows + static_cast<int>(rank) * kRowsA + h * kHalf + lane + 32 * j;
                const int i = lane + 32 * j;
                const int n = tc * BN + h * kBRowsPerWarp + i;
                if constexpr (kE8) {
                    constexpr uint32_t kOne = kSps == 4 ? 0x7F7F7F7Fu : 0x7Fu;   // 1.0 for padding rows
                    v.a[j] = row < a.M ? load_word(a.Ae + static_cast<int64_t>(row) * a.ks + kb * kSps) : kOne;
                    v.b[j] = (i < kBRowsPerWarp && n < a.N)
                                 ? load_word(a.We + static_cast<int64_t>(n / kBlkN) * a.ks + kb * kSps)
                                 : kOne;
                } else {
                    v.a[j] = row < a.M ? load_scales<kSps>(a.As + static_cast<int64_t>(row) * a.ks + kb * kSps)
                                       : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
                    v.b[j] = (i < kBRowsPerWarp && n < a.N)
                                 ? load_scales<kSps>(a.Ws + static_cast<int64_t>(n / kBlkN) * a.ks + kb * kSps)
                                 : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
                }
            }
        };
        // scale word of a loaded row (UE8M0 bytes: the four as loaded, or the
        // one [*,128] byte in every lane; 255 = NaN is refused)
        auto word_of = [&](const auto& r, uint32_t& bad) -> uint32_t {
            if constexpr (kE8) {
                const uint32_t w = kSps == 4 ? r : r * 0x01010101u;
                bad |= zero_byte(~w);
                return w;
            } else {
                return sf_word<kSps>(r, bad);
            }
        };
        auto advance = [&](int& i, int& kb) {
            if (++kb == item_kb1<kSplit>(a, i)) {
                i += item_step;
                kb = item_kb0<kSplit>(a, i);
            }
        };
        int t = first_item, kb = item_kb0<kSplit>(a, first_item);   // (item, stage) being converted
        int t1 = t, kb1 = kb;
        advance(t1, kb1);                  // stage n + 1
        int t2 = t1, kb2 = kb1;
        advance(t2, kb2);                  // stage n + 2
        Raw cur, p0, p1;
        load(cur, t, kb);
        load(p0, t1, kb1);
        int n = 0;
        uint32_t bad_all = 0;
        while (t < a.items) {
            load(p1, t2, kb2);
            const int s = n % C::kSt, r = n / C::kSt;
            if (r > 0 && !wait_warp<kPair>(empty_bar(s), (r - 1) & 1, sync, 2)) break;
            Slot& sl = slot[s];
            uint32_t bad = 0;
            uint32_t w4[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w4[j] = word_of(cur.a[j], bad);
            *reinterpret_cast<uint4*>(&sl.sfa[h][lane * 4]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = lane + 32 * j;
                if (i < kBRowsPerWarp) {
                    const int row = h * kBRowsPerWarp + i;   // weight row inside the tile
                    sl.sfb[(row >> 7) * 128 + (row & 31) * 4 + ((row & 127) >> 5)] = word_of(cur.b[j], bad);
                }
            }
            bad_all |= bad;
            ptx::fence_proxy_async_smem();   // the words are read by tcgen05.cp
            __syncwarp();
            if constexpr (kPair) {
                if (rank == 0u) {
                    if (lane == 0) ptx::mbar_arrive(full_bar(s));
                } else {
                    // The peer signals the leader with a 16-byte copy: its
                    // completion also orders the words written above (made
                    // visible to the async proxy by the fence) before the
                    // leader's tcgen05.cp reads them.
                    const uint32_t x = ptx::smem_u32(smem + C::kOffXfer + 16 * h);
                    ptx::bulk_copy_to_cluster_if(lane == 0 ? 1u : 0u, ptx::mapa(x, 0u), x, 16u,
                                                 at_leader(full_bar(s)));
                }
            } else {
                if (lane == 0) ptx::mbar_arrive(full_bar(s));
            }
            ++n;
            cur = p0;
            p0 = p1;
            t = t1;
            kb = kb1;
            t1 = t2;
            kb1 = kb2;
            advance(t2, kb2);
        }
        // A scale that is not a power of two breaks the caller's promise.
        if (__any_sync(0xFFFFFFFFu, bad_all != 0u) && lane == 0) atomicOr(a.status, kStatusBadScale);
    } else if ((warp == 1 || warp == 2) && (!kPair || rank == 0u)) {
        // ------------------------------------------------------------ MMA issuers
        const int h = warp - 1;
        constexpr uint32_t idesc_mx = ptx::idesc_mxf8(kHalf * kCG, BN);
        const uint64_t ad_base = ptx::smem_desc(ptx::smem_u32(sA) + h * (kHalf * kBK), 16, 1024, ptx::kLayoutSw128);
        const uint64_t bd_base = ptx::smem_desc(ptx::smem_u32(sB), 16, 1024, ptx::kLayoutSw128);
        const uint64_t sfa_base = ptx::smem_desc(ptx::smem_u32(slot[0].sfa[h]), 128, 128, ptx::kLayoutNone);
        const uint64_t sfb_base = ptx::smem_desc(ptx::smem_u32(slot[0].sfb), 128, 128, ptx::kLayoutNone);
        constexpr uint32_t kSlotStep = sizeof(Slot) >> 4;
        const uint32_t d = tmem + static_cast<uint32_t>(h * BN);
        int n = 0, ntile = 0;
        bool failed = false;
        for (int i = first_item; i < a.items && !failed; i += item_step, ++ntile) {
            // the accumulator must have been read by the epilogue
            if (ntile > 0 && !wait_warp<kPair>(acce_bar(h), (ntile - 1) & 1, sync, 3)) break;
            ptx::tc_fence_after();
            const int kb0 = item_kb0<kSplit>(a, i), kb1 = item_kb1<kSplit>(a, i);
            for (int kb = kb0; kb < kb1; ++kb, ++n) {
                const int s = n % C::kSt, r = n / C::kSt;
                if (!wait_warp<kPair>(full_bar(s), r & 1, sync, 4)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t t_sfa = tmem + C::kSfCol + 32u * h + 16u * (n & 1), t_sfb = t_sfa + 4u;
                const uint64_t so = static_cast<uint64_t>(s) * kSlotStep;
                if constexpr (kPair) {
                    ptx::mx_stage2_elect_pair(d, ad_base + static_cast<uint64_t>(s * (C::kABytes >> 4)),
                                              bd_base + static_cast<uint64_t>(s * (C::kBBytes >> 4)),
                                              ptx::idesc_sf_ids(idesc_mx, 0, 0), ptx::idesc_sf_ids(idesc_mx, 1, 1),
                                              ptx::idesc_sf_ids(idesc_mx, 2, 2), ptx::idesc_sf_ids(idesc_mx, 3, 3),
                                              t_sfa, t_sfb, sfa_base + so, sfb_base + so, kb > kb0 ? 1u : 0u);
                    ptx::commit_pair_elect(empty_bar(s));   // frees the stage in both CTAs
                } else {
                    ptx::mx_stage2_elect(d, ad_base + static_cast<uint64_t>(s * (C::kABytes >> 4)),
                                         bd_base + static_cast<uint64_t>(s * (C::kBBytes >> 4)),
                                         ptx::idesc_sf_ids(idesc_mx, 0, 0), ptx::idesc_sf_ids(idesc_mx, 1, 1),
                                         ptx::idesc_sf_ids(idesc_mx, 2, 2), ptx::idesc_sf_ids(idesc_mx, 3, 3), t_sfa,
                                         t_sfb, sfa_base + so, sfb_base + so, kb > kb0 ? 1u : 0u);
                    ptx::commit_elect(empty_bar(s));   // frees the stage once both halves' MMAs are done
                }
            }
            if (failed) break;
            // the tile's accumulator is complete (pair: in both CTAs)
            if constexpr (kPair) ptx::commit_pair_elect(accf_bar(h));
            else ptx::commit_elect(accf_bar(h));
        }
        // every tcgen05 op lands before teardown
        if constexpr (kPair) ptx::commit_pair_local_elect(drain_bar(h));
        else ptx::commit_elect(drain_bar(h));
        if (lane == 0) wait_slow(drain_bar(h), 0, sync, 5);
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // the pair's peer issues nothing
    } else {
        // ------------------------------------------------------------ epilogue (warps 4-11)
        const int ew = warp - kEpi0;            // 0 .. 7
        const int quad = warp & 3;              // TMEM lane quadrant
        const int chalf = ew >> 2;              // which half of the columns (split-K sum: which half of the rows)
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        ptx::grid_dependency_wait();            // D may still be read by the preceding kernel
        const bool v8 = ((reinterpret_cast<uintptr_t>(a.D) | (static_cast<uintptr_t>(a.N) * 2u)) & 31u) == 0;
        volatile uint32_t* gave_up = misc + 3;
        int ntile = 0;
        for (int i = first_item; i < a.items; i += item_step, ++ntile) {
            const Item it = item_at<kSplit>(a, i);
            bool failed = false;
            if constexpr (!kSplit) {
                for (int h = 0; h < 2 && !failed; ++h) {
                    if (!wait_warp<kPair>(accf_bar(h), ntile & 1, sync, 6)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int grow = it.tr * kTileRows + static_cast<int>(rank) * kRowsA + h * kHalf + quad * 32 + lane;
                    __nv_bfloat16* drow = a.D + static_cast<int64_t>(grow) * a.N;
                    // The warp's share of the accumulator goes to registers as
                    // packed bf16 first, and the accumulator is released before
                    // the stores: the next tile's MMAs for this half start
                    // while D is written.
                    constexpr int kChunks = C::kColsPerWarp / 16;
                    uint32_t w[kChunks][8];
#pragma unroll
                    for (int q = 0; q < kChunks; ++q) {
                        uint32_t rr[16];
                        ptx::tmem_ld<16>(t_lane + static_cast<uint32_t>(h * BN + chalf * C::kColsPerWarp + 16 * q), rr);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const __nv_bfloat162 p =
                                __floats2bfloat162_rn(__uint_as_float(rr[2 * j]), __uint_as_float(rr[2 * j + 1]));
                            w[q][j] = *reinterpret_cast<const uint32_t*>(&p);
                        }
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if constexpr (kPair) {
                        if (rank == 0u) {
                            if (lane == 0) ptx::mbar_arrive(acce_bar(h));
                        } else {
                            ptx::mbar_arrive_cluster_if(lane == 0 ? 1u : 0u, at_leader(acce_bar(h)));
                        }
                    } else {
                        if (lane == 0) ptx::mbar_arrive(acce_bar(h));
                    }
                    if (grow < a.M) {
#pragma unroll
                        for (int q = 0; q < kChunks; ++q) {
                            const int gcol = it.tc * BN + chalf * C::kColsPerWarp + 16 * q;
                            if (v8 && gcol + 16 <= a.N) {
                                ptx::st_global_v8(drow + gcol, w[q]);
                            } else {
                                if (gcol < a.N)
                                    *reinterpret_cast<uint4*>(drow + gcol) =
                                        make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
                                if (gcol + 8 < a.N)
                                    *reinterpret_cast<uint4*>(drow + gcol + 8) =
                                        make_uint4(w[q][4], w[q][5], w[q][6], w[q][7]);
                            }
                        }
                    }
                }
                if (failed) break;
                continue;
            }
            if constexpr (kSplit) {
                // ---- split-K, deterministic.  The tile's BN / 4 column groups
                // (four columns each) are cut into `splits` contiguous slices;
                // split s sums slice s over all splits in split order
                // (p_0 + p_1 + ...) and writes that slice of D.  Partials move in
                // warp units (32 rows x 4 columns, 512 bytes) of row block rb
                // (half h, lane quadrant) and group g, slice-major: slice s at
                // unit s * per, then rb * (its groups) + (g - its first group).
                // Every move is a bulk copy through shared memory: the operand
                // ring is idle once the CTA's only item is accumulated.  The
                // epilogue warps meet at named barriers from here on, so a warp
                // that gave up says so and all of them leave together.
                constexpr int G = BN / 4;
                const int S = a.splits;
                const volatile uint32_t* lo_tab = misc + 8;   // first group of each slice, and G at [S]
                auto lo_of = [&](int s) { return static_cast<int>(lo_tab[s]); };
                const int glo = lo_of(it.sp), ng = lo_of(it.sp + 1) - glo;   // this CTA's slice
                const int64_t pstride = int64_t(S) * a.per * 128;             // floats per item's partial
                const uint32_t stage = ptx::smem_u32(sA);
                for (int h = 0; h < 2 && !failed; ++h) failed = !wait_warp(accf_bar(h), ntile & 1, sync, 6);
                ptx::tc_fence_after();
                if (!failed) {
                    // The other slices' units of this partial, slice-major as in
                    // global memory: this warp's groups gA .. gB of each slice.
                    constexpr int kBatch = 8;
                    const int gA = chalf * (G / 2), gB = gA + G / 2;
                    for (int h = 0; h < 2; ++h) {
                        const int rb = h * 4 + quad;
                        const uint32_t t_h = t_lane + static_cast<uint32_t>(h * BN);
                        for (int s = 0, jj = 0; s < S; ++s) {
                            if (s == it.sp) continue;
                            const int lo = lo_of(s), n = lo_of(s + 1) - lo;
                            const int g0 = max(lo, gA), g1 = min(lo + n, gB);
                            const uint32_t st0 = stage + static_cast<uint32_t>(((jj * a.per + rb * n - lo) * 32 + lane) * 16);
                            ++jj;
                            for (int gb = g0; gb < g1; gb += kBatch) {
                                uint32_t v[kBatch][4];
    #pragma unroll
                                for (int b = 0; b < kBatch; ++b)
                                    if (gb + b < g1) ptx::tmem_ld<4>(t_h + static_cast<uint32_t>((gb + b) * 4), v[b]);
                                ptx::tmem_wait_ld();
    #pragma unroll
                                for (int b = 0; b < kBatch; ++b) {
                                    if (gb + b >= g1) break;
                                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(st0 + (gb + b) * 512),
                                                 "r"(v[b][0]), "r"(v[b][1]), "r"(v[b][2]), "r"(v[b][3])
                                                 : "memory");
                                }
                            }
                        }
                    }
                }
                if (failed && lane == 0) *gave_up = 1u;
                ptx::fence_proxy_async_smem();   // the staged units are read by bulk copies
                uint32_t* cnt = a.counters + it.t;
                epi_sync();
                if (*gave_up != 0u) break;
                if (ew == 0 && lane == 0) {
                    float* pbase = a.partial + static_cast<int64_t>(i) * pstride;
                    for (int s = 0, jj = 0; s < S; ++s) {
                        if (s == it.sp) continue;
                        const uint32_t n = static_cast<uint32_t>(lo_of(s + 1) - lo_of(s));
                        ptx::bulk_store(pbase + int64_t(s) * a.per * 128, stage + jj * a.per * 512, n * 8u * 512u);
                        ++jj;
                    }
                    ptx::bulk_commit();
                    ptx::bulk_wait_all();            // written, and the staging area free again
                    ptx::fence_proxy_async_all();
                    // Arrival count: each launch adds `splits` per tile, and the
                    // last arriver pads it to the next multiple of 16, so a launch
                    // starts on a multiple of 16 and needs no reset.
                    const uint32_t old = ptx::atom_add_acq_rel_gpu(cnt, 1u);
                    const uint32_t base = old & ~15u;
                    if (old - base == static_cast<uint32_t>(S - 1) && S < 16) atomicAdd(cnt, 16u - static_cast<uint32_t>(S));
                    const uint64_t t0 = ptx::globaltimer();
                    uint32_t ok = 1;
                    uint32_t spins = 0;
                    while (ptx::ld_acquire_gpu(cnt) - base < static_cast<uint32_t>(S)) {
                        if ((++spins & 15u) == 0 && ptx::globaltimer() - t0 > kTimeoutNs) {
                            *sync.abort_flag = 1u;
                            atomicOr(a.status, kStatusTimeout | (7u << 8));
                            ok = 0;
                            break;
                        }
                        __nanosleep(64);
                    }
                    ptx::fence_proxy_async_all();   // before the bulk copies of the other partials
                    misc[2] = ok;
                    if (ok) {
                        // this slice of every other split's partial, all in flight at once
                        const uint32_t bytes = static_cast<uint32_t>(ng) * 8u * 512u;
                        ptx::mbar_arrive_expect_tx(red_bar, bytes * static_cast<uint32_t>(S - 1));
                        const float* tbase = a.partial + static_cast<int64_t>(it.t) * S * pstride + int64_t(it.sp) * a.per * 128;
                        for (int j = 0, jj = 0; j < S; ++j) {
                            if (j == it.sp) continue;
                            ptx::bulk_load(stage + jj * bytes, tbase + j * pstride, bytes, red_bar);
                            ++jj;
                        }
                    }
                }
                epi_sync();
                if (*reinterpret_cast<volatile uint32_t*>(misc + 2) == 0u) break;
                const bool ok = wait_warp(red_bar, 0, sync, 8);
                if (!ok && lane == 0) {
                    *gave_up = 1u;
                    if (ew == 0) {   // the copies in flight land before the CTA leaves (bounded)
                        const uint64_t t1 = ptx::globaltimer();
                        while (!ptx::mbar_try_wait(red_bar, 0) && ptx::globaltimer() - t1 < (1ull << 26)) {
                        }
                    }
                }
                // D of the slice, bf16, staged row-major after the received units
                const int dstride = ng * 8 + 8;   // bytes per staged row
                const uint32_t dstage = stage + static_cast<uint32_t>((S - 1) * ng * 8 * 512);
                if (ok) {
                    // warp (quadrant, half chalf): rows chalf * 128 + quad * 32 + lane
                    const int rb = chalf * 4 + quad;
                    const uint32_t t_row = t_lane + static_cast<uint32_t>(chalf * BN + glo * 4);
                    constexpr int kBatch = 8;
                    for (int g0 = 0; g0 < ng; g0 += kBatch) {
                        uint32_t own[kBatch][4];
    #pragma unroll
                        for (int b = 0; b < kBatch; ++b)
                            if (g0 + b < ng) ptx::tmem_ld<4>(t_row + static_cast<uint32_t>((g0 + b) * 4), own[b]);
                        ptx::tmem_wait_ld();
    #pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            if (g0 + b >= ng) break;
                            const uint32_t src = stage + ((rb * ng + g0 + b) * 32 + lane) * 16;
                            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                            for (int j = 0, jj = 0; j < S; ++j) {
                                float4 v;
                                if (j == it.sp) {
                                    v = make_float4(__uint_as_float(own[b][0]), __uint_as_float(own[b][1]),
                                                    __uint_as_float(own[b][2]), __uint_as_float(own[b][3]));
                                } else {
                                    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                                 : "r"(src + static_cast<uint32_t>(jj * ng * 8 * 512)));
                                    ++jj;
                                }
                                if (j == 0) {
                                    acc = v;
                                } else {
                                    acc.x += v.x;
                                    acc.y += v.y;
                                    acc.z += v.z;
                                    acc.w += v.w;
                                }
                            }
                            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
                            const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
                            const uint32_t at = dstage + static_cast<uint32_t>((chalf * 128 + quad * 32 + lane) * dstride + (g0 + b) * 8);
                            asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(at),
                                         "r"(*reinterpret_cast<const uint32_t*>(&lo)),
                                         "r"(*reinterpret_cast<const uint32_t*>(&hi))
                                         : "memory");
                        }
                    }
                }
                ptx::tc_fence_before();
                epi_sync();   // the slice of D is staged (and TMEM read)
                if (*gave_up != 0u) break;
                // coalesced stores: a warp takes 32 / ng rows at a time, consecutive
                // lanes consecutive groups of a row (ng <= 32 for two splits or more)
                {
                    const int rpi = 32 / ng;                  // rows per warp iteration
                    const int lr = lane / ng, gi = lane - lr * ng;
                    const int row0 = it.tr * kRowsA, col = it.tc * BN + (glo + gi) * 4;
                    if (lr < rpi && col < a.N) {              // N % 8 == 0: the four columns are all inside
                        for (int r = ew * rpi + lr; r < kRowsA; r += 8 * rpi) {
                            const int row = row0 + r;
                            if (row >= a.M) break;
                            uint32_t x0, x1;
                            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                                         : "=r"(x0), "=r"(x1)
                                         : "r"(dstage + static_cast<uint32_t>(r * dstride + gi * 8)));
                            *reinterpret_cast<uint2*>(a.D + static_cast<int64_t>(row) * a.N + col) = make_uint2(x0, x1);
                        }
                    }
                }
                if (lane == 0) {
                    ptx::mbar_arrive(acce_bar(0));
                    ptx::mbar_arrive(acce_bar(1));
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (kPair) ptx::cluster_sync();   // no remote operation targets a CTA that has left
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (kPair) ptx::tmem_dealloc_g<2>(tmem, kTmemCols);
        else ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int BN, int kBlkN, int kBlkK, bool kSplit, bool kPair, bool kE8>
sgq_status run(const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a, int grid, cudaStream_t st) {
    using C = Cfg<BN, kSplit, kPair>;
    constexpr size_t kSmem = C::kSmem;
    auto kern = dual_gemm_kernel<BN, kBlkN, kBlkK, kSplit, kPair, kE8>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem)) !=
            cudaSuccess)
            return SGQ_ERR_CUDA;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kPair ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, a) != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

// Weight rows per tile: 224 (two 224-column accumulators and the scale slots
// fill TMEM's 512 columns) or 192; the host takes the width whose tiles fill
// the grid's rounds best.
constexpr int kBNWide = 224;
constexpr int kBNNarrow = 192;

template <int BN, bool kSplit, bool kPair, bool kE8>
sgq_status dispatch_bn(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a,
                       int grid, cudaStream_t st) {
    if (blk_n == 32)
        return blk_k == 32 ? run<BN, 32, 32, kSplit, kPair, kE8>(tmA, tmB, a, grid, st)
                           : run<BN, 32, 128, kSplit, kPair, kE8>(tmA, tmB, a, grid, st);
    return blk_k == 32 ? run<BN, 128, 32, kSplit, kPair, kE8>(tmA, tmB, a, grid, st)
                       : run<BN, 128, 128, kSplit, kPair, kE8>(tmA, tmB, a, grid, st);
}
// Kinds of launch: one CTA per tile, K split over CTAs, CTA pairs.
enum Kind : int { kPlain = 0, kSplitK = 1, kPairs = 2 };
// One translation unit per width, kind and scale format
// (gemm_dual_{224,192}{,s,p}{,e}.cu); `dispatch` picks among them.
#define SGQ_DUAL_DISPATCH_DECL(NAME)                                                                            \
    sgq_status NAME(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a, \
                    int grid, cudaStream_t st);
SGQ_DUAL_DISPATCH_DECL(dispatch_224)
SGQ_DUAL_DISPATCH_DECL(dispatch_192)
SGQ_DUAL_DISPATCH_DECL(dispatch_224_split)
SGQ_DUAL_DISPATCH_DECL(dispatch_192_split)
SGQ_DUAL_DISPATCH_DECL(dispatch_224_pair)
SGQ_DUAL_DISPATCH_DECL(dispatch_192_pair)
SGQ_DUAL_DISPATCH_DECL(dispatch_224_e8)
SGQ_DUAL_DISPATCH_DECL(dispatch_192_e8)
SGQ_DUAL_DISPATCH_DECL(dispatch_224_split_e8)
SGQ_DUAL_DISPATCH_DECL(dispatch_192_split_e8)
SGQ_DUAL_DISPATCH_DECL(dispatch_224_pair_e8)
SGQ_DUAL_DISPATCH_DECL(dispatch_192_pair_e8)
#undef SGQ_DUAL_DISPATCH_DECL
inline sgq_status dispatch(int bn, Kind kind, bool e8, int blk_n, int blk_k, const CUtensorMap& tmA,
                           const CUtensorMap& tmB, const DualArgs& a, int grid, cudaStream_t st) {
    using Fn = sgq_status (*)(int, int, const CUtensorMap&, const CUtensorMap&, const DualArgs&, int, cudaStream_t);
    static constexpr Fn table[2][3][2] = {
        {{dispatch_224, dispatch_224_e8}, {dispatch_224_split, dispatch_224_split_e8},
         {dispatch_224_pair, dispatch_224_pair_e8}},
        {{dispatch_192, dispatch_192_e8}, {dispatch_192_split, dispatch_192_split_e8},
         {dispatch_192_pair, dispatch_192_pair_e8}}};
    return table[bn == 224 ? 0 : 1][kind][e8 ? 1 : 0](blk_n, blk_k, tmA, tmB, a, grid, st);
}

}  // namespace dual
}  // namespace sgq
