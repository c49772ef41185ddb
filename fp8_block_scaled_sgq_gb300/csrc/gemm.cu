// Block-scaled FP8 GEMM for sm_103a:  D = (Aq * As)(Wq * Ws)^T, bf16 out.
//
// Defined by the vLLM "scaled_mm" API page (AiterInt8ScaledMMLinearKernel.
// apply_weights docstring: output = mm(scale_a * a, scale_b * b), scales
// broadcast numpy-style) in the "NT" layout of sglang PR #42604,
// Modifications: fp8_gemm_nt((Aq, As), (Wq, Ws), D, recipe=(1, blk_n, blk_k)).
// Weight scales are [n_blocks, k_blocks] (vLLM page, XPUFp8BlockScaledMMKernel).
//
// Design (one persistent CTA per SM, 11 warps):
//   warp 0      TMA producer: 128x128-byte K-major tiles of both operands
//               (128B swizzle) into a multi-stage shared-memory ring.
//   warp 1      MMA issuer: one thread issues tcgen05.mma into a TMEM
//               accumulator.  For each 128-wide K stage:
//                 - if every scale of the stage is an exact power of two,
//                   the scales are converted to UE8M0 bytes, copied to TMEM
//                   (tcgen05.cp) and applied inside the block-scaled MMA
//                   (kind::mxf8f6f4, one scale per row per 32-wide K chunk);
//                   consecutive such stages accumulate in TMEM;
//                 - otherwise the stage's partial product for each scale
//                   group is formed unscaled (kind::f8f6f4) and handed to the
//                   epilogue, which applies the fp32 scales ("promotion").
//   warp 2      scale loader: reads As/Ws for the stage, checks the
//               power-of-two property, writes the UE8M0 words (laid out for
//               tcgen05.cp) and the raw fp32 scales into the stage's slot.
//   warps 3-10  epilogue: tcgen05.ld of the accumulator (each warp its TMEM
//               lane quadrant and half of the columns), fp32 promotion
//               and accumulation in registers, bf16 store, or an fp32
//               split-K partial plus a last-arriver reduction.
// Small M (<= 64) runs "swap-AB": the weight rows fill the 128-row MMA M
// dimension and the tokens the MMA N dimension (16/32/64), with split-K over
// the persistent grid so all SMs stream weights.
//
// Every wait on an mbarrier is bounded; on time-out the CTA records a status
// word, stops issuing work and exits through the normal teardown.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "sgq_internal.h"

namespace sgq {

__device__ uint32_t g_gemm_status;

namespace {

constexpr int kBM = 128;          // MMA M: rows of the "A" operand per tile
constexpr int kBK = 128;          // K elements (bytes) per pipeline stage
constexpr int kNumThreads = 352;  // 11 warps
constexpr int kEpiWarp0 = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 480;  // two 16-column scale-factor slots at 480 and 496
constexpr uint64_t kTimeoutNs = 1ull << 30;

constexpr uint32_t kInfoPromote = 1u;
constexpr uint32_t kInfoLast = 2u;

constexpr uint32_t kStatusTimeout = 1u;

template <int BN>
struct alignas(128) SfSlot {
    uint32_t sfa[128];                  // UE8M0 words of the A operand (tcgen05.cp order)
    uint32_t sfb[BN < 128 ? 128 : BN];  // UE8M0 words of the B operand
    float lane_raw[4][128];             // fp32 scale per A row, per 32-wide K chunk
    float col_raw[4][64];               // fp32 scale per B row group, per chunk
    uint32_t pow2;                      // every scale of the stage is 2^e
};

template <int BN>
struct alignas(16) Info {
    uint32_t flags;
    uint32_t pad[3];
    float lane_s[128];
    float col_s[BN];
};

struct GemmArgs {
    const float* As;
    const float* Ws;
    __nv_bfloat16* D;
    float* partial;       // split-K workspace
    uint32_t* counters;   // split-K arrival counters (self-resetting)
    int M, N, K, blk_n, blk_k, ks;   // ks = K / blk_k (columns of As and Ws)
    int rows, cols;       // extents of the MMA A operand and B operand
    int tiles_r, tiles_c, kb_total, kb_per_split, splits, items, group_r;
    int force_promote;
};

// Scale of activation row m for the 32-wide K chunk q.
__device__ __forceinline__ float act_scale(const GemmArgs& a, int m, int q) {
    return __ldg(a.As + static_cast<int64_t>(m) * a.ks + (q * 32) / a.blk_k);
}
// Scale of weight row n for the 32-wide K chunk q.
__device__ __forceinline__ float wt_scale(const GemmArgs& a, int n, int q) {
    return __ldg(a.Ws + static_cast<int64_t>(n / a.blk_n) * a.ks + (q * 32) / a.blk_k);
}

__device__ __forceinline__ bool is_pow2_scale(float s) {
    const uint32_t b = __float_as_uint(s);
    const uint32_t e = b >> 23;
    return (b & 0x007FFFFFu) == 0 && e != 0 && e < 0xFFu;  // sign 0, normal, mantissa 0
}

// Walks the (item, k-stage) jobs of one CTA in order.
struct JobIter {
    int item, kb, kb1;
    int tile, split, tr, tc;
    __device__ void load(const GemmArgs& a) {
        split = item % a.splits;
        tile = item / a.splits;
        const int per_group = a.group_r * a.tiles_c;
        const int g = tile / per_group;
        const int first = g * a.group_r;
        const int gm = min(a.tiles_r - first, a.group_r);
        const int in = tile - g * per_group;
        tr = first + in % gm;
        tc = in / gm;
        kb = split * a.kb_per_split;
        kb1 = min(a.kb_total, kb + a.kb_per_split);
    }
    __device__ void begin(const GemmArgs& a) {
        item = blockIdx.x;
        if (item < a.items) load(a);
    }
    __device__ bool valid(const GemmArgs& a) const { return item < a.items; }
    __device__ bool last_kb() const { return kb + 1 == kb1; }
    __device__ void next(const GemmArgs& a) {
        if (++kb >= kb1) {
            item += gridDim.x;
            if (item < a.items) load(a);
        }
    }
};

struct Sync {
    volatile uint32_t* abort_flag;
};

__device__ bool wait_bar(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((++spins & 31u) == 0) {
            if (*s.abort_flag) return false;
            if (ptx::globaltimer() - t0 > kTimeoutNs) {
                *s.abort_flag = 1u;
                atomicOr(&g_gemm_status, kStatusTimeout | (where << 8));
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool epi_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, 1, 256, q;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int BN, int kStages, bool kSwap, int kAccBufs>
struct Cfg {
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = BN * kBK;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kCols = BN / 2;  // accumulator columns per epilogue thread
    static constexpr int kLd = kCols < 16 ? kCols : 16;
    static constexpr int kSfbCopies = BN > 128 ? BN / 128 : 1;
    static constexpr size_t kOffA = 0;
    static constexpr size_t kOffB = kOffA + size_t(kStages) * kABytes;
    static constexpr size_t kOffSf = kOffB + size_t(kStages) * kBBytes;
    static constexpr size_t kOffInfo = kOffSf + size_t(kStages) * sizeof(SfSlot<BN>);
    static constexpr size_t kOffBar = kOffInfo + size_t(kAccBufs) * sizeof(Info<BN>);
    static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
    static constexpr size_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr size_t kSmem = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(kAccBufs * BN <= int(kSfCol), "TMEM budget");
    static_assert(!kSwap || BN <= 64, "swap-AB token tile");
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int BN, int kStages, bool kSwap, int kAccBufs>
__global__ void __launch_bounds__(kNumThreads, 1)
    fp8_block_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
    using C = Cfg<BN, kStages, kSwap, kAccBufs>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    SfSlot<BN>* sf = reinterpret_cast<SfSlot<BN>*>(smem + C::kOffSf);
    Info<BN>* info = reinterpret_cast<Info<BN>*>(smem + C::kOffInfo);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    // misc[0]: TMEM base, misc[1]: abort flag, misc[2]: epilogue broadcast

    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * kStages + kAccBufs + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kAccBufs);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Sync sync{reinterpret_cast<volatile uint32_t*>(misc + 1)};

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(full_bar(s), 2);   // producer expect_tx + scale loader
            ptx::mbar_init(empty_bar(s), 1);  // tcgen05.commit
        }
        for (int b = 0; b < kAccBufs; ++b) {
            ptx::mbar_init(accf_bar(b), 2);   // MMA thread arrive + tcgen05.commit
            ptx::mbar_init(acce_bar(b), 8);   // one arrive per epilogue warp
        }
        ptx::mbar_init(drain_bar, 1);
        misc[1] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(misc), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // The weight operand does not depend on the preceding kernel, so the
        // weight halves of the first kStages stages go out before the
        // programmatic-dependency wait; activations only after it.
        const CUtensorMap* tmW = kSwap ? &tmA : &tmB;
        const CUtensorMap* tmX = kSwap ? &tmB : &tmA;
        auto w_dst = [&](int s) { return ptx::smem_u32(kSwap ? sA + s * C::kABytes : sB + s * C::kBBytes); };
        auto x_dst = [&](int s) { return ptx::smem_u32(kSwap ? sB + s * C::kBBytes : sA + s * C::kABytes); };
        auto w_row = [&](const JobIter& j) { return kSwap ? j.tr * kBM : j.tc * BN; };
        auto x_row = [&](const JobIter& j) { return kSwap ? j.tc * BN : j.tr * kBM; };
        JobIter it;
        it.begin(a);
        JobIter pre = it;
        int npre = 0;
        while (npre < kStages && pre.valid(a)) {
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(full_bar(npre), C::kStageBytes);
                ptx::tma_load_2d(w_dst(npre), tmW, pre.kb * kBK, w_row(pre), full_bar(npre));
            }
            pre.next(a);
            ++npre;
        }
        if (lane == 0) ptx::grid_dependency_wait();
        for (int s = 0; s < npre; ++s) {
            if (lane == 0) ptx::tma_load_2d(x_dst(s), tmX, it.kb * kBK, x_row(it), full_bar(s));
            it.next(a);
        }
        int stage = npre % kStages;
        uint32_t phase = npre / kStages;
        while (it.valid(a)) {
            if (!wait_bar(empty_bar(stage), phase ^ 1u, sync, 1)) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
                ptx::tma_load_2d(w_dst(stage), tmW, it.kb * kBK, w_row(it), full_bar(stage));
                ptx::tma_load_2d(x_dst(stage), tmX, it.kb * kBK, x_row(it), full_bar(stage));
            }
            it.next(a);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------- scale loader
        // Two-phase software pipeline.  Issue: the raw fp32 scales of up to
        // kStages jobs are fetched with cp.async (one commit group per job)
        // as soon as their slot is free.  Finish: when the oldest job's copies
        // have landed, its scales are checked for the power-of-two property,
        // packed into UE8M0 words in tcgen05.cp order and handed to the MMA
        // warp.  Global-load latency is paid once per ring, not per stage.
        ptx::grid_dependency_wait();
        const bool blk128 = a.blk_k == 128;
        const int nld = blk128 ? 1 : 4;           // distinct scale chunks per stage
        auto issue_raw = [&](SfSlot<BN>& slot, const JobIter& j) {
            const int q0 = j.kb * 4;
            const int nq = min(4, (a.K - j.kb * kBK) / 32);
            const int row0 = j.tr * kBM, col0 = j.tc * BN;
            if (!kSwap) {
                // A operand = activation rows: one scale per row and chunk
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = lane + 32 * i, g = row0 + r;
                    for (int c = 0; c < nld; ++c) {
                        float* dst = &slot.lane_raw[c][r];
                        if (c < nq && g < a.rows)
                            ptx::cp_async_4(ptx::smem_u32(dst),
                                            a.As + static_cast<int64_t>(g) * a.ks + ((q0 + c) * 32) / a.blk_k);
                        else
                            *dst = 1.0f;
                    }
                }
                // B operand = weight rows: one scale per n-block and chunk
                const int ngrp = (BN + a.blk_n - 1) / a.blk_n;
                for (int idx = lane; idx < ngrp * nld; idx += 32) {
                    const int gi = idx / nld, c = idx - gi * nld, g = col0 + gi * a.blk_n;
                    float* dst = &slot.col_raw[c][gi];
                    if (c < nq && g < a.cols)
                        ptx::cp_async_4(ptx::smem_u32(dst),
                                        a.Ws + static_cast<int64_t>(g / a.blk_n) * a.ks + ((q0 + c) * 32) / a.blk_k);
                    else
                        *dst = 1.0f;
                }
            } else {
                // A operand = weight rows: one scale per n-block and chunk
                const int nblk = kBM / a.blk_n;
                for (int idx = lane; idx < nblk * nld; idx += 32) {
                    const int bi = idx / nld, c = idx - bi * nld, g = row0 + bi * a.blk_n;
                    float* dst = &slot.lane_raw[c][bi];
                    if (c < nq && g < a.rows)
                        ptx::cp_async_4(ptx::smem_u32(dst),
                                        a.Ws + static_cast<int64_t>(g / a.blk_n) * a.ks + ((q0 + c) * 32) / a.blk_k);
                    else
                        *dst = 1.0f;
                }
                // B operand = token rows: one scale per token and chunk
                for (int idx = lane; idx < BN * nld; idx += 32) {
                    const int t = idx / nld, c = idx - t * nld, g = col0 + t;
                    float* dst = &slot.col_raw[c][t];
                    if (c < nq && g < a.cols)
                        ptx::cp_async_4(ptx::smem_u32(dst),
                                        a.As + static_cast<int64_t>(g) * a.ks + ((q0 + c) * 32) / a.blk_k);
                    else
                        *dst = 1.0f;
                }
            }
        };
        auto convert = [&](SfSlot<BN>& slot) {
            bool ok = true;
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = lane + 32 * i;
                const int li = kSwap ? r / a.blk_n : r;
                uint32_t word = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float s = slot.lane_raw[blk128 ? 0 : j][li];
                    ok &= is_pow2_scale(s);
                    word |= ((__float_as_uint(s) >> 23) & 0xFFu) << (8 * j);
                }
                w4[i] = word;
            }
            *reinterpret_cast<uint4*>(&slot.sfa[lane * 4]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
#pragma unroll
            for (int h = 0; h < C::kSfbCopies; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = h * 128 + lane + 32 * i;
                    uint32_t word = 0x7F7F7F7Fu;   // 2^0 for rows past the tile
                    if (c < BN) {
                        const int ci = kSwap ? c : c / a.blk_n;
                        word = 0;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float s = slot.col_raw[blk128 ? 0 : j][ci];
                            ok &= is_pow2_scale(s);
                            word |= ((__float_as_uint(s) >> 23) & 0xFFu) << (8 * j);
                        }
                    }
                    w4[i] = word;
                }
                *reinterpret_cast<uint4*>(&slot.sfb[h * 128 + lane * 4]) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            const bool all_ok = __all_sync(0xFFFFFFFFu, ok);
            if (lane == 0) slot.pow2 = all_ok ? 1u : 0u;
        };
        JobIter iss, fin;
        iss.begin(a);
        fin.begin(a);
        uint32_t n_iss = 0, n_fin = 0;
        bool failed = false;
        while (fin.valid(a) && !failed) {
            while (iss.valid(a) && n_iss - n_fin < static_cast<uint32_t>(kStages)) {
                const int si = static_cast<int>(n_iss % kStages);
                const uint32_t par = ((n_iss / kStages) & 1u) ^ 1u;
                if (n_iss != n_fin) {
                    if (!ptx::mbar_try_wait(empty_bar(si), par)) break;   // finish something first
                } else if (!wait_bar(empty_bar(si), par, sync, 3)) {
                    failed = true;
                    break;
                }
                issue_raw(sf[si], iss);
                ptx::cp_async_commit();
                ++n_iss;
                iss.next(a);
            }
            if (failed) break;
            const int sf_i = static_cast<int>(n_fin % kStages);
            ptx::cp_async_wait_pending(static_cast<int>(n_iss - n_fin) - 1);
            __syncwarp();
            convert(sf[sf_i]);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full_bar(sf_i));
            ++n_fin;
            fin.next(a);
        }
        ptx::cp_async_wait_pending(0);
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        const uint32_t idesc_f8 = ptx::idesc_f8(kBM, BN);
        const uint32_t idesc_mx = ptx::idesc_mxf8(kBM, BN);
        const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
        const int col_group = kSwap ? 1 : a.blk_n;
        JobIter it;
        it.begin(a);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t seg = 0;     // accumulator segments issued so far
        uint32_t mx_used = 0; // block-scaled stages issued so far (scale-slot parity)
        bool failed = false;
        bool seg_open = false;
        bool first = true;
        auto acc_buf = [&](uint32_t u) { return static_cast<int>(u % kAccBufs); };
        auto acc_par = [&](uint32_t u) { return (u / kAccBufs) & 1u; };
        // Hands the open accumulator segment to the epilogue.
        auto close_segment = [&](uint32_t flags) {
            const int b = acc_buf(seg);
            if (lane == 0) info[b].flags = flags;
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(accf_bar(b));
                ptx::tc_commit(accf_bar(b));
            }
            ++seg;
        };
        while (it.valid(a) && !failed) {
            if (!wait_bar(full_bar(stage), phase, sync, 2)) { failed = true; break; }
            ptx::tc_fence_after();
            SfSlot<BN>& slot = sf[stage];
            const int nq = min(4, (a.K - it.kb * kBK) / 32);
            const uint32_t a_st = sA0 + stage * C::kABytes;
            const uint32_t b_st = sB0 + stage * C::kBBytes;
            const bool mx = slot.pow2 != 0u && !a.force_promote;
            if (mx) {
                if (!seg_open) {
                    if (!wait_bar(acce_bar(acc_buf(seg)), acc_par(seg) ^ 1u, sync, 2)) { failed = true; break; }
                    ptx::tc_fence_after();
                    seg_open = true;
                    first = true;
                }
                if (lane == 0) {
                    const uint32_t sfs = kSfCol + 16u * (mx_used & 1u);
                    const uint32_t t_sfa = tmem + sfs, t_sfb = tmem + sfs + 4u;
                    ptx::tmem_cp_32x128b_x4(t_sfa, ptx::smem_desc(ptx::smem_u32(slot.sfa), 128, 128,
                                                                  ptx::kLayoutNone));
#pragma unroll
                    for (int h = 0; h < C::kSfbCopies; ++h)
                        ptx::tmem_cp_32x128b_x4(t_sfb + 4u * h,
                                                ptx::smem_desc(ptx::smem_u32(slot.sfb + 128 * h), 128, 128,
                                                               ptx::kLayoutNone));
                    const uint32_t d = tmem + static_cast<uint32_t>(acc_buf(seg) * BN);
                    for (int j = 0; j < nq; ++j) {
                        const uint64_t ad = ptx::smem_desc(a_st + 32u * j, 16, 1024, ptx::kLayoutSw128);
                        const uint64_t bd = ptx::smem_desc(b_st + 32u * j, 16, 1024, ptx::kLayoutSw128);
                        ptx::mma_mxf8(d, ad, bd, ptx::idesc_sf_ids(idesc_mx, j, j), t_sfa, t_sfb,
                                      first ? 0u : 1u);
                        first = false;
                    }
                }
                ++mx_used;
            } else {
                if (seg_open) {
                    close_segment(0u);
                    seg_open = false;
                }
                const int ngroups = a.blk_k == 128 ? 1 : nq;
                const int steps = a.blk_k == 128 ? nq : 1;
                for (int gidx = 0; gidx < ngroups; ++gidx) {
                    const int b = acc_buf(seg);
                    if (!wait_bar(acce_bar(b), acc_par(seg) ^ 1u, sync, 2)) { failed = true; break; }
                    ptx::tc_fence_after();
                    const int j = gidx;  // scale chunk (blk_k == 128: chunk 0 holds the block scale)
                    for (int r = lane; r < 128; r += 32)
                        info[b].lane_s[r] = slot.lane_raw[j][kSwap ? r / a.blk_n : r];
                    for (int c = lane; c < BN; c += 32) info[b].col_s[c] = slot.col_raw[j][c / col_group];
                    const bool last = it.last_kb() && gidx == ngroups - 1;
                    if (lane == 0) info[b].flags = kInfoPromote | (last ? kInfoLast : 0u);
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                        for (int t = 0; t < steps; ++t) {
                            const int jj = gidx * steps + t;   // 32-wide chunk inside the stage
                            const uint64_t ad = ptx::smem_desc(a_st + 32u * jj, 16, 1024, ptx::kLayoutSw128);
                            const uint64_t bd = ptx::smem_desc(b_st + 32u * jj, 16, 1024, ptx::kLayoutSw128);
                            ptx::mma_f8(d, ad, bd, idesc_f8, t > 0 ? 1u : 0u);
                        }
                        ptx::mbar_arrive(accf_bar(b));
                        ptx::tc_commit(accf_bar(b));
                    }
                    ++seg;
                }
                if (failed) break;
            }
            if (lane == 0) ptx::tc_commit(empty_bar(stage));  // frees the stage when its MMAs finish
            __syncwarp();
            const bool item_end = it.last_kb();
            it.next(a);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            if (item_end && seg_open) {
                close_segment(kInfoLast);
                seg_open = false;
            }
        }
        // Let every tcgen05 op issued above land before teardown.
        if (lane == 0) {
            ptx::tc_commit(drain_bar);
            wait_bar(drain_bar, 0, sync, 5);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        constexpr int kCols = C::kCols;
        constexpr int kLd = C::kLd;
        const int ew = warp - kEpiWarp0;          // 0..7
        const int quad = warp & 3;                // TMEM lane quadrant this warp may access
        const int half = ew >> 2;                 // which half of the columns
        const int r_in_tile = quad * 32 + lane;   // accumulator row (TMEM lane)
        const int c_begin = half * kCols;
        const int epi_tid = ew * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        JobIter it;
        it.begin(a);
        uint32_t seg = 0;
        float acc[kCols];
        while (it.valid(a)) {
            bool failed = false;
            bool first = true;
            while (true) {
                const int b = static_cast<int>(seg % kAccBufs);
                const uint32_t par = (seg / kAccBufs) & 1u;
                if (!wait_bar(accf_bar(b), par, sync, 4)) { failed = true; break; }
                ptx::tc_fence_after();
                const uint32_t flags = info[b].flags;
                const bool promote = (flags & kInfoPromote) != 0u;
                const float ls = promote ? info[b].lane_s[r_in_tile] : 1.0f;
#pragma unroll
                for (int c0 = 0; c0 < kCols; c0 += kLd) {
                    uint32_t r[kLd];
                    ptx::tmem_ld<kLd>(t_lane + static_cast<uint32_t>(b * BN + c_begin + c0), r);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < kLd; ++i) {
                        const float v = __uint_as_float(r[i]);
                        if (promote) {
                            const float sc = ls * info[b].col_s[c_begin + c0 + i];
                            acc[c0 + i] = first ? v * sc : fmaf(v, sc, acc[c0 + i]);
                        } else {
                            acc[c0 + i] = first ? v : acc[c0 + i] + v;
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(acce_bar(b));
                ++seg;
                first = false;
                if (flags & kInfoLast) break;
            }
            if (epi_any(failed || *sync.abort_flag)) break;
            // ------------------------------------------------ output
            const int row0 = it.tr * kBM, col0 = it.tc * BN;
            const int grow = row0 + r_in_tile;   // global row of the MMA A operand
            bool store = true;
            if (a.splits > 1) {
                // fp32 partial of this split; the last split to arrive sums all
                // partials in split order (deterministic) and stores the tile.
                float* part = a.partial + (static_cast<int64_t>(it.tile) * a.splits + it.split) * (kBM * BN) +
                              r_in_tile * BN + c_begin;
#pragma unroll
                for (int c = 0; c < kCols; c += 4)
                    *reinterpret_cast<float4*>(part + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                __threadfence();
                epi_sync();
                if (epi_tid == 0) {
                    const uint32_t old = atomicAdd(a.counters + it.tile, 1u);
                    misc[2] = (old == static_cast<uint32_t>(a.splits - 1)) ? 1u : 0u;
                }
                epi_sync();
                store = misc[2] != 0u;
                if (store) {
                    __threadfence();
                    const float* base = a.partial + static_cast<int64_t>(it.tile) * a.splits * (kBM * BN) +
                                        r_in_tile * BN + c_begin;
                    // p_0 + p_1 + ... in split order, all read back from L2
#pragma unroll
                    for (int c = 0; c < kCols; c += 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(base + c));
                        acc[c] = v.x;
                        acc[c + 1] = v.y;
                        acc[c + 2] = v.z;
                        acc[c + 3] = v.w;
                    }
                    for (int s = 1; s < a.splits; ++s) {
                        const float* p = base + static_cast<int64_t>(s) * (kBM * BN);
#pragma unroll
                        for (int c = 0; c < kCols; c += 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4*>(p + c));
                            acc[c] += v.x;
                            acc[c + 1] += v.y;
                            acc[c + 2] += v.z;
                            acc[c + 3] += v.w;
                        }
                    }
                    if (epi_tid == 0) a.counters[it.tile] = 0u;   // ready for the next launch
                }
            }
            if (store && !kSwap) {
                if (grow < a.M) {
                    __nv_bfloat16* drow = a.D + static_cast<int64_t>(grow) * a.N;
#pragma unroll
                    for (int c = 0; c < kCols; c += 8) {
                        const int gcol = col0 + c_begin + c;
                        if (gcol < a.N) {
                            uint4 v;
                            v.x = pack_bf16x2(acc[c], acc[c + 1]);
                            v.y = pack_bf16x2(acc[c + 2], acc[c + 3]);
                            v.z = pack_bf16x2(acc[c + 4], acc[c + 5]);
                            v.w = pack_bf16x2(acc[c + 6], acc[c + 7]);
                            *reinterpret_cast<uint4*>(drow + gcol) = v;
                        }
                    }
                }
            } else if (store) {
                if (grow < a.N) {
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        const int m = col0 + c_begin + c;
                        if (m < a.M) a.D[static_cast<int64_t>(m) * a.N + grow] = __float2bfloat16_rn(acc[c]);
                    }
                }
            }
            // advance to the next item (skip the remaining k-stages of this one)
            const int cur = it.item;
            while (it.valid(a) && it.item == cur) it.next(a);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// ======================================================================== host

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

// Split-K workspace, one per device, created on first need.
constexpr size_t kWsBytes = size_t(64) << 20;
constexpr int kMaxCounters = 1 << 16;
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
    int bn, tiles_r, tiles_c, kb_total, kb_per_split, splits, items, grid;
};

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

Plan make_plan(int64_t M, int64_t N, int64_t K, int sm_count) {
    Plan p{};
    p.swap = M <= 64;
    p.bn = p.swap ? (M <= 16 ? 16 : (M <= 32 ? 32 : 64)) : 256;
    const int64_t rows = p.swap ? N : M, cols = p.swap ? M : N;
    p.tiles_r = static_cast<int>((rows + kBM - 1) / kBM);
    p.tiles_c = static_cast<int>((cols + p.bn - 1) / p.bn);
    p.kb_total = static_cast<int>((K + kBK - 1) / kBK);
    const int64_t tiles = int64_t(p.tiles_r) * p.tiles_c;
    static const int ovh = env_int("SGQ_SPLIT_OVERHEAD", 2);
    static const int forced = env_int("SGQ_SPLITS", 0);
    int best_s = 1;
    double best = 1e300;
    const int max_s = p.kb_total < 32 ? p.kb_total : 32;
    for (int s = 1; s <= max_s; ++s) {
        const int kbp = (p.kb_total + s - 1) / s;
        if ((p.kb_total + kbp - 1) / kbp != s) continue;   // every split non-empty
        const int64_t items = tiles * s;
        if (s > 1 && (tiles > kMaxCounters ||
                      size_t(items) * kBM * p.bn * sizeof(float) > kWsBytes))
            continue;
        const int64_t waves = (items + sm_count - 1) / sm_count;
        const double cost = double(waves) * (kbp + ovh) + (s > 1 ? 0.5 : 0.0);
        if (forced > 0 ? s == forced : cost < best) {
            best = cost;
            best_s = s;
        }
    }
    p.splits = best_s;
    p.kb_per_split = (p.kb_total + best_s - 1) / best_s;
    p.items = static_cast<int>(tiles * best_s);
    p.grid = p.items < sm_count ? p.items : sm_count;
    return p;
}

template <int BN, int kStages, bool kSwap, int kAccBufs>
sgq_status run(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args, int grid,
               cudaStream_t st) {
    using C = Cfg<BN, kStages, kSwap, kAccBufs>;
    auto kern = fp8_block_gemm_kernel<BN, kStages, kSwap, kAccBufs>;
    static bool configured[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem)) != cudaSuccess)
            return SGQ_ERR_CUDA;
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kNumThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, args) != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

}  // namespace

sgq_status launch_fp8_block_gemm(const void* Aq, const float* As, const void* Wq, const float* Ws,
                                 void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                 uint32_t flags, cudaStream_t st) {
    if (get_encoder() != SGQ_OK) return SGQ_ERR_CUDA;
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    if (di.cc_major != 10 || di.cc_minor != 3) return SGQ_ERR_UNSUPPORTED;
    const Plan p = make_plan(M, N, K, di.sm_count);
    GemmArgs a{};
    a.As = As;
    a.Ws = Ws;
    a.D = static_cast<__nv_bfloat16*>(D);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.blk_n = blk_n;
    a.blk_k = blk_k;
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
    a.force_promote = (flags & SGQ_GEMM_FORCE_PROMOTE) ? 1 : 0;
    if (p.splits > 1) {
        DevWs ws;
        rc = get_workspace(st, &ws);
        if (rc != SGQ_OK) return rc;
        a.partial = ws.partial;
        a.counters = ws.counters;
    }
    CUtensorMap ta, tb;
    const void* opA = p.swap ? Wq : Aq;
    const void* opB = p.swap ? Aq : Wq;
    if (make_tmap(&ta, opA, a.rows, K, kBM) != SGQ_OK) return SGQ_ERR_CUDA;
    if (make_tmap(&tb, opB, a.cols, K, p.bn) != SGQ_OK) return SGQ_ERR_CUDA;
    if (!p.swap) return run<256, 4, false, 1>(ta, tb, a, p.grid, st);
    switch (p.bn) {
        case 16: return run<16, 8, true, 2>(ta, tb, a, p.grid, st);
        case 32: return run<32, 8, true, 2>(ta, tb, a, p.grid, st);
        default: return run<64, 7, true, 2>(ta, tb, a, p.grid, st);
    }
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
    if (dev >= 0 && dev < 64 && g_ws[dev].counters) {
        // an aborted split-K launch may have left arrival counts behind
        if (cudaMemset(g_ws[dev].counters, 0, kMaxCounters * sizeof(uint32_t)) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return SGQ_ERR_CUDA;
    }
    return (v & kStatusTimeout) ? SGQ_ERR_TIMEOUT : SGQ_ERR_CUDA;
}

}  // namespace sgq
