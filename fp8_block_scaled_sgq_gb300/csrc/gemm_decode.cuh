// Decode-sized block-scaled FP8 GEMM for sm_103a (M <= 32 tokens):
//   D = (Aq * As)(Wq * Ws)^T, fp32 accumulation, bf16 out.
//
// The operation is the one of gemm_kernel.cuh (vLLM "scaled_mm" API page,
// AiterInt8ScaledMMLinearKernel.apply_weights docstring, in the "NT" layout of
// sglang PR #42604, Modifications: fp8_gemm_nt((Aq, As), (Wq, Ws), D,
// recipe=(1, blk_n, blk_k))).  At decode sizes the weights are almost all the
// bytes, and a chain of such GEMMs (one layer's linears) is bound by how much
// of each GEMM's weight stream overlaps the previous GEMM, so this kernel is
// organised around that:
//
//  * Work: the weight matrix is cut into units of 128 rows x 128 K (16 KB);
//    unit u is row tile u / kst, K stage u % kst (kst = K / 128).  CTA c of a
//    grid of G takes the contiguous units [c*U/G, (c+1)*U/G) ("stream-K").
//    The host picks G so that a CTA holds about one row tile (for 7168 x 2048:
//    56 CTAs of 16 units, no tile split at all), which leaves most SMs free.
//  * The weights do not depend on the preceding kernel (the library's launch
//    contract), so the producer streams the first kR units into a shared-
//    memory ring and prefetches the rest of its range into L2 without waiting
//    for it.  The next GEMM on the stream launches as soon as this grid has
//    started (programmatic dependent launch) and does the same on the free
//    SMs, so its weights arrive while this grid still works.
//  * The activations are the preceding kernel's output: two loader warps wait
//    for it, then copy the codes and scales (cp.async) -- or quantise the bf16
//    activations themselves (kQuant) -- straight into the ring's token tiles.
//  * MMA: 128 weight rows on the MMA's M side, the BN (16 or 32) tokens on its
//    N side ("swap-AB"); UE8M0 scales through the block-scaled MMA
//    (kind::mxf8f6f4, one scale per row per 32-wide K chunk); a unit whose
//    scales are not all powers of two takes the fp32 promotion step instead.
//    A narrow MMA costs its issuing warp about as much as a wide one, so four
//    warps issue (units at positions pos % 4 of a tile segment, into
//    accumulators of their own), each with elect.sync.
//  * A row tile whose units are split over several CTAs is reduced by the
//    last CTA to arrive, which adds the fp32 partials in CTA order (a fixed
//    order: repeated runs give the same bits); a tile held by one CTA is
//    stored directly.
//
// Warps: 0 producer (weight tiles by TMA, L2 prefetch, weight-scale words),
// 1, 2, 3 and 8 MMA issuers, 4-7 epilogue (TMEM lane quadrants 0-3), 9 and 10
// activation loaders.  Every wait is bounded; on time-out the CTA records a
// status word and leaves through the normal teardown.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstdio>

#include "ptx.cuh"
#include "quant_math.cuh"
#include "sgq_internal.h"

namespace sgq {
namespace dec {

constexpr int kRows = 128;                 // weight rows per unit (MMA M)
constexpr int kUnitK = 128;                // K bytes per unit
constexpr int kUnitBytes = kRows * kUnitK; // weight bytes per unit
constexpr uint64_t kTimeoutNs = 1ull << 30;
constexpr uint64_t kTestTimeoutNs = 1ull << 20;   // about 1 ms
constexpr uint64_t kAbortPollNs = 20000;
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kInfoPromote = 1u;
constexpr uint32_t kInfoLast = 2u;
constexpr int kNI = 4;                     // MMA-issuing warps
constexpr int kWarps = 11;
constexpr int kThreads = 32 * kWarps;
constexpr int kEpi0 = 4;                   // first epilogue warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;           // scale-factor slots after the accumulators
constexpr int kSmemMax = 232448;           // 227 KB per CTA

// MMA issuer index of a warp (warps 1, 2, 3 and 8), or -1.
__device__ __forceinline__ int issuer_of_warp(int w) { return w >= 1 && w <= 3 ? w - 1 : (w == 8 ? 3 : -1); }

struct DecArgs {
    const uint8_t* Aq;      // E4M3 [M, K] (copy mode)
    const float* As;        // fp32 [M, K / blk_k] (copy mode)
    const uint16_t* x;      // bf16 [M, K] (kQuant)
    uint8_t* xq_out;        // kQuant: optional codes out [M, K]
    float* xs_out;          // kQuant: optional scales out [M, K / blk_k]
    const float* Ws;        // fp32 [ceil(N / blk_n), K / blk_k]
    __nv_bfloat16* D;       // bf16 [M, N]
    float* partial;         // fp32 [G][2][BN][128] partial tiles
    uint32_t* counters;     // [tiles] arrival counters (self-resetting)
    uint32_t* status;       // device status word
    int M, N, K, ks;        // ks = K / blk_k
    int tiles, kst, units;  // row tiles, K stages (K / 128), tiles * kst
    int ue8m0, force_promote;
    // Testing (SGQ_GEMM_TEST_TIMEOUT): CTA 0's producer never loads its unit
    // number stall_unit (< 0: off), and waits give up after kTestTimeoutNs.
    int stall_unit;
    unsigned long long* trace;  // per-CTA event timestamps (SGQ_TRACE builds only)
};

// Optional event trace for development builds (-DSGQ_TRACE): one row of
// kTraceSlots globaltimer stamps per CTA.  Slots: 0 start, 1 loaders past the
// grid-dependency wait, 2 / 3 first weight tiles issued / producer done, 4
// first unit full (issuer 0), 5 last MMA issued (issuer 0), 7 loaders' last
// unit released, 8 + 4k .. 11 + 4k tile segment k (k < 5): accumulators read,
// partial published, partials summed, D stored.
constexpr int kTraceSlots = 32;
__device__ __forceinline__ void trace_ev(const DecArgs& a, int slot) {
#ifdef SGQ_TRACE
    if (a.trace != nullptr && slot >= 0 && slot < kTraceSlots)
        a.trace[blockIdx.x * kTraceSlots + slot] = ptx::globaltimer();
#else
    (void)a;
    (void)slot;
#endif
}

template <int BN>
struct alignas(128) Slot {
    uint32_t sfa[128];      // UE8M0 words of the weight rows (tcgen05.cp order)
    uint32_t sfb[128];      // UE8M0 words of the tokens (entries >= BN stay 2^0)
    float wraw[4][4];       // raw weight scales: [n-block of the unit][32-wide K chunk]
    float araw[BN][4];      // raw token scales: [token][chunk]
    uint32_t wok;           // every weight scale of the unit is 2^e
    uint32_t aok[2];        // ... every token scale (per loader warp)
};

template <int BN>
struct alignas(16) Info {
    uint32_t flags;
    uint32_t pad[3];
    float lane_s[128];
    float col_s[BN];
};

template <int BN, int kR, int kBlkN, int kBlkK, bool kQuant>
struct Cfg {
    static constexpr int kBBytes = BN * kUnitK;               // token tile per stage
    static constexpr int kSps = kUnitK / kBlkK;               // scale columns per unit (4 or 1)
    static constexpr int kNblk = kRows / kBlkN;               // weight n-blocks per unit (4 or 1)
    static constexpr size_t kOffW = 0;
    static constexpr size_t kOffB = kOffW + size_t(kR) * kUnitBytes;
    static constexpr size_t kOffSlot = kOffB + size_t(kR) * kBBytes;
    static constexpr size_t kOffInfo = kOffSlot + size_t(kR) * sizeof(Slot<BN>);
    static constexpr size_t kOffBar = kOffInfo + 2 * kNI * sizeof(Info<BN>);
    // barriers: full[kR], empty[kR], accf[kNI][2], acce[kNI][2], drain[kNI]
    static constexpr int kNumBars = 2 * kR + 5 * kNI;
    static constexpr size_t kOffMisc = kOffBar + 8 * kNumBars;
    static constexpr size_t kSmem = kOffMisc + 64 + 1024;     // + 1 KB alignment slack
    static_assert(BN == 16 || BN == 32, "token tile");
    static_assert(kOffB % 1024 == 0 && kBBytes % 1024 == 0, "128-byte swizzle atoms");
    static_assert(kOffSlot % 128 == 0 && kOffInfo % 16 == 0, "slot alignment");
    static_assert(kSmem <= size_t(kSmemMax), "shared memory");
    static_assert(2 * kNI * BN <= int(kSfCol), "accumulators before the scale slots");
    static_assert(kSfCol + 32 * kNI <= kTmemCols, "scale slots");
};

struct Sync {
    volatile uint32_t* abort_flag;
    uint32_t* status;
    uint64_t limit;   // ns a wait may last before the kernel gives up
};

static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((++spins & 15u) == 0) {
            const uint64_t dt = ptx::globaltimer() - t0;
            if (dt > kAbortPollNs && *s.abort_flag) return false;
            if (dt > s.limit) {
                *s.abort_flag = 1u;
                atomicOr(s.status, kStatusTimeout | (where << 8));
                return false;
            }
        }
        if (spins > 8) __nanosleep(32);
    }
}
// Warp-wide bounded wait (lane 0 polls; the result is broadcast).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    uint32_t ok = 1;
    if ((threadIdx.x & 31) == 0 && !ptx::mbar_try_wait(bar, parity)) ok = wait_slow(bar, parity, s, where) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// First unit of CTA c, and the CTA that holds unit u, for U units over G CTAs.
__device__ __forceinline__ int unit_begin(int c, int U, int G) {
    return static_cast<int>((static_cast<int64_t>(c) * U) / G);
}
__device__ __forceinline__ int unit_owner(int u, int U, int G) {
    return static_cast<int>((static_cast<int64_t>(u + 1) * G - 1) / U);
}

// UE8M0 word of one scale row (bytes = exponent fields of the four 32-wide
// chunk scales; one scale per unit is repeated), and whether any scale is not
// a positive normal power of two.
__device__ __forceinline__ uint32_t zero_byte(uint32_t w) { return (w - 0x01010101u) & ~w & 0x80808080u; }
template <int kSps>
__device__ __forceinline__ uint32_t sf_word(const float* row, uint32_t& bad) {
    if constexpr (kSps == 1) {
        const uint32_t b = __float_as_uint(row[0]);
        const uint32_t w = __byte_perm(b << 1, 0u, 0x3333);
        bad |= (b & 0x807FFFFFu) | zero_byte(w) | zero_byte(~w);
        return w;
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(row);
        const uint32_t lo = __byte_perm(v.x << 1, v.y << 1, 0x0073);
        const uint32_t hi = __byte_perm(v.z << 1, v.w << 1, 0x0073);
        const uint32_t w = __byte_perm(lo, hi, 0x5410);
        bad |= ((v.x | v.y | v.z | v.w) & 0x807FFFFFu) | zero_byte(w) | zero_byte(~w);
        return w;
    }
}

// Named barrier 1 over the 128 epilogue threads, plain and as an OR-reduction.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, 1, 128, q;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

template <int BN, int kR, int kBlkN, int kBlkK, bool kQuant>
__global__ void __launch_bounds__(kThreads, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const DecArgs a) {
    using C = Cfg<BN, kR, kBlkN, kBlkK, kQuant>;
    constexpr int kSps = C::kSps;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem + C::kOffW;
    uint8_t* sB = smem + C::kOffB;
    Slot<BN>* slot = reinterpret_cast<Slot<BN>*>(smem + C::kOffSlot);
    Info<BN>* info = reinterpret_cast<Info<BN>*>(smem + C::kOffInfo);   // [issuer * 2 + buffer]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    // misc[0]: TMEM base, misc[1]: abort flag, misc[2]: last-arriver broadcast

    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kR + s); };
    auto accf_bar = [&](int m, int b) { return bar0 + 8u * (2 * kR + m * 2 + b); };
    auto acce_bar = [&](int m, int b) { return bar0 + 8u * (2 * kR + 2 * kNI + m * 2 + b); };
    auto drain_bar = [&](int m) { return bar0 + 8u * (2 * kR + 4 * kNI + m); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Sync sync{reinterpret_cast<volatile uint32_t*>(misc + 1), a.status,
                    a.stall_unit >= 0 ? kTestTimeoutNs : kTimeoutNs};

    const int G = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    const int u0 = unit_begin(cta, a.units, G);
    const int u1 = unit_begin(cta + 1, a.units, G);
    const int nu = u1 - u0;
    const int kst = a.kst;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kR; ++s) {
            // producer: expect_tx + weight-scale words; the two loader warps
            ptx::mbar_init(full_bar(s), 4);
            ptx::mbar_init(empty_bar(s), 1);   // tcgen05.commit of the unit's MMAs
        }
        for (int m = 0; m < kNI; ++m) {
            for (int b = 0; b < 2; ++b) {
                ptx::mbar_init(accf_bar(m, b), 2);   // issuer arrive + tcgen05.commit
                ptx::mbar_init(acce_bar(m, b), 4);   // one arrive per epilogue warp
            }
            ptx::mbar_init(drain_bar(m), 1);
        }
        misc[1] = 0;
        ptx::fence_mbar_init();
    }
    // token words past BN stay 2^0 (0x7F) in every slot
    for (int i = threadIdx.x; i < kR * 128; i += kThreads) slot[i / 128].sfb[i % 128] = 0x7F7F7F7Fu;
    if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmW);
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(misc), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    // The next kernel on the stream may launch now (its weight stream overlaps
    // this grid); it still waits for this grid to finish before it touches
    // anything this grid writes.  Triggered after the TMEM allocation, so a
    // CTA of the next grid can never hold columns this grid still needs.
    if (threadIdx.x == 0) trace_ev(a, 0);

    // A tile segment: the units of row tile t inside this CTA's range.
    auto seg_begin = [&](int t) { return max(u0, t * kst); };
    auto seg_end = [&](int t) { return min(u1, (t + 1) * kst); };
    const int iss = issuer_of_warp(warp);

    if (warp == 0) {
        // --------------------------------------------------- producer
        // Weight tiles by TMA and weight-scale words; no wait for the preceding
        // grid until a ring slot must be reused (weights are static).
        const uint32_t leader = lane == 0 ? 1u : 0u;
        const uint32_t w0 = ptx::smem_u32(sW);
        constexpr int kNblk = C::kNblk;
        constexpr int kNS = kNblk * kSps;   // raw weight scales per unit (<= 16)
        const int nb_total = (a.N + kBlkN - 1) / kBlkN;
        auto tma_unit = [&](int i) {
            const int s = i % kR, u = u0 + i;
            ptx::mbar_arrive_expect_tx_if(leader, full_bar(s), kUnitBytes);
            ptx::tma_load_2d_if(leader, w0 + s * kUnitBytes, &tmW, (u % kst) * kUnitK, (u / kst) * kRows, full_bar(s));
        };
        auto load_scale = [&](int i) -> float {   // lane's raw weight scale of unit i
            const int u = u0 + i, t = u / kst, kb = u % kst;
            const int nb = t * kNblk + lane / kSps;
            return (lane < kNS && nb < nb_total) ? __ldg(a.Ws + static_cast<int64_t>(nb) * a.ks + kb * kSps + lane % kSps)
                                                 : 1.0f;
        };
        const int npre = nu < kR ? nu : kR;
        for (int i = 0; i < npre; ++i)
            if (i != a.stall_unit || cta != 0) tma_unit(i);   // (testing: a unit never loaded)
        if (lane == 0) trace_ev(a, 2);
        // the rest of the range into L2 while the preceding grid runs
        for (int i = kR + lane; i < nu; i += 32) {
            const int u = u0 + i;
            ptx::tma_prefetch_l2_2d(&tmW, (u % kst) * kUnitK, (u / kst) * kRows);
        }
        // raw weight scales of a ring's worth of units, one load each per lane,
        // all in flight together
        float v[kR];
#pragma unroll
        for (int s = 0; s < kR; ++s) v[s] = s < nu ? load_scale(s) : 1.0f;
        bool failed = false;
        for (int base = 0; base < nu && !failed; base += kR) {
#pragma unroll
            for (int s = 0; s < kR; ++s) {
                const int i = base + s;
                if (i >= nu) break;
                if (i >= kR) {
                    // A ring slot frees only once the activations (the preceding
                    // grid's output) are multiplied in: wait for that grid first,
                    // so the bounded wait below never times the preceding kernel.
                    if (i == kR) ptx::grid_dependency_wait();
                    if (!wait_warp(empty_bar(s), ((i / kR) - 1) & 1, sync, 1)) {
                        failed = true;
                        break;
                    }
                    tma_unit(i);
                }
                Slot<BN>& sl = slot[s];
                if (lane < kNS) sl.wraw[lane / kSps][lane % kSps] = v[s];
                if (i + kR < nu) v[s] = load_scale(i + kR);
                __syncwarp();
                const int t = (u0 + i) / kst;
                uint32_t bad = 0, w4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = lane + 32 * j;
                    const bool valid = t * kRows + row < a.N;
                    w4[j] = valid ? sf_word<kSps>(&sl.wraw[row / kBlkN][0], bad) : 0x7F7F7F7Fu;
                }
                *reinterpret_cast<uint4*>(&sl.sfa[lane * 4]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                const bool ok = __all_sync(0xFFFFFFFFu, bad == 0u);
                if (lane == 0) sl.wok = ok ? 1u : 0u;
                ptx::fence_proxy_async_smem();   // the words are read by tcgen05.cp
                __syncwarp();
                ptx::mbar_arrive_if(leader, full_bar(s));
            }
        }
        if (lane == 0) trace_ev(a, 3);
        // The next kernel on the stream may launch now.  Not earlier: its
        // weight stream would queue ahead of this grid's activation and refill
        // loads; from here it overlaps this grid's last MMAs and epilogue.  It
        // still waits for this grid to finish before it touches anything this
        // grid writes.  (Always after the TMEM allocation, so a CTA of the next
        // grid can never hold columns this grid still needs.)
        if (lane == 0) ptx::launch_dependents();
        // After an abort, give weight tiles still in flight time to land
        // before the CTA's shared memory is released.
        if (*sync.abort_flag != 0u) {
            const uint64_t t0 = ptx::globaltimer();
            while (ptx::globaltimer() - t0 < 50000) __nanosleep(1000);
        }
    } else if (warp == 9 || warp == 10) {
        // --------------------------------------------------- activation loaders
        const int lw = warp - 9;
        const int lt = lw * 32 + lane;   // 0 .. 63
        ptx::grid_dependency_wait();     // the activations are the preceding kernel's output
        if (lt == 0) trace_ev(a, 1);
        // A unit is released (its token words built, its full barrier arrived
        // on) once its copies land; before that, every later unit whose ring
        // slot is already free is issued, so all free slots fill together.
        auto release = [&](int i, uint32_t bad) {
            Slot<BN>& sl = slot[i % kR];
            const bool ok = __all_sync(0xFFFFFFFFu, bad == 0u);
            if (lane == 0) sl.aok[lw] = ok ? 1u : 0u;
            ptx::fence_proxy_async_smem();   // token tile and words: read by the tensor core
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(full_bar(i % kR));
        };
        if constexpr (!kQuant) {
            // codes: BN tokens x 8 chunks of 16 bytes, copied into the swizzled
            // token tile; scales: kSps per token into the slot (tokens past M:
            // neither -- their MMA columns are never read back)
            constexpr int kV = BN * 8 / 64;
            auto issue = [&](int n) {
                const int sn = n % kR, kb = (u0 + n) % kst;
                const uint32_t bt = ptx::smem_u32(sB + sn * C::kBBytes);
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int idx = lt + 64 * j, tk = idx >> 3, c = idx & 7;
                    if (tk < a.M)
                        ptx::cp_async_16(bt + tk * 128 + ((c ^ (tk & 7)) << 4),
                                         a.Aq + static_cast<int64_t>(tk) * a.K + kb * kUnitK + c * 16);
                }
                if (lt < BN && lt < a.M) {
                    const float* src = a.As + static_cast<int64_t>(lt) * a.ks + kb * kSps;
                    const uint32_t dst = ptx::smem_u32(&slot[sn].araw[lt][0]);
                    if constexpr (kSps == 4)
                        ptx::cp_async_16(dst, src);
                    else
                        ptx::cp_async_4(dst, src);
                }
                ptx::cp_async_commit();
            };
            // non-blocking: is the ring slot of unit n free (MMAs of unit n - kR done)?
            auto slot_free = [&](int n) -> bool {
                const int r = n / kR;
                uint32_t ok = 1;
                if (r > 0 && lane == 0) ok = ptx::mbar_test_wait(empty_bar(n % kR), (r - 1) & 1) ? 1u : 0u;
                return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0u;
            };
            int issued = 0;
            bool failed = false;
            for (int j = 0; j < nu && !failed; ++j) {
                while (issued <= j) {   // unit j itself must be in flight
                    const int r = issued / kR;
                    if (r > 0 && !wait_warp(empty_bar(issued % kR), (r - 1) & 1, sync, 2)) {
                        failed = true;
                        break;
                    }
                    issue(issued++);
                }
                if (failed) break;
                // units up to j + kR - 1 can use slots freed by units already released
                while (issued < nu && issued < j + kR && slot_free(issued)) issue(issued++);
                ptx::cp_async_wait_pending(issued - 1 - j);   // unit j's copies (this thread's) landed
                uint32_t bad = 0;
                Slot<BN>& sl = slot[j % kR];
                if (lt < BN && lt < a.M) sl.sfb[(lt & 31) * 4 + (lt >> 5)] = sf_word<kSps>(&sl.araw[lt][0], bad);
                release(j, bad);
            }
            ptx::cp_async_wait_pending(0);
        } else {
            // bf16 activations: BN tokens x 16 vectors of 8; the kBlkK / 8
            // neighbouring lanes of a group share its amax (shuffle), as in the
            // stand-alone quantisation kernel, so codes and scales match it.
            // The next unit's loads go out before this unit is quantised.
            constexpr int kV = BN * 16 / 64;
            constexpr int kTpg = kBlkK / 8;
            const bool ue = a.ue8m0 != 0;
            uint4 vn[kV];
            auto load = [&](int i) {
                const int kb = (u0 + i) % kst;
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int idx = lt + 64 * j, tk = idx >> 4, c = idx & 15;
                    vn[j] = tk < a.M ? __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(tk) * a.K +
                                                                            kb * kUnitK + c * 8))
                                     : make_uint4(0, 0, 0, 0);
                }
            };
            load(0);
            for (int i = 0; i < nu; ++i) {
                const int s = i % kR, r = i / kR;
                const int u = u0 + i, t = u / kst, kb = u % kst;
                uint4 v[kV];
#pragma unroll
                for (int j = 0; j < kV; ++j) v[j] = vn[j];
                if (i + 1 < nu) load(i + 1);
                if (r > 0 && !wait_warp(empty_bar(s), (r - 1) & 1, sync, 2)) break;
                uint8_t* bt = sB + s * C::kBBytes;
                Slot<BN>& sl = slot[s];
                uint32_t bad = 0;
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int idx = lt + 64 * j, tk = idx >> 4, c = idx & 15;
                    float f[8];
                    qm::unpack8(v[j], f);
                    float amax = qm::amax8(f);
#pragma unroll
                    for (int off = kTpg / 2; off > 0; off >>= 1)
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
                    const float scl = qm::group_scale(amax, ue);
                    const uint2 q = qm::quantize8(f, scl, ue);
                    *reinterpret_cast<uint2*>(bt + tk * 128 + ((((c >> 1) ^ (tk & 7)) << 4) | ((c & 1) << 3))) = q;
                    const int gq = (c * 8) / kBlkK;
                    const bool lead = (c % kTpg) == 0;
                    const bool tin = tk < a.M;
                    if (lead) sl.araw[tk][gq] = tin ? scl : 0.0f;
                    if (a.xq_out != nullptr && t == 0 && tin) {
                        *reinterpret_cast<uint2*>(a.xq_out + static_cast<int64_t>(tk) * a.K + kb * kUnitK + c * 8) = q;
                        if (lead) a.xs_out[static_cast<int64_t>(tk) * a.ks + kb * kSps + gq] = scl;
                    }
                }
                // A token's 16 vectors sit in one half-warp, so its group scales
                // were all written by this warp: its first lane builds the word.
                __syncwarp();
#pragma unroll
                for (int j = 0; j < kV; ++j) {
                    const int tk = (lt + 64 * j) >> 4;
                    if ((lane & 15) == 0 && tk < a.M)
                        sl.sfb[(tk & 31) * 4 + (tk >> 5)] = sf_word<kSps>(&sl.araw[tk][0], bad);
                }
                release(i, bad);
            }
        }
        if (lt == 0) trace_ev(a, 7);
    } else if (iss >= 0) {
        // --------------------------------------------------- MMA issuers
        // Issuer m takes the units at positions pos % kNI == m of each tile
        // segment, into accumulators of its own (two buffers, so the epilogue
        // of one segment overlaps the next segment's MMAs).
        const int m = iss;
        constexpr uint32_t idesc_f8 = ptx::idesc_f8(kRows, BN);
        constexpr uint32_t idesc_mx = ptx::idesc_mxf8(kRows, BN);
        const uint64_t wd_base = ptx::smem_desc(ptx::smem_u32(sW), 16, 1024, ptx::kLayoutSw128);
        const uint64_t bd_base = ptx::smem_desc(ptx::smem_u32(sB), 16, 1024, ptx::kLayoutSw128);
        const uint64_t sfa_base = ptx::smem_desc(ptx::smem_u32(slot[0].sfa), 128, 128, ptx::kLayoutNone);
        const uint64_t sfb_base = ptx::smem_desc(ptx::smem_u32(slot[0].sfb), 128, 128, ptx::kLayoutNone);
        constexpr uint32_t kSlotStep = sizeof(Slot<BN>) >> 4;
        // (every unit waits for activations: the bounded waits start after the
        // preceding grid, like the loaders')
        ptx::grid_dependency_wait();
        uint32_t seg = 0;       // accumulator segments handed to the epilogue
        uint32_t mx_used = 0;   // block-scaled units issued (scale-slot parity)
        bool seg_open = false;
        uint32_t acc_flag = 0;
        bool failed = false;
        Info<BN>* my_info = info + m * 2;
        auto acc_col = [&](uint32_t sg) { return tmem + static_cast<uint32_t>((m * 2 + (sg & 1u)) * BN); };
        // the segment's buffer must have been read by the epilogue
        auto acquire_buf = [&](uint32_t sg) -> bool {
            if (sg >= 2 && !wait_warp(acce_bar(m, sg & 1u), ((sg >> 1) - 1) & 1u, sync, 3)) return false;
            ptx::tc_fence_after();
            return true;
        };
        auto hand_over = [&](uint32_t sg, uint32_t flags) {
            if (lane == 0) my_info[sg & 1u].flags = flags;
            __syncwarp();
            ptx::mbar_arrive_elect(accf_bar(m, sg & 1u));
            ptx::commit_elect(accf_bar(m, sg & 1u));
        };
        for (int i = 0; i < nu && !failed; ++i) {
            const int s = i % kR, r = i / kR;
            const int u = u0 + i, t = u / kst;
            const int sb = seg_begin(t), se = seg_end(t);
            const int pos = u - sb;
            if (pos % kNI != m) continue;
            const bool my_last = pos + kNI >= se - sb;
            if (!wait_warp(full_bar(s), r & 1, sync, 4)) { failed = true; break; }
            ptx::tc_fence_after();
            if (lane == 0 && m == 0 && i == 0) trace_ev(a, 4);
            Slot<BN>& sl = slot[s];
            const bool mx = sl.wok != 0u && sl.aok[0] != 0u && sl.aok[1] != 0u && a.force_promote == 0;
            const uint64_t wd = wd_base + static_cast<uint64_t>(s * (kUnitBytes >> 4));
            const uint64_t bd = bd_base + static_cast<uint64_t>(s * (C::kBBytes >> 4));
            if (mx) {
                if (!seg_open) {
                    if (!acquire_buf(seg)) { failed = true; break; }
                    seg_open = true;
                    acc_flag = 0;
                }
                const uint32_t t_sfa = tmem + kSfCol + 32u * m + 16u * (mx_used & 1u), t_sfb = t_sfa + 4u;
                const uint64_t so = static_cast<uint64_t>(s) * kSlotStep;
                // scale copies, four MMAs (+32 bytes along K inside the swizzle
                // atom = +2 in the descriptors), and the commit that frees the slot
                ptx::mx_stage_elect(acc_col(seg), wd, bd, ptx::idesc_sf_ids(idesc_mx, 0, 0),
                                    ptx::idesc_sf_ids(idesc_mx, 1, 1), ptx::idesc_sf_ids(idesc_mx, 2, 2),
                                    ptx::idesc_sf_ids(idesc_mx, 3, 3), t_sfa, t_sfb, sfa_base + so, sfb_base + so,
                                    acc_flag, empty_bar(s));
                acc_flag = 1;
                ++mx_used;
            } else {
                if (seg_open) {   // hand the open block-scaled run to the epilogue
                    hand_over(seg, 0u);
                    ++seg;
                    seg_open = false;
                }
                // promotion: one unscaled accumulator per scale group (one per
                // unit for blk_k = 128, one per 32-wide chunk for 32), scaled by
                // the epilogue in fp32
                constexpr int kGroups = kSps;
                constexpr int kSteps = 4 / kGroups;
                for (int g = 0; g < kGroups && !failed; ++g) {
                    if (!acquire_buf(seg)) { failed = true; break; }
                    Info<BN>& inf = my_info[seg & 1u];
                    for (int row = lane; row < 128; row += 32) inf.lane_s[row] = sl.wraw[row / kBlkN][g];
                    for (int c = lane; c < BN; c += 32) inf.col_s[c] = sl.araw[c][g];
                    const uint32_t d = acc_col(seg);
                    for (int j = 0; j < kSteps; ++j) {
                        const int jj = g * kSteps + j;
                        ptx::mma_f8_elect(d, wd + 2u * jj, bd + 2u * jj, idesc_f8, j > 0 ? 1u : 0u);
                    }
                    hand_over(seg, kInfoPromote | ((my_last && g == kGroups - 1) ? kInfoLast : 0u));
                    ++seg;
                }
                if (failed) break;
                ptx::commit_elect(empty_bar(s));   // frees the ring slot when these MMAs are done
            }
            if (my_last && seg_open) {
                hand_over(seg, kInfoLast);
                ++seg;
                seg_open = false;
            }
        }
        if (lane == 0 && m == 0) trace_ev(a, 5);
        // every tcgen05 op issued above lands before teardown
        ptx::commit_elect(drain_bar(m));
        if (lane == 0) wait_slow(drain_bar(m), 0, sync, 5);
        __syncwarp();
    } else {
        // --------------------------------------------------- epilogue (warps 4-7)
        const int ew = warp - kEpi0;
        const int quad = warp & 3;                // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;         // weight row inside the tile (TMEM lane)
        const int et = ew * 32 + lane;            // 0 .. 127
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        ptx::grid_dependency_wait();              // D, the partials and counters are shared with earlier grids
        uint32_t segc[kNI] = {};                  // segments consumed per issuer
        float acc[BN];
        bool failed = false;
        // Adds issuer m's next segment into acc (first: overwrite); true if it
        // was the issuer's last segment of the tile segment.
        auto consume = [&](int m, bool first) -> bool {
            const uint32_t sg = segc[m]++;
            const int b = static_cast<int>(sg & 1u);
            if (!wait_warp(accf_bar(m, b), (sg >> 1) & 1u, sync, 6)) {
                failed = true;
                return true;
            }
            ptx::tc_fence_after();
            const Info<BN>& inf = info[m * 2 + b];
            const uint32_t flags = inf.flags;
            const bool promote = (flags & kInfoPromote) != 0u;
            const float ls = promote ? inf.lane_s[row] : 1.0f;
            const uint32_t col = static_cast<uint32_t>((m * 2 + b) * BN);
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t rr[16];
                ptx::tmem_ld<16>(t_lane + col + static_cast<uint32_t>(c0), rr);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float v = __uint_as_float(rr[k]);
                    if (promote) {
                        const float sc = ls * inf.col_s[c0 + k];
                        acc[c0 + k] = first ? v * sc : fmaf(v, sc, acc[c0 + k]);
                    } else {
                        acc[c0 + k] = first ? v : acc[c0 + k] + v;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(acce_bar(m, b));
            return (flags & kInfoLast) != 0u;
        };
        int t = u0 / kst;
        while (t * kst < u1) {
            const int sb = seg_begin(t), se = seg_end(t);
            // issuer segments in a fixed round-robin order: issuer 0, 1, 2, 3, 0, ...
            // (issuer m has units in the segment only if it is longer than m)
            bool done[kNI];
#pragma unroll
            for (int m = 0; m < kNI; ++m) done[m] = se - sb <= m;
            bool first = true, all_done = false;
            while (!all_done && !failed) {
                all_done = true;
#pragma unroll
                for (int m = 0; m < kNI; ++m) {
                    if (!done[m] && !failed) {
                        done[m] = consume(m, first);
                        first = false;
                    }
                    all_done = all_done && done[m];
                }
            }
            const bool abort_now = failed || *sync.abort_flag != 0u;
            if (epi_any(abort_now)) break;
            const int tk4 = 8 + 4 * (t - u0 / kst);
            if (et == 0) trace_ev(a, tk4);
            const int c_first = unit_owner(t * kst, a.units, G);
            const int c_last = unit_owner((t + 1) * kst - 1, a.units, G);
            const int grow = t * kRows + row;
            const bool live = grow < a.N;
            bool store = true;
            if (c_first != c_last) {
                // partial of this CTA: column-major [BN][128] (a warp's column
                // is one 128-byte line); slot 0 if the tile is this CTA's first
                // segment, else 1
                const int my_slot = (t == u0 / kst) ? 0 : 1;
                float* part = a.partial + (static_cast<int64_t>(cta) * 2 + my_slot) * (BN * kRows) + row;
                if (live) {
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c < a.M) part[c * kRows] = acc[c];
                }
                epi_sync();
                if (et == 0) {
                    // the barrier orders every epilogue thread's partial before this
                    // arrival, whose release publishes them; the last arriver's
                    // acquire makes the other CTAs' partials visible
                    const uint32_t old = ptx::atom_add_acq_rel_gpu(a.counters + t, 1u);
                    misc[2] = old == static_cast<uint32_t>(c_last - c_first) ? 1u : 0u;
                }
                epi_sync();
                store = misc[2] != 0u;
                if (et == 0) trace_ev(a, tk4 + 1);
                if (store && live) {
                    // p(c_first) + p(c_first + 1) + ... + p(c_last), in CTA order;
                    // this CTA's own term from registers.  The loads of four
                    // contributors go out before their adds, 16 columns at a time.
                    constexpr int kSB = 4;
                    const int mc = a.M < BN ? a.M : BN;
#pragma unroll
                    for (int c0 = 0; c0 < BN; c0 += 16) {
                        float sum[16];
                        for (int cc0 = c_first; cc0 <= c_last; cc0 += kSB) {
                            float v[kSB][16];
#pragma unroll
                            for (int h = 0; h < kSB; ++h) {
                                const int cc = cc0 + h;
                                const bool other = cc <= c_last && cc != cta;
                                const int sl = (t == unit_begin(cc, a.units, G) / kst) ? 0 : 1;
                                const float* p = a.partial + (static_cast<int64_t>(cc) * 2 + sl) * (BN * kRows) + row;
#pragma unroll
                                for (int k = 0; k < 16; ++k)
                                    v[h][k] = (other && c0 + k < mc) ? __ldcg(p + (c0 + k) * kRows) : acc[c0 + k];
                            }
#pragma unroll
                            for (int h = 0; h < kSB; ++h) {
                                if (cc0 + h <= c_last) {
#pragma unroll
                                    for (int k = 0; k < 16; ++k) sum[k] = cc0 + h == c_first ? v[h][k] : sum[k] + v[h][k];
                                }
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 16; ++k) acc[c0 + k] = sum[k];
                    }
                }
                if (store && et == 0) {
                    a.counters[t] = 0u;   // ready for the next launch
                    trace_ev(a, tk4 + 2);
                }
            }
            if (store && live) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c < a.M) a.D[static_cast<int64_t>(c) * a.N + grow] = __float2bfloat16_rn(acc[c]);
            }
            if (et == 0) trace_ev(a, tk4 + 3);
            ++t;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

// Ring depth: as many 16 KB weight units as fit in 227 KB beside the token
// tiles, the scale slots and the hand-over records.
template <int BN>
struct Ring {
    static constexpr int kR = BN == 16 ? 11 : 10;
};

// Launches one instantiation with programmatic stream serialisation.
template <int BN, int kBlkN, int kBlkK, bool kQuant>
sgq_status run(const CUtensorMap& tmW, const DecArgs& a, int grid, cudaStream_t st) {
    constexpr int kR = Ring<BN>::kR;
    using C = Cfg<BN, kR, kBlkN, kBlkK, kQuant>;
    auto kern = decode_gemm_kernel<BN, kR, kBlkN, kBlkK, kQuant>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::kSmem)) !=
            cudaSuccess)
            return SGQ_ERR_CUDA;
        configured[dev] = true;
#ifdef SGQ_TRACE
        int nb = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads, C::kSmem);
        cudaFuncAttributes fa{};
        cudaFuncGetAttributes(&fa, kern);
        fprintf(stderr, "decode kernel BN=%d smem=%zu regs=%d: %d CTAs per SM\n", BN, C::kSmem, fa.numRegs, nb);
#endif
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tmW, a) != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

template <int kBlkN, int kBlkK>
sgq_status dispatch(int bn, bool quant, const CUtensorMap& tmW, const DecArgs& a, int grid, cudaStream_t st) {
    if (bn == 16)
        return quant ? run<16, kBlkN, kBlkK, true>(tmW, a, grid, st) : run<16, kBlkN, kBlkK, false>(tmW, a, grid, st);
    return quant ? run<32, kBlkN, kBlkK, true>(tmW, a, grid, st) : run<32, kBlkN, kBlkK, false>(tmW, a, grid, st);
}

// One translation unit per weight-block width (gemm_decode_n32.cu, _n128.cu).
sgq_status dispatch_n32(int blk_k, int bn, bool quant, const CUtensorMap& tmW, const DecArgs& a, int grid,
                        cudaStream_t st);
sgq_status dispatch_n128(int blk_k, int bn, bool quant, const CUtensorMap& tmW, const DecArgs& a, int grid,
                         cudaStream_t st);

}  // namespace dec
}  // namespace sgq
