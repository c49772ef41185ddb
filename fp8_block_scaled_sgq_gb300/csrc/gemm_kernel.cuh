// Block-scaled FP8 GEMM kernel for sm_103a:  D = (Aq * As)(Wq * Ws)^T, bf16 out.
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
//                   the UE8M0 bytes are copied to TMEM (tcgen05.cp) and
//                   applied inside the block-scaled MMA (kind::mxf8f6f4, one
//                   scale per row per 32-wide K chunk); consecutive such
//                   stages accumulate in TMEM;
//                 - otherwise each scale group's partial product is formed
//                   unscaled (kind::f8f6f4) and handed to the epilogue, which
//                   applies the fp32 scales ("promotion").
//   warp 2      scale loader: fetches As/Ws for the stages ahead with
//               cp.async, checks the power-of-two property, and writes the
//               UE8M0 words (laid out for tcgen05.cp) into the stage's slot.
//   warps 3-10  epilogue: tcgen05.ld of the accumulator (each warp its TMEM
//               lane quadrant and half of the columns), fp32 promotion and
//               accumulation in registers, bf16 store, or an fp32 split-K
//               partial plus a last-arriver reduction in split order.
// Small M (<= 64) runs "swap-AB": the weight rows fill the 128-row MMA M
// dimension and the tokens the MMA N dimension (16/32/64), with split-K over
// the persistent grid so the weights stream through all SMs.
//
// Every wait on an mbarrier is bounded; on time-out the CTA records a status
// word, stops issuing work and leaves through the normal teardown.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "ptx.cuh"
#include "quant_math.cuh"
#include "sgq_internal.h"

namespace sgq {
namespace gemm {

constexpr int kBM = 128;          // MMA M: rows of the "A" operand per tile
constexpr int kBK = 128;          // K elements (bytes) per pipeline stage
constexpr int kEpiWarp0 = 3;      // warps: 0 producer, 1 MMA, 2 scale, 3.. epilogue, then scale 2, MMA 2
constexpr uint64_t kTimeoutNs = 1ull << 30;
constexpr uint64_t kTestTimeoutNs = 1ull << 20;   // about 1 ms
// A wait reads the (global) abort flag only once it has lasted this long: the
// load costs a memory round trip, which a wait that is about to complete
// would add to its latency.
constexpr uint64_t kAbortPollNs = 20000;

constexpr uint32_t kInfoPromote = 1u;
constexpr uint32_t kInfoLast = 2u;
constexpr uint32_t kStatusTimeout = 1u;

template <int BN, int kLaneRows, int kColRows>
struct alignas(128) SfSlot {
    uint32_t sfa[128];                  // UE8M0 words of the A operand (tcgen05.cp order)
    uint32_t sfb[(BN + 127) / 128 * 128];  // UE8M0 words of the B operand (128 per tcgen05.cp)
    // Raw fp32 scales of the stage, one row per scale row and 4 columns:
    //   lane_raw: A operand -- activation rows (normal) or weight n-blocks (swap)
    //   col_raw:  B operand -- weight n-blocks (normal) or tokens (swap)
    // Column j holds 32-wide K chunk j; when one scale covers the whole stage
    // (blk_k = 128) it sits in column `kcol`.  With grouped scale loads these
    // are filled only for stages that need the fp32 promotion step.
    float lane_raw[kLaneRows][4];
    float col_raw[kColRows][4];
    uint32_t pow2;                      // every scale of the stage is 2^e
    uint32_t kcol;
    // CTA pair: the peer's pow2 flag (word 0), staged in the peer's slot and
    // copied into the leader's slot by the transfer that signals the stage.
    alignas(16) uint32_t xfer[4];
};

// Raw fp32 scales of up to four consecutive K stages of one item, loaded by
// one TMA box per operand: row r, column c = the scale column of the box's
// first column + c.  Both arrays are TMA destinations: 128-byte aligned.
template <int kLaneRows, int kColRows, int kW>
struct alignas(128) ScaleGroup {
    alignas(128) float lane[kLaneRows][kW];
    alignas(128) float col[kColRows][kW];
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
    uint32_t* status;     // device status word
    unsigned long long* trace;  // per-CTA event timestamps (SGQ_TRACE builds only)
    int M, N, K, ks;      // ks = K / blk_k (columns of As and Ws)
    int rows, cols;       // extents of the MMA A operand and B operand
    int tiles_r, tiles_c, kb_total, kb_per_split, splits, items, group_r;
    int force_promote;
    int prefetch;         // < 0: the configuration's weight prefetch depth; else at most this many stages
};

// Arguments only some configurations read, in a parameter of their own
// (growing GemmArgs costs the other configurations registers).
//  - Fused quantisation: the bf16 activations, UE8M0 rounding of the
//    activation scales, and optional outputs for the codes [M, K] and scales
//    [M, K/blk_k] (written by the CTAs of the first weight tile row; null: not
//    written).
//  - Per-channel scaling (fp8_scaled_mm): A scales (1 or M values), B scales
//    (1 or N values) and an optional bf16 bias [N].
struct ExtArgs {
    const uint16_t* x;   // bf16 activations [M, K]
    uint8_t* xq_out;
    float* xs_out;
    int ue8m0;
    const float* sa;
    const float* sb;
    const uint16_t* bias;
    int sa_n, sb_n;
    // Testing (SGQ_GEMM_TEST_TIMEOUT): CTA 0's producer never loads its job
    // number stall_job (< 0: off), and waits give up after kTestTimeoutNs.
    int stall_job;
};

// Walks the (item, k-stage) jobs of one CTA (or CTA pair) in order.
struct JobIter {
    int item, kb, kb0, nkb, pos, step;
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
        kb0 = split * a.kb_per_split;
        nkb = min(a.kb_total, kb0 + a.kb_per_split) - kb0;
        pos = 0;
        kb = kb0;
    }
    // first item and stride: the CTA's (or CTA pair's) index and count
    __device__ void begin(const GemmArgs& a, int first, int stride) {
        item = first;
        step = stride;
        if (item < a.items) load(a);
    }
    __device__ bool valid(const GemmArgs& a) const { return item < a.items; }
    __device__ bool last_kb() const { return pos + 1 == nkb; }
    // Advances one stage; returns true when it moved to a new item.
    __device__ bool next(const GemmArgs& a) {
        if (++pos >= nkb) {
            item += step;
            if (item < a.items) load(a);
            return true;
        }
        kb = kb0 + pos;
        return false;
    }
};

// Optional event trace for development builds (-DSGQ_TRACE): one row of
// kTraceSlots globaltimer stamps per CTA.  Compiled out otherwise.  Slots:
//   0 CTA start, 1 producer past the grid-dependency wait, 2 its weight
//   prefetch issued, 3 its prologue done, 4 epilogue past the wait (fused),
//   5 producer entering its main loop, 8+j stage j issued (j mod 32),
//   40+j MMA issuer saw stage j full, 72+j scale words of stage j ready,
//   104+j scale warp saw stage j's raw scales (or its quantised codes),
//   136/137/138/139 + 4i item i: accumulators read, split-K partial sent,
//   item done, last accumulator segment picked (i mod 16), 200+j MMA job j
//   issued, 216+j observed full barrier (alternating issuers), 232+w / 244+w
//   warp w before / after the final barrier, 255 CTA end.
constexpr int kTraceSlots = 256;
__device__ __forceinline__ void trace_ev(const GemmArgs& a, int slot) {
#ifdef SGQ_TRACE
    if (a.trace != nullptr && slot >= 0 && slot < kTraceSlots)
        a.trace[blockIdx.x * kTraceSlots + slot] = ptx::globaltimer();
#else
    (void)a;
    (void)slot;
#endif
}

struct Sync {
    volatile uint32_t* abort_flag;
    uint32_t* status;
    uint64_t limit;   // ns a wait may last before the kernel gives up (kTimeoutNs unless testing)
};

// kCl: acquire at cluster scope (barriers that the other CTA of a pair arrives on).
template <bool kCl>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    return kCl ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
}
template <bool kCl>
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where,
                                              bool backoff) {
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (try_wait_scoped<kCl>(bar, parity)) return true;
        if ((++spins & 15u) == 0) {
            const uint64_t dt = ptx::globaltimer() - t0;
            if (dt > kAbortPollNs && *s.abort_flag) return false;
            if (dt > s.limit) {
                *s.abort_flag = 1u;
                atomicOr(s.status, kStatusTimeout | (where << 8));
                return false;
            }
        }
        if (backoff && spins > 8) __nanosleep(64);
    }
}
// Single-thread bounded wait.
template <bool kCl = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where) {
    if (try_wait_scoped<kCl>(bar, parity)) return true;
    return wait_slow<kCl>(bar, parity, s, where, false);
}
// Warp-wide bounded wait: lane 0 polls (the other lanes park at the warp
// barrier, keeping shared-memory traffic off the TMA path), then the result is
// broadcast.  __syncwarp orders lane 0's acquire before the other lanes' reads.
template <bool kCl = false>
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Sync& s, uint32_t where,
                                              bool backoff) {
    uint32_t ok = 1;
    if ((threadIdx.x & 31) == 0 && !try_wait_scoped<kCl>(bar, parity))
        ok = wait_slow<kCl>(bar, parity, s, where, backoff) ? 1u : 0u;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Named barrier 1 over the epilogue warps (kThr threads).
template <int kThr>
__device__ __forceinline__ bool epi_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\n"
        "bar.red.or.pred p, 1, %2, q;\nselp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "n"(kThr)
        : "memory");
    return r != 0;
}
template <int kThr>
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThr) : "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Bits of a scale that must be zero for it to be a UE8M0 value 2^e (sign and
// mantissa), and its exponent byte.
__device__ __forceinline__ uint32_t scale_bad_bits(uint32_t b) {
    const uint32_t e = b >> 23;
    return (b & 0x807FFFFFu) | static_cast<uint32_t>(e == 0u || e == 0xFFu);
}

// UE8M0 word of one scale row: byte q = exponent byte of the chunk-q scale
// (kNld == 1: the one scale at column kcol, repeated).  `bad` collects any
// scale that is not a positive normal power of two.
__device__ __forceinline__ uint32_t has_zero_byte(uint32_t w) { return (w - 0x01010101u) & ~w & 0x80808080u; }
template <int kNld>
__device__ __forceinline__ uint32_t sf_word(const float* row, int kcol, uint32_t& bad) {
    if (kNld == 1) {
        const uint32_t b = __float_as_uint(row[kcol]);
        const uint32_t w = __byte_perm(b << 1, 0u, 0x3333);
        bad |= (b & 0x807FFFFFu) | has_zero_byte(w) | has_zero_byte(~w);
        return w;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(row);
    const uint32_t lo = __byte_perm(v.x << 1, v.y << 1, 0x0073);
    const uint32_t hi = __byte_perm(v.z << 1, v.w << 1, 0x0073);
    const uint32_t w = __byte_perm(lo, hi, 0x5410);
    bad |= ((v.x | v.y | v.z | v.w) & 0x807FFFFFu) | has_zero_byte(w) | has_zero_byte(~w);
    return w;
}

template <int BN, int kStages, bool kSwap, int kAccBufs, int kBlkN, int kBlkK, bool kScaleTma, bool kPair,
          bool kAlt, bool kFuse, bool kChan, bool kCK>
struct Cfg {
    // Swap-AB tiles are narrow (N <= 64): an MMA costs about as much to issue
    // as a full-width one, so two warps issue alternate K stages of each item
    // into separate accumulators, which the epilogue adds in a fixed order.
    // kAlt (wide tiles): two warps take turns issuing the K stages into the
    // one accumulator, each preparing its next stage while the other issues.
    static constexpr int kMmaWarps = (kSwap || kAlt) ? 2 : 1;
    static constexpr int kAccSets = kSwap ? kMmaWarps : 1;   // accumulator sets (one per swap issuer)
    // Two CTAs per SM (registers, shared memory, TMEM sized for it; four
    // epilogue warps, one per TMEM lane quadrant) would let the next GEMM on
    // the stream become resident and stream its weights while this one runs.
    // Measured on decode tiles it is slower (the two GEMMs' loads share the
    // SM's TMA queue and the activation tiles wait behind the next GEMM's
    // weights), so no configuration uses it; the layout stays parametrised.
    static constexpr bool kTwoPerSm = false;
    static constexpr int kEpiWarps = kTwoPerSm ? 4 : 8;
    // Scale warps: two take alternate stages; with alternating issuers one
    // does all stages and the second's place goes to the second issuer (a
    // 13th warp would cap registers at 128, as one SM sub-partition would
    // hold four warps, and the 128-column epilogue would spill).
    static constexpr int kSfWarps = kAlt ? 1 : 2;
    static constexpr int kSf2Warp = kEpiWarp0 + kEpiWarps;                    // second scale warp
    static constexpr int kMma2Warp = kEpiWarp0 + kEpiWarps + (kSfWarps - 1);  // second MMA issuer
    static constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps + (kSfWarps - 1) + (kMmaWarps - 1));
    static constexpr int kMinBlocks = kTwoPerSm ? 2 : 1;
    // TMEM: accumulators from column 0, then two 16-column scale slots per issuer
    static constexpr uint32_t kTmemCols = kTwoPerSm ? 128u : 512u;
    static constexpr uint32_t kSfCol = kTmemCols - 32u;
    // Weight stages loaded before the programmatic-dependency wait.  Loads of
    // one SM leave in issue order, so a deep weight prefetch delays the first
    // activation tiles behind it; the swap-AB (decode) tiles start with none.
    // With fused quantisation no activation tile goes through the TMA, so all
    // ring stages of weights (and their scale boxes) go out before the wait.
    static constexpr int kPrefetch = kFuse ? kStages : ((kSwap && !kTwoPerSm) ? 0 : kStages);
    // CTA pair (cluster of two, cta_group::2): the tile is 256 x BN; each CTA
    // holds 128 A rows and BN/2 B rows per stage, the leader issues the MMAs.
    static constexpr int kCG = kPair ? 2 : 1;
    static constexpr int kTileRows = kBM * kCG;            // A rows per tile
    static constexpr int kABytes = kBM * kBK;
    static constexpr int kBBytes = (BN / kCG) * kBK;       // B bytes per CTA and stage
    static constexpr uint32_t kXferBytes = kPair ? 16u : 0u;      // the peer's scale-ready transfer
    // Fused quantisation (swap-AB): the epilogue warps read each stage's bf16
    // activation tile with plain loads and write its E4M3 codes into the
    // stage's B tile; the full barrier counts only the weight tile's bytes.
    // The epilogue warps quantise, all of them on each stage in turn: the
    // first stage, which the MMAs wait for, is ready soonest that way
    // (measured: one warp per stage, eight stages at a time, was slower).
    static constexpr int kQW = kEpiWarps;
    static constexpr int kStageBytes = kFuse ? kABytes : kCG * (kABytes + kBBytes) + kXferBytes;
    static constexpr int kCols = BN * 4 / kEpiWarps;  // accumulator columns per epilogue thread
    static constexpr int kLd = kCols < 16 ? kCols : 16;
    static constexpr int kSfbCopies = (BN + 127) / 128;
    static constexpr int kNld = kBlkK == 128 ? 1 : 4;    // distinct scale chunks per stage
    static constexpr int kScalesPerStage = kBK / kBlkK;  // As/Ws columns per stage
    static constexpr int kColGroups = kSwap ? BN : (BN + kBlkN - 1) / kBlkN;
    static constexpr int kLaneGroups = kSwap ? kBM / kBlkN : kBM;
    // rows of the raw scale boxes (A-operand side, B-operand side)
    static constexpr int kLaneScaleRows = kSwap ? kBM / kBlkN : kBM;
    static constexpr int kColScaleRows = kSwap ? BN : (BN + kBlkN - 1) / kBlkN;
    using Slot = SfSlot<BN, kLaneScaleRows, kColScaleRows>;
    // Grouped scale loads (TMA path): each TMA operation costs an SM about the
    // same time whatever its size, so one box per operand brings the scales of
    // kG consecutive stages.  Box: kGW columns (for one scale per stage, 8, so
    // that a group starting at any column fits behind a 16-byte aligned start).
    static constexpr int kG = 4;
    static constexpr int kGW = kScalesPerStage == 1 ? 8 : kG * kScalesPerStage;
    using Group = ScaleGroup<kLaneScaleRows, kFuse ? 1 : kColScaleRows, kGW>;   // fused: no token box
    static constexpr int kGBufs = 2;
    static constexpr uint32_t kGroupBytes = 4u * kGW * (kLaneScaleRows + (kFuse ? 0 : kColScaleRows));
    static constexpr size_t kOffA = 0;
    static constexpr size_t kOffB = kOffA + size_t(kStages) * kABytes;
    static constexpr size_t kOffSf = kOffB + size_t(kStages) * kBBytes;
    static constexpr size_t kOffGrp = kOffSf + size_t(kStages) * sizeof(Slot);
    static constexpr size_t kOffInfo = kOffGrp + (kScaleTma ? size_t(kGBufs) * sizeof(Group) : 0);
    // Split-K over a cluster of two (kCK): split 1's fp32 partial tile goes to
    // split 0's shared memory in one bulk copy (both CTAs hold this buffer).
    static constexpr int kCKBytes = kCK ? kBM * BN * 4 : 0;
    static constexpr size_t kOffCK = kOffInfo + size_t(kAccSets * kAccBufs) * sizeof(Info<BN>);
    static constexpr size_t kOffBar = kOffCK + size_t(kCKBytes);
    static constexpr int kHandBar0 = 3 * kStages + (2 * kAccBufs + 1) * kMmaWarps + 2 * kGBufs;
    static constexpr int kQBar0 = kHandBar0 + (kAlt ? 2 : 0);
    static constexpr int kCKBar0 = kQBar0 + (kFuse ? kStages : 0);
    static constexpr int kNumBars = kCKBar0 + (kCK ? 2 : 0);
    static constexpr size_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr size_t kSmem = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(kAccSets * kAccBufs * BN <= int(kSfCol) - 32 * (kMmaWarps - 1), "TMEM budget");
    static_assert(!kAlt || (!kSwap && !kPair), "alternating issuers: single-CTA wide tiles");
    static_assert(!kFuse || (kSwap && kScaleTma), "fused quantisation: swap-AB tiles with TMA scale groups");
    static_assert(!kChan || (!kPair && !kAlt && !kFuse && !kScaleTma), "per-channel scaling: plain tiles");
    static_assert(!kCK || (kSwap && !kPair && !kAlt), "cluster split-K: swap-AB tiles");
    static_assert(kOffCK % 16 == 0, "bulk-copy buffer alignment");
    static_assert(kOffSf % 128 == 0, "scale slots aligned");
    static_assert(!kTwoPerSm || kSmem <= 113 * 1024, "two CTAs per SM: shared memory");
    static_assert(!kSwap || BN <= 64, "swap-AB token tile");
    static_assert(!kPair || (!kSwap && BN == 256 && kScaleTma && kAccBufs == 1), "CTA-pair configuration");
    static_assert(kColGroups <= 64, "raw column-scale slot");
    static_assert(kGW * 4 % 16 == 0, "scale box row: whole 16-byte units");
    static_assert(offsetof(Group, lane) % 128 == 0 && offsetof(Group, col) % 128 == 0 && sizeof(Group) % 128 == 0,
                  "TMA destinations in a scale group start on 128-byte boundaries");
    static_assert(kOffGrp % 128 == 0, "scale groups start on a 128-byte boundary");
    static_assert(kStages <= 8, "cp.async group depth");
    static_assert(kSmem <= 232448, "shared memory budget");
};

template <int BN, int kStages, bool kSwap, int kAccBufs, int kBlkN, int kBlkK, bool kScaleTma, bool kPair,
          bool kAlt, bool kFuse, bool kChan, bool kCK>
__global__ void __launch_bounds__(
    (Cfg<BN, kStages, kSwap, kAccBufs, kBlkN, kBlkK, kScaleTma, kPair, kAlt, kFuse, kChan, kCK>::kThreads),
    (Cfg<BN, kStages, kSwap, kAccBufs, kBlkN, kBlkK, kScaleTma, kPair, kAlt, kFuse, kChan, kCK>::kMinBlocks))
    fp8_block_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                          const GemmArgs a, const ExtArgs fz) {
    using C = Cfg<BN, kStages, kSwap, kAccBufs, kBlkN, kBlkK, kScaleTma, kPair, kAlt, kFuse, kChan, kCK>;
    constexpr int kCG = C::kCG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + C::kOffA;
    uint8_t* sB = smem + C::kOffB;
    typename C::Slot* sf = reinterpret_cast<typename C::Slot*>(smem + C::kOffSf);
    typename C::Group* grp = reinterpret_cast<typename C::Group*>(smem + C::kOffGrp);
    Info<BN>* info = reinterpret_cast<Info<BN>*>(smem + C::kOffInfo);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    // misc[0]: TMEM base, misc[1]: abort flag, misc[2]: epilogue broadcast,
    // misc[4..5]: accumulator state passed between alternating issuers

    const uint32_t bar0 = ptx::smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    // accumulator barriers per (MMA warp m, buffer b)
    constexpr int kMW = C::kMmaWarps;
    auto accf_bar = [&](int m, int b) { return bar0 + 8u * (2 * kStages + m * kAccBufs + b); };
    auto acce_bar = [&](int m, int b) { return bar0 + 8u * (2 * kStages + (kMW + m) * kAccBufs + b); };
    auto drain_bar = [&](int m) { return bar0 + 8u * (2 * kStages + 2 * kMW * kAccBufs + m); };
    auto sraw_bar = [&](int s) { return bar0 + 8u * (2 * kStages + (2 * kAccBufs + 1) * kMW + s); };
    // scale-group ring: loaded (TMA) / released (both scale warps)
    auto gfull_bar = [&](int d) { return bar0 + 8u * (3 * kStages + (2 * kAccBufs + 1) * kMW + d); };
    auto gempty_bar = [&](int d) { return bar0 + 8u * (3 * kStages + (2 * kAccBufs + 1) * kMW + C::kGBufs + d); };
    // alternating issuers: the turn token of issuer w
    auto hand_bar = [&](uint32_t w) { return bar0 + 8u * (C::kHandBar0 + w); };
    // fused quantisation: stage s's codes and scales written (epilogue warps)
    auto qdone_bar = [&](int s) { return bar0 + 8u * (C::kQBar0 + s); };
    // cluster split-K: partial landed in split 0 / split 0 done reading (in split 1)
    auto ckfull_bar = [&]() { return bar0 + 8u * C::kCKBar0; };
    auto ckfree_bar = [&]() { return bar0 + 8u * (C::kCKBar0 + 1); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Sync sync{reinterpret_cast<volatile uint32_t*>(misc + 1), a.status,
                    fz.stall_job >= 0 ? kTestTimeoutNs : kTimeoutNs};
    // CTA pair: rank 0 leads (issues every tcgen05 op of the pair); a pair
    // walks the items with index blockIdx.x / 2.
    const uint32_t rank = kPair ? ptx::cluster_rank() : 0u;
    const int first_item = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int item_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    // first activation row of this CTA's share of the tile
    auto a_row0 = [&](const JobIter& j) { return j.tr * C::kTileRows + static_cast<int>(rank) * kBM; };
    // the same barrier in the leader (cluster address)
    auto at_leader = [&](uint32_t bar) { return kPair ? ptx::mapa(bar, 0u) : bar; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // producer expect_tx + scale loader (pair: the peer's scale loader
            // signals with a transfer counted in the expected bytes)
            ptx::mbar_init(full_bar(s), kChan ? 1 : 2);   // per-channel scaling: no scale warps
            ptx::mbar_init(empty_bar(s), 1);  // tcgen05.commit
        }
        for (int m = 0; m < kMW; ++m) {
            for (int b = 0; b < kAccBufs; ++b) {
                ptx::mbar_init(accf_bar(m, b), 2);   // MMA thread arrive + tcgen05.commit
                // one arrive per epilogue warp (pair leader: of both CTAs)
                ptx::mbar_init(acce_bar(m, b), C::kEpiWarps * (kPair ? 2 : 1));
            }
            ptx::mbar_init(drain_bar(m), 1);
        }
        for (int s = 0; s < kStages; ++s) ptx::mbar_init(sraw_bar(s), 1);   // raw scales landed (cp.async path)
        for (int d = 0; d < C::kGBufs; ++d) {
            ptx::mbar_init(gfull_bar(d), 1);    // producer expect_tx
            ptx::mbar_init(gempty_bar(d), C::kSfWarps);   // one arrive per scale warp
        }
        if (kAlt) {
            ptx::mbar_init(hand_bar(0), 1);
            ptx::mbar_init(hand_bar(1), 1);
        }
        if constexpr (kFuse)
            for (int s = 0; s < kStages; ++s) ptx::mbar_init(qdone_bar(s), C::kQW);
        if constexpr (kCK) {
            ptx::mbar_init(ckfull_bar(), 1);   // split 0's expect_tx; the bulk copy brings the bytes
            ptx::mbar_init(ckfree_bar(), 1);   // split 0's remote arrive
        }
        misc[1] = 0;
        misc[4] = 0;
        misc[5] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if (kScaleTma) {
            ptx::prefetch_tmap(&tmSA);
            ptx::prefetch_tmap(&tmSB);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc_g<kCG>(ptx::smem_u32(misc), C::kTmemCols);
        ptx::tmem_relinquish_g<kCG>();
    }
    ptx::tc_fence_before();
    __syncthreads();
    // Both CTAs' barriers exist before any remote arrive.  Cluster split-K
    // only arrives here and waits just before its first remote operation (in
    // the epilogue, or at exit): the weight stream does not wait on the peer.
    if (kPair) ptx::cluster_sync();
    if (kCK) ptx::cluster_arrive_relaxed();
    bool ck_wait_pending = kCK;
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    if (threadIdx.x == 0) {
        trace_ev(a, 0);
        // The next kernel on the stream may launch now; it still waits for this
        // grid to finish (griddepcontrol.wait) before touching its outputs.
        ptx::launch_dependents();
    }

    // Fused quantisation, by the epilogue warps: vector v (8 consecutive
    // elements; v = token * 16 + chunk) of stage s's bf16 activation tile,
    // held in registers, becomes 8 E4M3 codes in the stage's B tile (the
    // 128-byte swizzled layout the TMA would have written), and its group's
    // fp32 scale goes to the slot's col_raw, 0 for groups past K or tokens past
    // M (as the scale box would read them).  kBlkK/8 neighbouring lanes share a
    // group (shuffle amax), as in the stand-alone quantisation kernel, so the
    // codes and scales are the same.
    constexpr int kVpt = kFuse ? BN * 16 / (C::kEpiWarps * 32) : 1;   // vectors per thread and stage
    auto x_vec = [&](const JobIter& j, int v) -> uint4 {
        const int tk = v >> 4, c = v & 15;
        const int row = j.tc * BN + tk, k = j.kb * kBK + c * 8;
        if (row >= a.M || k >= a.K) return make_uint4(0, 0, 0, 0);
        return __ldg(reinterpret_cast<const uint4*>(fz.x + static_cast<int64_t>(row) * a.K + k));
    };
    auto quantize_vec = [&](const uint4& w, int v, int s, const JobIter& j, typename C::Slot& slot) {
        constexpr int kTpg = kBlkK / 8;
        uint8_t* bq = sB + s * C::kBBytes;
        const int col0 = j.tc * BN;
        const int kbase = j.kb * kBK;
        const bool ue = fz.ue8m0 != 0;
        const int tk = v >> 4, c = v & 15;
        float f[8];
        qm::unpack8(w, f);
        float amax = qm::amax8(f);
#pragma unroll
        for (int off = kTpg / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        const float sc = qm::group_scale(amax, ue);
        const uint2 q = qm::quantize8(f, sc, ue);
        *reinterpret_cast<uint2*>(bq + tk * 128 + ((((c >> 1) ^ (tk & 7)) << 4) | ((c & 1) << 3))) = q;
        const int gq = (c * 8) / kBlkK;               // scale column within the stage
        const bool kin = kbase + gq * kBlkK < a.K;    // the group lies inside K
        const bool tin = col0 + tk < a.M;
        const bool leader_lane = (v % kTpg) == 0;
        if (leader_lane) slot.col_raw[tk][gq] = (kin && tin) ? sc : 0.0f;
        if (fz.xq_out != nullptr && j.tr == 0 && kin && tin) {
            const int64_t row = col0 + tk;
            *reinterpret_cast<uint2*>(fz.xq_out + row * a.K + kbase + c * 8) = q;
            if (leader_lane) fz.xs_out[row * a.ks + j.kb * C::kScalesPerStage + gq] = sc;
        }
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // The weight operand does not depend on the preceding kernel, so the
        // weight halves of the first C::kPrefetch stages go out before the
        // programmatic-dependency wait; activations only after it.
        // The whole warp runs the loop; lane 0 issues through predicated asm.
        {
            const uint32_t leader = lane == 0 ? 1u : 0u;
            const CUtensorMap* tmW = kSwap ? &tmA : &tmB;
            const CUtensorMap* tmX = kSwap ? &tmB : &tmA;
            const CUtensorMap* tmWs = kSwap ? &tmSA : &tmSB;   // weight scales
            const CUtensorMap* tmXs = kSwap ? &tmSB : &tmSA;   // activation scales
            const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
            auto w_dst = [&](int s) { return kSwap ? sA0 + s * C::kABytes : sB0 + s * C::kBBytes; };
            auto x_dst = [&](int s) { return kSwap ? sB0 + s * C::kBBytes : sA0 + s * C::kABytes; };
            auto w_row = [&](const JobIter& j) {
                return kSwap ? j.tr * kBM : j.tc * BN + static_cast<int>(rank) * (BN / kCG);
            };
            auto x_row = [&](const JobIter& j) { return kSwap ? j.tc * BN : a_row0(j); };
            auto ws_row = [&](const JobIter& j) { return kSwap ? j.tr * (kBM / kBlkN) : j.tc * (BN / kBlkN); };
            auto xs_row = [&](const JobIter& j) { return kSwap ? j.tc * BN : a_row0(j); };
            // Operand tiles signal the stage's full barrier; with a CTA pair both
            // CTAs' tiles land on the leader's, which expects the bytes of both.
            auto load_tile = [&](uint32_t dst, const CUtensorMap* m, int32_t x, int32_t y, int s) {
                if (kPair)
                    ptx::tma_load_2d_pair_if(leader, dst, m, x, y, at_leader(full_bar(s)));
                else
                    ptx::tma_load_2d_if(leader, dst, m, x, y, full_bar(s));
            };
            auto load_w = [&](int s, const JobIter& j) {
                ptx::mbar_arrive_expect_tx_if(leader && rank == 0u, full_bar(s), C::kStageBytes);
                load_tile(w_dst(s), tmW, j.kb * kBK, w_row(j), s);
            };
            auto load_x = [&](int s, const JobIter& j) {
                if constexpr (!kFuse) load_tile(x_dst(s), tmX, j.kb * kBK, x_row(j), s);
            };
            // Scale group: at the first stage of every kG-stage group of an item,
            // one box per operand with the raw scales of the whole group.
            uint32_t gcount = 0;
            bool group_ok = true;
            auto load_group = [&](const JobIter& j) {
                if (!kScaleTma || (j.pos % C::kG) != 0) return;
                const int d = static_cast<int>(gcount % C::kGBufs);
                if (!wait_bar(gempty_bar(d), ((gcount / C::kGBufs) & 1u) ^ 1u, sync, 1)) {
                    group_ok = false;
                    return;
                }
                const int gx = (j.kb * C::kScalesPerStage) & ~3;   // 16-byte aligned first column
                typename C::Group& g = grp[d];
                ptx::mbar_arrive_expect_tx_if(leader, gfull_bar(d), C::kGroupBytes);
                const uint32_t lane_dst = ptx::smem_u32(&g.lane[0][0]), col_dst = ptx::smem_u32(&g.col[0][0]);
                ptx::tma_load_2d_if(leader, kSwap ? lane_dst : col_dst, tmWs, gx, ws_row(j), gfull_bar(d));
                // (fused quantisation computes the activation scales itself)
                if constexpr (!kFuse)
                    ptx::tma_load_2d_if(leader, kSwap ? col_dst : lane_dst, tmXs, gx, xs_row(j), gfull_bar(d));
                ++gcount;
            };
            JobIter it;
            it.begin(a, first_item, item_step);
            JobIter pre = it;
            int npre = 0;
            const int prefetch = a.prefetch >= 0 && a.prefetch < C::kPrefetch ? a.prefetch : C::kPrefetch;
            while (npre < prefetch && pre.valid(a)) {
                if constexpr (kFuse) load_group(pre);   // weight scales only: static like the weights
                load_w(npre, pre);
                pre.next(a);
                ++npre;
            }
            if (lane == 0) trace_ev(a, 2);
            // Without a weight prefetch the wait sits inside the first loop
            // iteration, after that stage's weight load: the loop's code is
            // fetched while the warp waits, not after.
            bool dep_waited = npre > 0;
            if (dep_waited) {
                ptx::grid_dependency_wait();
                if (lane == 0) trace_ev(a, 1);
                for (int s = 0; s < npre && group_ok; ++s) {
                    if constexpr (!kFuse) {
                        load_group(it);
                        load_x(s, it);
                    }
                    it.next(a);
                }
            }
            if (lane == 0) trace_ev(a, 3);
            int stage = npre % kStages;
            uint32_t phase = npre / kStages;
            int nj = npre;
            while (it.valid(a) && group_ok) {
                if (lane == 0 && nj == npre) trace_ev(a, 5);
                if (!wait_bar(empty_bar(stage), phase ^ 1u, sync, 1)) break;
                if (lane == 0) trace_ev(a, 8 + (nj & 31));
                ++nj;
                if (nj - 1 == fz.stall_job && blockIdx.x == 0) {   // testing: this job is never loaded
                    it.next(a);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                    continue;
                }
                load_w(stage, it);
                if (!dep_waited) {
                    ptx::grid_dependency_wait();
                    dep_waited = true;
                    if (lane == 0) trace_ev(a, 1);
                }
                load_group(it);
                load_x(stage, it);
                it.next(a);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
        __syncwarp();
    } else if (!kChan && (warp == 2 || (C::kSfWarps > 1 && warp == C::kSf2Warp))) {
        // ---------------------------------------------------------- scale loader
        // Turns each stage's raw fp32 scales into UE8M0 words in tcgen05.cp
        // order, checks the power-of-two property, and releases the stage to
        // the MMA warp (second arrival on its full barrier).
        //
        // Fast path (kScaleTma): the producer loads the raw scale boxes with
        // TMA together with the operand tiles, so they arrive kStages ahead;
        // this warp only converts.  Fallback (scale rows not 16-byte aligned):
        // this warp fetches the raw scales itself with cp.async, up to kStages
        // jobs ahead of the conversion.
        constexpr int kNld = C::kNld;
        constexpr int kLR = C::kLaneScaleRows, kCR = C::kColScaleRows;
        auto convert = [&](typename C::Slot& slot, const JobIter& j, int kcol) {
            const int row0 = kSwap ? j.tr * kBM : a_row0(j), col0 = j.tc * BN;
            uint32_t bad = 0;
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = lane + 32 * i;
                const int li = kSwap ? r / kBlkN : r;
                const bool valid = (kSwap ? row0 + li * kBlkN : row0 + r) < a.rows;
                w4[i] = valid ? sf_word<kNld>(&slot.lane_raw[li][0], kcol, bad) : 0x7F7F7F7Fu;  // 2^0 past the end
            }
            *reinterpret_cast<uint4*>(&slot.sfa[lane * 4]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
#pragma unroll
            for (int h = 0; h < C::kSfbCopies; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = h * 128 + lane + 32 * i;
                    const int ci = kSwap ? c : c / kBlkN;
                    const bool valid = c < BN && (kSwap ? col0 + c : col0 + ci * kBlkN) < a.cols;
                    w4[i] = valid ? sf_word<kNld>(&slot.col_raw[ci < kCR ? ci : 0][0], kcol, bad) : 0x7F7F7F7Fu;
                }
                *reinterpret_cast<uint4*>(&slot.sfb[h * 128 + lane * 4]) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            const bool all_ok = __all_sync(0xFFFFFFFFu, bad == 0u);
            if (lane == 0) {
                slot.pow2 = all_ok ? 1u : 0u;
                slot.kcol = static_cast<uint32_t>(kcol);
                // pair: the leader decides per stage from both halves' flags
                if (kPair && rank != 0u) {
                    slot.xfer[0] = all_ok ? 1u : 0u;
                    slot.xfer[1] = slot.xfer[2] = slot.xfer[3] = 0u;
                }
            }
        };
        // Grouped path: converts stage j from the group buffer g, whose column 0
        // is scale column gx; keeps the stage's raw scales in the slot when the
        // fp32 promotion step may need them.
        // Fused quantisation: the B-side (token) scales come from the slot, where
        // the epilogue warps left them.
        auto convert_g = [&](typename C::Slot& slot, const JobIter& j, const typename C::Group& g, int c0,
                             bool keep_raw) {
            const int row0 = kSwap ? j.tr * kBM : a_row0(j), col0 = j.tc * BN;

            uint32_t bad = 0;
            uint32_t w4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = lane + 32 * i;
                const int li = kSwap ? r / kBlkN : r;
                const bool valid = (kSwap ? row0 + li * kBlkN : row0 + r) < a.rows;
                w4[i] = valid ? sf_word<kNld>(&g.lane[li][c0], 0, bad) : 0x7F7F7F7Fu;  // 2^0 past the end
            }
            *reinterpret_cast<uint4*>(&slot.sfa[lane * 4]) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
#pragma unroll
            for (int h = 0; h < C::kSfbCopies; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = h * 128 + lane + 32 * i;
                    const int ci = kSwap ? c : c / kBlkN;
                    const bool valid = c < BN && (kSwap ? col0 + c : col0 + ci * kBlkN) < a.cols;
                    const int cr = ci < kCR ? ci : 0;
                    if constexpr (kFuse)
                        w4[i] = valid ? sf_word<kNld>(&slot.col_raw[cr][0], 0, bad) : 0x7F7F7F7Fu;
                    else
                        w4[i] = valid ? sf_word<kNld>(&g.col[cr][c0], 0, bad) : 0x7F7F7F7Fu;
                }
                *reinterpret_cast<uint4*>(&slot.sfb[h * 128 + lane * 4]) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            const bool all_ok = __all_sync(0xFFFFFFFFu, bad == 0u);
            if (keep_raw || !all_ok) {
                // chunk q of the stage -> raw column q (one scale per stage: column 0)
                for (int r = lane; r < kLR; r += 32)
#pragma unroll
                    for (int q = 0; q < 4; ++q) slot.lane_raw[r][q] = q < kNld ? g.lane[r][c0 + q] : 0.0f;
                if constexpr (!kFuse)
                    for (int r = lane; r < kCR; r += 32)
#pragma unroll
                        for (int q = 0; q < 4; ++q) slot.col_raw[r][q] = q < kNld ? g.col[r][c0 + q] : 0.0f;
            }
            if (lane == 0) {
                slot.pow2 = all_ok ? 1u : 0u;
                slot.kcol = 0u;
                if (kPair && rank != 0u) {   // the leader decides per stage from both halves' flags
                    slot.xfer[0] = all_ok ? 1u : 0u;
                    slot.xfer[1] = slot.xfer[2] = slot.xfer[3] = 0u;
                }
            }
        };
        if (kScaleTma) {
            // The converter warps (2, and 11 unless it issues MMAs) take
            // alternate stages.  A stage is converted once its slot is free
            // (empty barrier) and its scale group has landed; each warp
            // releases a group once past its end.
            const uint32_t sub = warp == 2 ? 0u : 1u;
            // A pair's promotion path reads the peer's raw scales: keep them always.
            const bool keep_raw = kPair || a.force_promote != 0;
            JobIter it;
            it.begin(a, first_item, item_step);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t nfin = 0;
            uint32_t gcount = 0;
            int gx = 0;
            bool gready = false;
            while (it.valid(a)) {
                const int d = static_cast<int>(gcount % C::kGBufs);
                if ((it.pos % C::kG) == 0) {
                    gx = (it.kb * C::kScalesPerStage) & ~3;
                    gready = false;
                }
                const bool gend = (it.pos % C::kG) == C::kG - 1 || it.last_kb();
                if ((nfin % C::kSfWarps) == sub) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, sync, 3)) break;
                    if (!gready) {
                        if (!wait_bar(gfull_bar(d), (gcount / C::kGBufs) & 1u, sync, 3)) break;
                        gready = true;
                    }
                    // fused: the epilogue warps have quantised the stage
                    if constexpr (kFuse) {
                        if (!wait_bar(qdone_bar(stage), phase, sync, 3)) break;
                    }
                    if (lane == 0) trace_ev(a, 104 + (nfin & 31));
                    convert_g(sf[stage], it, grp[d], it.kb * C::kScalesPerStage - gx, keep_raw);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (kPair && rank != 0u) {
                            // the peer signals the leader's barrier with a 16-byte
                            // async copy of its flag word; the warp's fences above
                            // order the scale words before it
                            const uint32_t x = ptx::smem_u32(&sf[stage].xfer[0]);
                            ptx::bulk_copy_to_cluster_if(1u, ptx::mapa(x, 0u), x, C::kXferBytes,
                                                         at_leader(full_bar(stage)));
                        } else {
                            ptx::mbar_arrive(full_bar(stage));
                        }
                        trace_ev(a, 72 + (nfin & 31));
                    }
                }
                if (gend) {
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(gempty_bar(d));
                    ++gcount;
                }
                ++nfin;
                it.next(a);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        } else if (warp == 2) {
            // Per item, each lane precomputes the scale rows it fetches:
            //   lane side (A operand): activation rows lane+32i (normal), or the
            //     (n-block, chunk) pair `lane` of the tile (swap);
            //   column side (B operand): the (n-block, chunk) pair `lane`
            //     (normal), or (token, chunk) pairs lane+32j (swap).
            constexpr int kLaneLoads = kSwap ? 1 : 4;        // source rows per lane
            constexpr int kLaneChunks = kSwap ? 1 : kNld;    // chunks fetched per source row
            constexpr int kColLoads = kSwap ? (BN * kNld + 31) / 32 : 1;
            ptx::grid_dependency_wait();
            const float* lane_src[kLaneLoads];
            uint32_t lane_dst[kLaneLoads];
            int lane_chunk[kLaneLoads];
            const float* col_src[kColLoads];
            uint32_t col_dst[kColLoads];
            int col_chunk[kColLoads];
            auto setup_item = [&](const JobIter& j) {
                const int row0 = kSwap ? j.tr * kBM : a_row0(j), col0 = j.tc * BN;
                if (!kSwap) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int g = row0 + lane + 32 * i;
                        lane_src[i] = g < a.rows ? a.As + static_cast<int64_t>(g) * a.ks : nullptr;
                        lane_dst[i] = ptx::smem_u32(&sf[0].lane_raw[lane + 32 * i][0]);
                        lane_chunk[i] = 0;
                    }
                    const int gi = lane / kNld, c = lane % kNld;
                    const int g = col0 + gi * kBlkN;
                    col_src[0] = (gi < C::kColGroups && g < a.cols)
                                     ? a.Ws + static_cast<int64_t>(g / kBlkN) * a.ks + c : nullptr;
                    col_dst[0] = ptx::smem_u32(&sf[0].col_raw[gi < kCR ? gi : 0][c]);
                    col_chunk[0] = gi < C::kColGroups ? c : 4;
                } else {
                    const int bi = lane / kNld, c = lane % kNld;
                    const int g = row0 + bi * kBlkN;
                    lane_src[0] = (bi < C::kLaneGroups && g < a.rows)
                                      ? a.Ws + static_cast<int64_t>(g / kBlkN) * a.ks + c : nullptr;
                    lane_dst[0] = ptx::smem_u32(&sf[0].lane_raw[bi < kLR ? bi : 0][c]);
                    lane_chunk[0] = bi < C::kLaneGroups ? c : 4;
#pragma unroll
                    for (int jj = 0; jj < kColLoads; ++jj) {
                        const int idx = lane + 32 * jj;
                        const int t = idx / kNld, cc = idx % kNld;
                        const int g = col0 + t;
                        col_src[jj] = (t < BN && g < a.cols) ? a.As + static_cast<int64_t>(g) * a.ks + cc : nullptr;
                        col_dst[jj] = ptx::smem_u32(&sf[0].col_raw[t < kCR ? t : 0][cc]);
                        col_chunk[jj] = t < BN ? cc : 4;
                    }
                }
            };
            // chunk == 4 marks a lane/slot with nothing to fetch
            auto issue_raw = [&](int si, const JobIter& j) {
                const uint32_t slot_off = static_cast<uint32_t>(si * sizeof(typename C::Slot));
                const int nq = min(4, (a.K - j.kb * kBK) / 32);
                const int soff = j.kb * C::kScalesPerStage;
#pragma unroll
                for (int i = 0; i < kLaneLoads; ++i) {
                    if (lane_chunk[i] >= 4) continue;
#pragma unroll
                    for (int cc = 0; cc < kLaneChunks; ++cc) {
                        const int c = kSwap ? lane_chunk[i] : cc;
                        const uint32_t dst = lane_dst[i] + slot_off + static_cast<uint32_t>(kSwap ? 0 : cc * 4);
                        if (lane_src[i] != nullptr && c < nq)
                            ptx::cp_async_4(dst, lane_src[i] + soff + (kSwap ? 0 : cc));
                        else
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst), "f"(1.0f) : "memory");
                    }
                }
#pragma unroll
                for (int i = 0; i < kColLoads; ++i) {
                    if (col_chunk[i] >= 4) continue;
                    if (col_src[i] != nullptr && col_chunk[i] < nq)
                        ptx::cp_async_4(col_dst[i] + slot_off, col_src[i] + soff);
                    else
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(col_dst[i] + slot_off), "f"(1.0f) : "memory");
                }
            };
            JobIter iss, fin;
            iss.begin(a, first_item, item_step);
            fin.begin(a, first_item, item_step);
            if (iss.valid(a)) setup_item(iss);
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
                    issue_raw(si, iss);
                    ptx::cp_async_commit();
                    ++n_iss;
                    if (iss.next(a) && iss.valid(a)) setup_item(iss);
                }
                if (failed) break;
                const int sf_i = static_cast<int>(n_fin % kStages);
                ptx::cp_async_wait_pending(static_cast<int>(n_iss - n_fin) - 1);
                __syncwarp();
                convert(sf[sf_i], fin, 0);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(full_bar(sf_i));
                    trace_ev(a, 72 + (n_fin & 31));
                }
                ++n_fin;
                fin.next(a);
            }
            ptx::cp_async_wait_pending(0);
        }
        __syncwarp();
    } else if (kAlt && (warp == 1 || warp == C::kMma2Warp)) {
        // ------------------------------------------------- alternating MMA issuers
        // One MMA instruction keeps its issuing warp busy about as long as the
        // tensor core takes to execute it, so whatever else a single issuer does
        // per K stage (operand wait, scale-factor copies, commit) leaves the
        // tensor core idle.  Here two warps share the one accumulator and take
        // turns: warp 1 issues K stages 0, 2, 4, ... of the CTA's job stream,
        // warp 12 stages 1, 3, 5, ...  Before its turn a warp waits for its
        // stage's operands and copies the stage's scale factors into TMEM slots
        // of its own, overlapping the other warp's MMAs.  The turn passes with a
        // token: tcgen05.fence::before_thread_sync and an mbarrier arrive by the
        // holder, a bounded wait and tcgen05.fence::after_thread_sync by the
        // next, which orders the next warp's MMAs after the holder's.  The token
        // carries the accumulator state (segments issued; segment open;
        // accumulate flag) in shared memory.  The MMA sequence is the one a
        // single issuer would produce.
        const uint32_t mw = warp == 1 ? 0u : 1u;
        constexpr uint32_t idesc_f8 = ptx::idesc_f8(kBM, BN);
        constexpr uint32_t idesc_mx = ptx::idesc_mxf8(kBM, BN);
        const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
        const uint32_t leader = lane == 0 ? 1u : 0u;
        volatile uint32_t* state = misc + 4;   // [0] segments issued, [1] bit 0 open, bit 1 accumulate
        JobIter it;
        it.begin(a, first_item, item_step);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t n = 0;        // position in the job stream (both warps count every stage)
        uint32_t turns = 0;    // turns taken by this warp
        uint32_t mx_used = 0;  // this warp's block-scaled stages (its scale-slot parity)
        bool failed = false;
        auto acc_buf = [&](uint32_t u) { return static_cast<int>(u % kAccBufs); };
        auto acc_par = [&](uint32_t u) { return (u / kAccBufs) & 1u; };
        const uint32_t sf_col0 = C::kSfCol - 32u * mw;
        auto hand_over = [&](int b) {
            ptx::mbar_arrive_if(leader, accf_bar(0, b));
            ptx::tc_commit_g_if<1>(leader, accf_bar(0, b));
        };
        // Publishes the state and passes the turn to the other warp.
        auto pass_turn = [&](uint32_t seg, uint32_t flags) {
            if (lane == 0) {
                state[0] = seg;
                state[1] = flags;
            }
            __syncwarp();
            ptx::tc_fence_before();
            ptx::mbar_arrive_if(leader, hand_bar(mw ^ 1u));
        };
        const uint64_t ad_base = ptx::smem_desc(sA0, 16, 1024, ptx::kLayoutSw128);
        const uint64_t bd_base = ptx::smem_desc(sB0, 16, 1024, ptx::kLayoutSw128);
        const uint64_t sfa_base = ptx::smem_desc(ptx::smem_u32(sf[0].sfa), 128, 128, ptx::kLayoutNone);
        const uint64_t sfb_base = ptx::smem_desc(ptx::smem_u32(sf[0].sfb), 128, 128, ptx::kLayoutNone);
        constexpr uint32_t kSlotStep = sizeof(typename C::Slot) >> 4;
        const bool ragged_k = (a.K % kBK) != 0;
        while (it.valid(a) && !failed) {
            if ((n & 1u) != mw) {   // the other warp's stage
                it.next(a);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
                ++n;
                continue;
            }
            const bool item_last = it.last_kb();
            if (!wait_bar(full_bar(stage), phase, sync, 2)) { failed = true; break; }
            ptx::tc_fence_after();
            if (lane == 0) trace_ev(a, 40 + (n & 31));
            typename C::Slot& slot = sf[stage];
            const int nq = ragged_k ? min(4, (a.K - it.kb * kBK) / 32) : 4;
            const uint64_t ad0 = ad_base + static_cast<uint64_t>(stage * (C::kABytes >> 4));
            const uint64_t bd0 = bd_base + static_cast<uint64_t>(stage * (C::kBBytes >> 4));
            const bool mx = slot.pow2 != 0u && !a.force_promote;
            const uint32_t t_sfa = tmem + sf_col0 + 16u * (mx_used & 1u), t_sfb = t_sfa + 4u;
            if (mx) {
                const uint64_t slot_off = static_cast<uint64_t>(stage) * kSlotStep;
                ptx::tmem_cp_g_if<1>(leader, t_sfa, sfa_base + slot_off);
#pragma unroll
                for (int h = 0; h < C::kSfbCopies; ++h)
                    ptx::tmem_cp_g_if<1>(leader, t_sfb + 4u * h, sfb_base + slot_off + 32u * h);
                ++mx_used;
            }
            // take the turn (the first stage of the job stream needs none)
            if (n != 0) {
                const uint32_t r = turns - (mw == 0 ? 1u : 0u);   // tokens received before this one
                if (!wait_bar_warp(hand_bar(mw), r & 1u, sync, 6, false)) { failed = true; break; }
                ptx::tc_fence_after();
            }
            if (lane == 0) trace_ev(a, 216 + (n & 15));
            ++turns;
            uint32_t seg = state[0];
            const uint32_t st_flags = state[1];
            bool seg_open = (st_flags & 1u) != 0u;
            uint32_t acc_flag = (st_flags >> 1) & 1u;
            if (mx) {
                if (!seg_open) {
                    if (!wait_bar(acce_bar(0, acc_buf(seg)), acc_par(seg) ^ 1u, sync, 2)) { failed = true; break; }
                    ptx::tc_fence_after();
                    acc_flag = 0;
                }
                const int b = acc_buf(seg);
                const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                if (nq == 4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        ptx::mma_mxf8_g_if<1>(leader, d, ad0 + 2u * j, bd0 + 2u * j,
                                              ptx::idesc_sf_ids(idesc_mx, j, j), t_sfa, t_sfb,
                                              j == 0 ? acc_flag : 1u);
                } else {
                    for (int j = 0; j < nq; ++j)
                        ptx::mma_mxf8_g_if<1>(leader, d, ad0 + 2u * j, bd0 + 2u * j,
                                              ptx::idesc_sf_ids(idesc_mx, j, j), t_sfa, t_sfb,
                                              j == 0 ? acc_flag : 1u);
                }
                // The item's last stage closes the segment.  The state handed on
                // already shows it closed; the epilogue is signalled right after.
                pass_turn(item_last ? seg + 1u : seg, item_last ? 0u : 3u);
                if (lane == 0) trace_ev(a, 200 + (n & 15));
                ptx::tc_commit_g_if<1>(leader, empty_bar(stage));
                if (item_last) {
                    if (lane == 0) info[b].flags = kInfoLast;
                    __syncwarp();
                    hand_over(b);
                }
            } else {
                if (seg_open) {   // hand the open block-scaled segment to the epilogue
                    const int b = acc_buf(seg);
                    if (lane == 0) info[b].flags = 0u;
                    __syncwarp();
                    hand_over(b);
                    ++seg;
                }
                constexpr bool kBlk128 = kBlkK == 128;
                const int ngroups = kBlk128 ? 1 : nq;
                const int steps = kBlk128 ? nq : 1;
                for (int gidx = 0; gidx < ngroups; ++gidx) {
                    const int b = acc_buf(seg);
                    if (!wait_bar(acce_bar(0, b), acc_par(seg) ^ 1u, sync, 2)) { failed = true; break; }
                    ptx::tc_fence_after();
                    const int q = C::kNld == 1 ? static_cast<int>(slot.kcol) : gidx;
                    const bool last = item_last && gidx == ngroups - 1;
                    for (int r = lane; r < 128; r += 32) info[b].lane_s[r] = slot.lane_raw[r][q];
                    for (int c = lane; c < BN; c += 32) info[b].col_s[c] = slot.col_raw[c / kBlkN][q];
                    if (lane == 0) info[b].flags = kInfoPromote | (last ? kInfoLast : 0u);
                    __syncwarp();
                    const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
                    for (int t = 0; t < steps; ++t) {
                        const int jj = gidx * steps + t;
                        ptx::mma_f8_g_if<1>(leader, d, ad0 + 2u * jj, bd0 + 2u * jj, idesc_f8, t > 0 ? 1u : 0u);
                    }
                    hand_over(b);
                    ++seg;
                }
                if (failed) break;
                pass_turn(seg, 0u);
                if (lane == 0) trace_ev(a, 200 + (n & 15));
                ptx::tc_commit_g_if<1>(leader, empty_bar(stage));
            }
            it.next(a);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            ++n;
        }
        // Let every tcgen05 op issued above land before teardown.
        ptx::tc_commit_local_g_if<1>(leader, drain_bar(static_cast<int>(mw)));
        if (lane == 0) wait_bar(drain_bar(static_cast<int>(mw)), 0, sync, 5);
        __syncwarp();
    } else if (kChan && (warp == 2 || warp == C::kSf2Warp)) {
        // per-channel scaling: no per-stage scales, so no scale warps
    } else if (warp == 1 || (kMW > 1 && warp == C::kMma2Warp)) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs this loop in lock-step; every tcgen05 instruction
        // is issued by lane 0 through a predicate inside the asm, so the warp
        // never diverges and descriptors stay warp-uniform.  With two issuers,
        // issuer mw takes the K stages at positions pos % 2 == mw of each item
        // and owns accumulators, scale slots and barriers of its own.
        // With a CTA pair only the leader's warp issues (for both CTAs).
        const int mw = warp == 1 ? 0 : 1;
        constexpr uint32_t idesc_f8 = ptx::idesc_f8(C::kTileRows, BN);
        constexpr uint32_t idesc_mx = ptx::idesc_mxf8(C::kTileRows, BN);
        const uint32_t sA0 = ptx::smem_u32(sA), sB0 = ptx::smem_u32(sB);
        const uint32_t leader = lane == 0 ? 1u : 0u;
        constexpr int kColGroup = kSwap ? 1 : kBlkN;
        JobIter it;
        it.begin(a, first_item, item_step);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t seg = 0;      // accumulator segments issued so far
        uint32_t mx_used = 0;  // block-scaled stages issued so far (scale-slot parity)
        uint32_t mma_jobs = 0;
        bool failed = false;
        bool seg_open = false;
        uint32_t acc_flag = 0;  // 0 for the first MMA of an open segment
        auto acc_buf = [&](uint32_t u) { return static_cast<int>(u % kAccBufs); };
        auto acc_par = [&](uint32_t u) { return (u / kAccBufs) & 1u; };
        Info<BN>* my_info = info + mw * kAccBufs;
        const uint32_t acc_col0 = static_cast<uint32_t>(mw * kAccBufs * BN);
        const uint32_t sf_col0 = C::kSfCol - 32u * static_cast<uint32_t>(mw);
        // Signals segment b to the epilogue(s): the MMA thread's arrive (after
        // the Info writes; pair: also on the peer's barrier, release at cluster
        // scope) and a commit that fires when the MMAs are done (both CTAs).
        auto hand_over = [&](int b) {
            ptx::mbar_arrive_if(leader, accf_bar(mw, b));
            if (kPair) ptx::mbar_arrive_cluster_if(leader, ptx::mapa(accf_bar(mw, b), 1u));
            ptx::tc_commit_g_if<kCG>(leader, accf_bar(mw, b));
        };
        // Hands the open accumulator segment to the epilogue.
        auto close_segment = [&](uint32_t flags) {
            const int b = acc_buf(seg);
            if (lane == 0) {
                my_info[b].flags = flags;
                if (kPair) ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&my_info[b].flags), 1u), flags);
            }
            __syncwarp();
            hand_over(b);
            ++seg;
        };
        // Descriptors are linear in the start address: a stage's descriptor is
        // the stage-0 descriptor plus (stage offset >> 4).
        const uint64_t ad_base = ptx::smem_desc(sA0, 16, 1024, ptx::kLayoutSw128);
        const uint64_t bd_base = ptx::smem_desc(sB0, 16, 1024, ptx::kLayoutSw128);
        const uint64_t sfa_base = ptx::smem_desc(ptx::smem_u32(sf[0].sfa), 128, 128, ptx::kLayoutNone);
        const uint64_t sfb_base = ptx::smem_desc(ptx::smem_u32(sf[0].sfb), 128, 128, ptx::kLayoutNone);
        constexpr uint32_t kSlotStep = sizeof(typename C::Slot) >> 4;
        // A K stage shorter than 128 exists only when K % 128 != 0 (last stage).
        const bool ragged_k = (a.K % kBK) != 0;
        while ((!kPair || rank == 0u) && it.valid(a) && !failed) {
            if (kMW > 1 && (it.pos % kMW) != mw) {   // the other issuer's stage
                it.next(a);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
                continue;
            }
            // this issuer's last stage of the item
            const bool my_last = it.pos + kMW >= it.nkb;
            if (!wait_bar<kPair>(full_bar(stage), phase, sync, 2)) { failed = true; break; }
            ptx::tc_fence_after();
            if (lane == 0) trace_ev(a, 40 + (mma_jobs & 31));
            ++mma_jobs;
            typename C::Slot& slot = sf[stage];
            const int nq = ragged_k ? min(4, (a.K - it.kb * kBK) / 32) : 4;
            const uint64_t ad0 = ad_base + static_cast<uint64_t>(stage * (C::kABytes >> 4));
            const uint64_t bd0 = bd_base + static_cast<uint64_t>(stage * (C::kBBytes >> 4));
            // pair: block-scaled only when the scales of both CTAs' stages are 2^e;
            // per-channel scaling accumulates unscaled MMAs over the whole K range
            const bool mx = kChan || (slot.pow2 != 0u && !a.force_promote && (!kPair || slot.xfer[0] != 0u));
            if (mx) {
                if (!seg_open) {
                    if (!wait_bar<kPair>(acce_bar(mw, acc_buf(seg)), acc_par(seg) ^ 1u, sync, 2)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    seg_open = true;
                    acc_flag = 0;
                }
                const uint32_t sfs = sf_col0 + 16u * (mx_used & 1u);
                const uint32_t t_sfa = tmem + sfs, t_sfb = tmem + sfs + 4u;
                const uint32_t d = tmem + acc_col0 + static_cast<uint32_t>(acc_buf(seg) * BN);
                if constexpr (kChan) {
                    for (int j = 0; j < nq; ++j)
                        ptx::mma_f8_g_if<kCG>(leader, d, ad0 + 2u * j, bd0 + 2u * j, idesc_f8, j == 0 ? acc_flag : 1u);
                } else {
                const uint64_t slot_off = static_cast<uint64_t>(stage) * kSlotStep;
                ptx::tmem_cp_g_if<kCG>(leader, t_sfa, sfa_base + slot_off);
#pragma unroll
                for (int h = 0; h < C::kSfbCopies; ++h)
                    ptx::tmem_cp_g_if<kCG>(leader, t_sfb + 4u * h, sfb_base + slot_off + 32u * h);
                if (nq == 4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        // +32 bytes along K inside the swizzle atom = +2 in the start field
                        ptx::mma_mxf8_g_if<kCG>(leader, d, ad0 + 2u * j, bd0 + 2u * j,
                                                ptx::idesc_sf_ids(idesc_mx, j, j), t_sfa, t_sfb,
                                                j == 0 ? acc_flag : 1u);
                    }
                } else {
                    for (int j = 0; j < nq; ++j)
                        ptx::mma_mxf8_g_if<kCG>(leader, d, ad0 + 2u * j, bd0 + 2u * j,
                                                ptx::idesc_sf_ids(idesc_mx, j, j), t_sfa, t_sfb,
                                                j == 0 ? acc_flag : 1u);
                }
                }
                acc_flag = 1;
                ++mx_used;
            } else {
                if (seg_open) {
                    close_segment(0u);
                    seg_open = false;
                }
                constexpr bool kBlk128 = kBlkK == 128;
                const int ngroups = kBlk128 ? 1 : nq;
                const int steps = kBlk128 ? nq : 1;
                for (int gidx = 0; gidx < ngroups; ++gidx) {
                    const int b = acc_buf(seg);
                    if (!wait_bar<kPair>(acce_bar(mw, b), acc_par(seg) ^ 1u, sync, 2)) { failed = true; break; }
                    ptx::tc_fence_after();
                    const int j = gidx;  // scale chunk (blk_k == 128: chunk 0 holds the block scale)
                    const int q = C::kNld == 1 ? static_cast<int>(slot.kcol) : j;
                    const bool last = my_last && gidx == ngroups - 1;
                    const uint32_t flags = kInfoPromote | (last ? kInfoLast : 0u);
                    for (int r = lane; r < 128; r += 32)
                        my_info[b].lane_s[r] = slot.lane_raw[kSwap ? r / kBlkN : r][q];
                    for (int c = lane; c < BN; c += 32) my_info[b].col_s[c] = slot.col_raw[c / kColGroup][q];
                    if (lane == 0) my_info[b].flags = flags;
                    if (kPair) {
                        // the peer's Info: its own row scales, the same column scales
                        for (int r = lane; r < 128; r += 32)
                            ptx::st_cluster_f32(ptx::mapa(ptx::smem_u32(&my_info[b].lane_s[r]), 1u),
                                                ptx::ld_cluster_f32(ptx::mapa(ptx::smem_u32(&slot.lane_raw[r][q]), 1u)));
                        for (int c = lane; c < BN; c += 32)
                            ptx::st_cluster_f32(ptx::mapa(ptx::smem_u32(&my_info[b].col_s[c]), 1u),
                                                slot.col_raw[c / kColGroup][q]);
                        if (lane == 0) ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(&my_info[b].flags), 1u), flags);
                        asm volatile("fence.acq_rel.cluster;" ::: "memory");
                    }
                    __syncwarp();
                    const uint32_t d = tmem + acc_col0 + static_cast<uint32_t>(b * BN);
                    for (int t = 0; t < steps; ++t) {
                        const int jj = gidx * steps + t;   // 32-wide chunk inside the stage
                        ptx::mma_f8_g_if<kCG>(leader, d, ad0 + 2u * jj, bd0 + 2u * jj, idesc_f8, t > 0 ? 1u : 0u);
                    }
                    hand_over(b);
                    ++seg;
                }
                if (failed) break;
            }
            ptx::tc_commit_g_if<kCG>(leader, empty_bar(stage));  // frees the stage (both CTAs) when its MMAs finish
            if (lane == 0) trace_ev(a, 200 + ((mma_jobs - 1) & 15));
            it.next(a);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            if (my_last && seg_open) {
                close_segment(kInfoLast);
                seg_open = false;
            }
        }
        // Let every tcgen05 op issued above land before teardown.
        if (!kPair || rank == 0u) {
            ptx::tc_commit_local_g_if<kCG>(leader, drain_bar(mw));
            if (lane == 0) wait_bar(drain_bar(mw), 0, sync, 5);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        constexpr int kCols = C::kCols;
        constexpr int kLd = C::kLd;
        const int ew = warp - kEpiWarp0;          // 0 .. kEpiWarps-1
        const int quad = warp & 3;                // TMEM lane quadrant this warp may access
        const int half = ew >> 2;                 // which half of the columns (8 warps)
        const int r_in_tile = quad * 32 + lane;   // accumulator row (TMEM lane)
        const int c_begin = half * kCols;
        const int epi_tid = ew * 32 + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        JobIter it;
        it.begin(a, first_item, item_step);
        uint32_t seg0 = 0, seg1 = 0;   // segments consumed per MMA issuer
        uint32_t n_items = 0;
        float acc[kCols];
        float acc1[kCols];             // second issuer's sum (two-issuer configurations)
        uint32_t qn = 0;               // fused quantisation: stages quantised so far
        bool dep_done = false;         // ... and the wait for the preceding grid
        // Adds one accumulator segment of issuer m into `dst` (first: overwrite).
        auto consume = [&](int m, uint32_t sg, bool first, float (&dst)[kCols]) {
            const int b = static_cast<int>(sg % kAccBufs);
            const Info<BN>& inf = info[m * kAccBufs + b];
            const uint32_t flags = inf.flags;
            const bool promote = (flags & kInfoPromote) != 0u;
            const float ls = promote ? inf.lane_s[r_in_tile] : 1.0f;
            const uint32_t col = static_cast<uint32_t>((m * kAccBufs + b) * BN + c_begin);
#pragma unroll
            for (int c0 = 0; c0 < kCols; c0 += kLd) {
                uint32_t r[kLd];
                ptx::tmem_ld<kLd>(t_lane + col + static_cast<uint32_t>(c0), r);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < kLd; ++i) {
                    const float v = __uint_as_float(r[i]);
                    if (promote) {
                        const float sc = ls * inf.col_s[c_begin + c0 + i];
                        dst[c0 + i] = first ? v * sc : fmaf(v, sc, dst[c0 + i]);
                    } else {
                        dst[c0 + i] = first ? v : dst[c0 + i] + v;
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            // the accumulator may be overwritten: tell the issuing CTA
            if (kPair && rank != 0u)
                ptx::mbar_arrive_cluster_if(lane == 0 ? 1u : 0u, at_leader(acce_bar(m, b)));
            else if (lane == 0)
                ptx::mbar_arrive(acce_bar(m, b));
            return (flags & kInfoLast) != 0u;
        };
        while (it.valid(a)) {
            bool failed = false;
            // read now, used after the accumulators: the load's latency hides
            // behind the waits instead of following them
            const bool aborted_before = *sync.abort_flag != 0u;
            if constexpr (kFuse) {
                // Quantise this item's activation tiles before waiting for its
                // accumulators: the loads of up to kBatch stages are issued
                // first, then each stage is written once its ring slot is free.
                constexpr int kBatch = 8 / kVpt;
                if (!dep_done) {
                    ptx::grid_dependency_wait();   // x may be the preceding kernel's output
                    dep_done = true;
                    if (epi_tid == 0) trace_ev(a, 4);
                }
                JobIter q = it;
                for (int p0 = 0; p0 < it.nkb && !failed; p0 += kBatch) {
                    uint4 xv[kBatch][kVpt];
                    JobIter ql = q;
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        const bool live = p0 + b < it.nkb;
#pragma unroll
                        for (int i = 0; i < kVpt; ++i)
                            xv[b][i] = live ? x_vec(ql, epi_tid + i * C::kEpiWarps * 32) : make_uint4(0, 0, 0, 0);
                        if (live && p0 + b + 1 < it.nkb) ql.next(a);
                    }
                    // each stage is released as soon as it is written: the MMAs
                    // start on the first one (measured faster than one release
                    // per batch)
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        if (p0 + b < it.nkb && !failed) {
                            const uint32_t n = qn + static_cast<uint32_t>(p0 + b);
                            const int s = static_cast<int>(n % kStages);
                            if (!wait_bar_warp(empty_bar(s), ((n / kStages) & 1u) ^ 1u, sync, 4, false)) {
                                failed = true;
                            } else {
#pragma unroll
                                for (int i = 0; i < kVpt; ++i)
                                    quantize_vec(xv[b][i], epi_tid + i * C::kEpiWarps * 32, s, q, sf[s]);
                                ptx::fence_proxy_async_smem();   // codes: read by the MMA (async proxy)
                                __syncwarp();
                                if (lane == 0) ptx::mbar_arrive(qdone_bar(s));
                                if (p0 + b + 1 < it.nkb) q.next(a);
                            }
                        }
                    }
                }
                qn += static_cast<uint32_t>(it.nkb);
            }
            if (C::kAccSets == 1) {
                bool first = true;
                while (true) {
                    const int b = static_cast<int>(seg0 % kAccBufs);
                    if (!wait_bar_warp<kPair>(accf_bar(0, b), (seg0 / kAccBufs) & 1u, sync, 4, true)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    const bool last = consume(0, seg0, first, acc);
                    ++seg0;
                    first = false;
                    if (last) break;
                }
            } else {
                // Issuer 1 has stages in the item only when it has two or more.
                bool done0 = false, done1 = it.nkb < 2;
                bool first0 = true, first1 = true;
                while (!(done0 && done1)) {
                    // lane 0 polls both issuers' next segment; take whichever is ready
                    int pick = -1;
                    if (lane == 0) {
                        const uint64_t t0 = ptx::globaltimer();
                        uint32_t spins = 0;
                        while (true) {
                            if (!done0 && ptx::mbar_test_wait(accf_bar(0, static_cast<int>(seg0 % kAccBufs)),
                                                              (seg0 / kAccBufs) & 1u)) { pick = 0; break; }
                            if (!done1 && ptx::mbar_test_wait(accf_bar(1, static_cast<int>(seg1 % kAccBufs)),
                                                              (seg1 / kAccBufs) & 1u)) { pick = 1; break; }
                            if ((++spins & 15u) == 0) {
                                const uint64_t dt = ptx::globaltimer() - t0;
                                if (dt > kAbortPollNs && *sync.abort_flag) break;
                                if (dt > sync.limit) {
                                    *sync.abort_flag = 1u;
                                    atomicOr(sync.status, kStatusTimeout | (4u << 8));
                                    break;
                                }
                            }
                            if (spins > 8) __nanosleep(64);
                        }
                    }
                    pick = __shfl_sync(0xFFFFFFFFu, pick, 0);
                    __syncwarp();
                    if (pick < 0) { failed = true; break; }
                    if (epi_tid == 0) trace_ev(a, 139 + 4 * (n_items & 15));   // (the last pick stays)
                    ptx::tc_fence_after();
                    if (pick == 0) {
                        done0 = consume(0, seg0, first0, acc);
                        ++seg0;
                        first0 = false;
                    } else {
                        done1 = consume(1, seg1, first1, acc1);
                        ++seg1;
                        first1 = false;
                    }
                }
                // fixed order: issuer 0's sum + issuer 1's sum
                if (!failed && it.nkb >= 2) {
#pragma unroll
                    for (int c = 0; c < kCols; ++c) acc[c] += acc1[c];
                }
            }
            if (epi_any<C::kEpiWarps * 32>(failed || aborted_before)) break;
            if (epi_tid == 0) trace_ev(a, 136 + 4 * (n_items & 15));
            // ------------------------------------------------ output
            const int row0 = kSwap ? it.tr * kBM : a_row0(it), col0 = it.tc * BN;
            const int grow = row0 + r_in_tile;   // global row of the MMA A operand
            bool store = true;
            if (kCK && a.splits > 1) {
                // The two K splits of the tile are the two CTAs of this cluster
                // (item = tile * 2 + split, cluster = items 2c and 2c + 1).  Split
                // 1 stages its fp32 partial in its own shared memory and sends
                // it to split 0's in one bulk copy, which completes split 0's
                // barrier; split 0 adds p_0 + p_1 (split order, as the global
                // path) and stores.  Split 0 frees the buffer with a remote
                // arrive before split 1 may send the next item's partial.
                if (ck_wait_pending) {
                    ptx::cluster_wait();
                    ck_wait_pending = false;
                }
                float* ckbuf = reinterpret_cast<float*>(smem + C::kOffCK);
                const uint32_t ckbuf_s = ptx::smem_u32(ckbuf);
                const uint32_t ck_rank = ptx::cluster_rank();
                bool ck_ok = true;
                if (ck_rank == 1u) {
                    if (n_items > 0)
                        ck_ok = wait_bar_warp<true>(ckfree_bar(), (n_items - 1) & 1u, sync, 7, true);
                    if (ck_ok) {
#pragma unroll
                        for (int c = 0; c < kCols; c += 4)
                            *reinterpret_cast<float4*>(ckbuf + epi_tid * kCols + c) =
                                make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                        ptx::fence_proxy_async_smem();   // read by the bulk copy (async proxy)
                    }
                    if (epi_any<C::kEpiWarps * 32>(!ck_ok)) break;
                    if (epi_tid == 0)
                        ptx::bulk_copy_to_cluster_if(1u, ptx::mapa(ckbuf_s, 0u), ckbuf_s, C::kCKBytes,
                                                     ptx::mapa(ckfull_bar(), 0u));
                    if (epi_tid == 0) trace_ev(a, 137 + 4 * (n_items & 15));
                    store = false;
                } else {
                    if (epi_tid == 0) ptx::mbar_arrive_expect_tx(ckfull_bar(), C::kCKBytes);
                    ck_ok = wait_bar_warp<true>(ckfull_bar(), n_items & 1u, sync, 7, true);
                    if (epi_tid == 0) trace_ev(a, 137 + 4 * (n_items & 15));
                    if (ck_ok) {
#pragma unroll
                        for (int c = 0; c < kCols; c += 4) {
                            const float4 v = *reinterpret_cast<const float4*>(ckbuf + epi_tid * kCols + c);
                            acc[c] += v.x;
                            acc[c + 1] += v.y;
                            acc[c + 2] += v.z;
                            acc[c + 3] += v.w;
                        }
                    }
                    if (epi_any<C::kEpiWarps * 32>(!ck_ok)) break;   // (also: every thread has read)
                    // the peer waits for the buffer only before a next item
                    if (epi_tid == 0 && it.item + it.step < a.items)
                        ptx::mbar_arrive_cluster_if(1u, ptx::mapa(ckfree_bar(), 1u));
                }
            } else if (a.splits > 1) {
                // fp32 partial of this split; the last split to arrive sums all
                // partials in split order (deterministic) and stores the tile.
                // Rows past the operand's end carry nothing: neither written nor read.
                const bool live = grow < a.rows;
                const int64_t tile_base = static_cast<int64_t>(it.tile) * a.splits * (kBM * BN);
                if (kSwap) {
                    // column-major tile: one column of a warp's 32 rows is one 128-byte line
                    float* part = a.partial + tile_base + (static_cast<int64_t>(it.split) * BN + c_begin) * kBM +
                                  r_in_tile;
                    if (live) {
#pragma unroll
                        for (int c = 0; c < kCols; ++c) part[c * kBM] = acc[c];
                    }
                } else {
                    float* part = a.partial + tile_base + static_cast<int64_t>(it.split) * (kBM * BN) +
                                  r_in_tile * BN + c_begin;
                    if (live) {
#pragma unroll
                        for (int c = 0; c < kCols; c += 4)
                            *reinterpret_cast<float4*>(part + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                    }
                }
                epi_sync<C::kEpiWarps * 32>();
                if (epi_tid == 0) {
                    trace_ev(a, 137 + 4 * (n_items & 15));
                    // The barrier orders every epilogue thread's partial before this
                    // arrival, whose release publishes them; the last arriver's
                    // acquire makes the other splits' partials visible.
                    const uint32_t old = ptx::atom_add_acq_rel_gpu(a.counters + it.tile, 1u);
                    const bool last_split = old == static_cast<uint32_t>(a.splits - 1);
                    misc[2] = last_split ? 1u : 0u;
                }
                epi_sync<C::kEpiWarps * 32>();
                store = misc[2] != 0u;
                if (store && live) {
                    if (kSwap) {
                        // p_0 + p_1 + ... in split order; this split's own term from
                        // registers.  The loads of kSB splits go out before their
                        // adds: one L2 round trip per kSB splits, not per split.
                        constexpr int kSB = kCols <= 8 ? 4 : (kCols <= 16 ? 2 : 1);
                        const float* base = a.partial + tile_base + static_cast<int64_t>(c_begin) * kBM + r_in_tile;
                        float (&sum)[kCols] = acc1;   // free once the issuers' sums are combined
                        for (int sp0 = 0; sp0 < a.splits; sp0 += kSB) {
                            float v[kSB][kCols];
#pragma unroll
                            for (int j = 0; j < kSB; ++j) {
                                const int sp = sp0 + j;
                                const bool load = sp < a.splits && sp != it.split;
                                const float* p = base + static_cast<int64_t>(sp) * (BN * kBM);
#pragma unroll
                                for (int c = 0; c < kCols; ++c) v[j][c] = load ? __ldcg(p + c * kBM) : 0.0f;
                            }
#pragma unroll
                            for (int j = 0; j < kSB; ++j) {
                                const int sp = sp0 + j;
                                if (sp < a.splits) {
#pragma unroll
                                    for (int c = 0; c < kCols; ++c) {
                                        const float x = sp == it.split ? acc[c] : v[j][c];
                                        sum[c] = sp == 0 ? x : sum[c] + x;
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int c = 0; c < kCols; ++c) acc[c] = sum[c];
                    } else {
                        const float* base = a.partial + tile_base + r_in_tile * BN + c_begin;
                        // p_0 + p_1 + ... in split order, all read back from L2
#pragma unroll
                        for (int c = 0; c < kCols; c += 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4*>(base + c));
                            acc[c] = v.x;
                            acc[c + 1] = v.y;
                            acc[c + 2] = v.z;
                            acc[c + 3] = v.w;
                        }
                        for (int sp = 1; sp < a.splits; ++sp) {
                            const float* p = base + static_cast<int64_t>(sp) * (kBM * BN);
#pragma unroll
                            for (int c = 0; c < kCols; c += 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4*>(p + c));
                                acc[c] += v.x;
                                acc[c + 1] += v.y;
                                acc[c + 2] += v.z;
                                acc[c + 3] += v.w;
                            }
                        }
                    }
                }
                if (store && epi_tid == 0) a.counters[it.tile] = 0u;   // ready for the next launch
            }
            if constexpr (kChan) {
                // D = acc * sa * sb + bias: the MMA rows are tokens (weights when swapped)
                if (store && grow < a.rows) {
                    const float row_s = kSwap ? fz.sb[fz.sb_n == 1 ? 0 : grow] : fz.sa[fz.sa_n == 1 ? 0 : grow];
                    const float row_b = (kSwap && fz.bias) ? __uint_as_float(uint32_t(fz.bias[grow]) << 16) : 0.0f;
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        const int gc = col0 + c_begin + c;   // token (swapped) or output column
                        if (gc < a.cols) {
                            const float col_s = kSwap ? fz.sa[fz.sa_n == 1 ? 0 : gc] : fz.sb[fz.sb_n == 1 ? 0 : gc];
                            const float col_b = (!kSwap && fz.bias) ? __uint_as_float(uint32_t(fz.bias[gc]) << 16) : 0.0f;
                            acc[c] = fmaf(acc[c] * row_s, col_s, row_b + col_b);
                        }
                    }
                }
            }
            if constexpr (!kSwap) {
                // A thread owns one row: 32-byte stores (a full sector per row
                // and half the store instructions) when D's rows allow them,
                // else two 16-byte ones.  The 16-byte stores alone measured 16%
                // of a short-K GEMM's time (8192 x 24576 x 1536: 410 us, 344 us
                // without any D store, 336 us with 32-byte stores).
                // (not with per-channel scaling: its epilogue then spills)
                static_assert(kCols % 16 == 0, "16-column store chunks");
                const bool v8 = !kChan &&
                                ((reinterpret_cast<uintptr_t>(a.D) | (static_cast<uintptr_t>(a.N) * 2u)) & 31u) == 0;
                if (store && grow < a.M) {
                    __nv_bfloat16* drow = a.D + static_cast<int64_t>(grow) * a.N;
#pragma unroll
                    for (int c = 0; c < kCols; c += 16) {
                        const int gcol = col0 + c_begin + c;
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(acc[c + 2 * i], acc[c + 2 * i + 1]);
                        if (v8) {
                            if (gcol < a.N) ptx::st_global_v8(drow + gcol, w);
                        } else {
                            if (gcol < a.N)
                                *reinterpret_cast<uint4*>(drow + gcol) = make_uint4(w[0], w[1], w[2], w[3]);
                            if (gcol + 8 < a.N)
                                *reinterpret_cast<uint4*>(drow + gcol + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            } else {
                if (store && grow < a.N) {
#pragma unroll
                    for (int c = 0; c < kCols; ++c) {
                        const int m = col0 + c_begin + c;
                        if (m < a.M) a.D[static_cast<int64_t>(m) * a.N + grow] = __float2bfloat16_rn(acc[c]);
                    }
                }
            }
            if (epi_tid == 0) trace_ev(a, 138 + 4 * (n_items & 15));
            ++n_items;
            // advance to the next item (skip the remaining k-stages of this one)
            while (it.valid(a) && !it.next(a)) {
            }
        }
    }

    if (lane == 0 && warp < 12) trace_ev(a, 232 + warp);
    ptx::tc_fence_before();
    __syncthreads();
    if (lane == 0 && warp < 11) trace_ev(a, 244 + warp);   // slot 255 is the end stamp
    if (threadIdx.x == 0) trace_ev(a, 255);
    // A pair's leader writes the peer's TMEM and reads its shared memory until
    // its drain completes: neither CTA leaves before both are here.
    // no CTA of a cluster leaves while the other may still address its shared memory
    if (kPair) ptx::cluster_sync();
    if (kCK) {
        // No remote arrive is in flight (the last item sends none) and split
        // 0 has seen split 1's last bulk copy land, so execution order is all
        // that is left to enforce.
        if (ck_wait_pending) ptx::cluster_wait();
        ptx::cluster_arrive_relaxed();
        ptx::cluster_wait();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_g<kCG>(tmem, C::kTmemCols);
    }
}

// Launches one instantiation with programmatic stream serialisation (CTA
// pairs: as clusters of two, at most as many pairs as can be resident).
template <int BN, int kStages, bool kSwap, int kAccBufs, int kBlkN, int kBlkK, bool kScaleTma, bool kPair = false,
          bool kAlt = false, bool kFuse = false, bool kChan = false, bool kCK = false>
sgq_status run(const CUtensorMap* maps, const GemmArgs& args, const ExtArgs& fz, int grid, cudaStream_t st) {
    using C = Cfg<BN, kStages, kSwap, kAccBufs, kBlkN, kBlkK, kScaleTma, kPair, kAlt, kFuse, kChan, kCK>;
    auto kern = fp8_block_gemm_kernel<BN, kStages, kSwap, kAccBufs, kBlkN, kBlkK, kScaleTma, kPair, kAlt, kFuse, kChan,
                                      kCK>;
    constexpr bool kCluster = kPair || kCK;
    static bool configured[64] = {};
    static int max_pairs[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kCluster ? 2 : 1;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(C::kSmem)) != cudaSuccess)
            return SGQ_ERR_CUDA;
        if (kCluster) {
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3(static_cast<unsigned>(grid));
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess || n < 1) return SGQ_ERR_CUDA;
            max_pairs[dev] = n;
        }
        configured[dev] = true;
    }
    if (kCluster) {
        // clusters of two: a CTA pair (one item each) or the two K splits of a tile
        int pairs = grid / 2;
        if (pairs > max_pairs[dev]) pairs = max_pairs[dev];
        if (pairs > (kPair ? args.items : args.items / 2)) pairs = kPair ? args.items : args.items / 2;
        grid = 2 * pairs;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    if (cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], args, fz) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

// Which kernel configuration a launch uses (chosen by the host's plan).
struct Variant {
    bool swap;        // swap-AB narrow tiles (decode)
    bool pair;        // 256 x 256 tiles on CTA pairs
    bool alt;         // 128 x 256 tiles with two alternating MMA issuers
    bool scale_tma;   // scale boxes loaded by TMA
    bool fuse;        // swap-AB tiles that quantise the bf16 activations themselves
    bool chan;        // per-channel scaling (fp8_scaled_mm): unscaled MMAs, scales in the epilogue
    bool ck;          // swap-AB split-K over clusters of two (two splits exactly)
    int bn;           // MMA N of the swap-AB tile
};

// One translation unit per [blk_n, blk_k] recipe instantiates all tile shapes.
// maps: A operand, B operand, A-operand scales, B-operand scales.
// Pair tiles (256 x 256, cta_group::2) need TMA-loaded scales.
template <int kBlkN, int kBlkK, bool kScaleTma>
sgq_status dispatch_tile(const Variant& v, const CUtensorMap* maps, const GemmArgs& a, const ExtArgs& fz, int grid,
                         cudaStream_t st) {
    if (v.fuse) {
        if constexpr (kScaleTma) {
            switch (v.bn) {
                case 16: return run<16, 8, true, 2, kBlkN, kBlkK, true, false, false, true>(maps, a, fz, grid, st);
                case 32: return run<32, 8, true, 2, kBlkN, kBlkK, true, false, false, true>(maps, a, fz, grid, st);
                default: return run<64, 8, true, 2, kBlkN, kBlkK, true, false, false, true>(maps, a, fz, grid, st);
            }
        } else {
            return SGQ_ERR_UNSUPPORTED;
        }
    }
    if (v.pair) {
        // six stages fit beside [128,128]-recipe scale groups, five beside [32,32]
        constexpr int kPairStages = kBlkK == 32 ? 5 : 6;
        if constexpr (kScaleTma)
            return run<256, kPairStages, false, 1, kBlkN, kBlkK, true, true>(maps, a, fz, grid, st);
        else
            return SGQ_ERR_UNSUPPORTED;
    }
    if (!v.swap) {
        if (v.alt) return run<256, 4, false, 1, kBlkN, kBlkK, kScaleTma, false, true>(maps, a, fz, grid, st);
        return run<256, 4, false, 1, kBlkN, kBlkK, kScaleTma>(maps, a, fz, grid, st);
    }
    if (v.ck) {   // two splits exchanged through shared memory (BN <= 32: room for the buffer)
        if (v.bn == 16)
            return run<16, 8, true, 2, kBlkN, kBlkK, kScaleTma, false, false, false, false, true>(maps, a, fz, grid, st);
        return run<32, 8, true, 2, kBlkN, kBlkK, kScaleTma, false, false, false, false, true>(maps, a, fz, grid, st);
    }
    switch (v.bn) {
        case 16: return run<16, 8, true, 2, kBlkN, kBlkK, kScaleTma>(maps, a, fz, grid, st);
        case 32: return run<32, 8, true, 2, kBlkN, kBlkK, kScaleTma>(maps, a, fz, grid, st);
        default: return run<64, 7, true, 2, kBlkN, kBlkK, kScaleTma>(maps, a, fz, grid, st);
    }
}
template <int kBlkN, int kBlkK>
sgq_status dispatch(const Variant& v, const CUtensorMap* maps, const GemmArgs& a, const ExtArgs& fz, int grid,
                    cudaStream_t st) {
    return v.scale_tma ? dispatch_tile<kBlkN, kBlkK, true>(v, maps, a, fz, grid, st)
                       : dispatch_tile<kBlkN, kBlkK, false>(v, maps, a, fz, grid, st);
}

sgq_status dispatch_32_32(const Variant&, const CUtensorMap*, const GemmArgs&, const ExtArgs&, int, cudaStream_t);
sgq_status dispatch_32_128(const Variant&, const CUtensorMap*, const GemmArgs&, const ExtArgs&, int, cudaStream_t);
sgq_status dispatch_128_32(const Variant&, const CUtensorMap*, const GemmArgs&, const ExtArgs&, int, cudaStream_t);
sgq_status dispatch_128_128(const Variant&, const CUtensorMap*, const GemmArgs&, const ExtArgs&, int, cudaStream_t);
sgq_status dispatch_chan(const Variant&, const CUtensorMap*, const GemmArgs&, const ExtArgs&, int, cudaStream_t);

}  // namespace gemm
}  // namespace sgq
