// Per-token-group activation quantisation and per-block weight quantisation,
// bf16 -> FP8 E4M3 codes + fp32 scales, for sm_103a.  The per-group rule is in
// quant_math.cuh.
//
// Memory path: 16-byte bf16 loads (8 elements per thread), a warp-shuffle
// amax over the lanes of one group, packed 8-byte code stores and one
// coalesced fp32 scale store per group.  The kernel is HBM-bound.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"
#include "quant_math.cuh"
#include "sgq_internal.h"

namespace sgq {
namespace {

using qm::group_scale;
using qm::quantize8;
using qm::unpack8;

// One thread per 8 consecutive elements; kTpg = group/8 consecutive lanes own
// one group.  Loop trip counts are warp-uniform so the shuffles see full warps.
// kE8: the group scales (powers of two) are stored as UE8M0 bytes (their
// biased exponent field) in xs, uint8 [M, K / group], instead of fp32.
template <int kGroup, bool kUe8m0, bool kE8 = false>
__global__ void __launch_bounds__(256) quant_token_group_kernel(const uint4* __restrict__ x,
                                                                uint2* __restrict__ xq,
                                                                void* __restrict__ xs_out,
                                                                int64_t nvec) {
    static_assert(!kE8 || kUe8m0, "UE8M0 bytes need power-of-two scales");
    // Let a programmatically-dependent GEMM launch now, so that its weight
    // prefetch overlaps this kernel; it still waits for this grid to finish
    // before it reads xq / xs.
    ptx::launch_dependents();
    // Launched with programmatic stream serialisation: the launch overlaps the
    // previous kernel on the stream, so wait for it before touching memory
    // (x may be its output; xq/xs may still be read by it).
    ptx::grid_dependency_wait();
    constexpr int kTpg = kGroup / 8;
    // Each warp iteration loads kUnroll warp-wide chunks of 32 vectors before
    // processing any, so every thread keeps kUnroll 16-byte loads in flight
    // (an HBM-bound stream needs tens of KB outstanding per SM).
    constexpr int kUnroll = 4;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = nwarps * 32;
    for (int64_t base = warp * 32; base < nvec; base += stride * kUnroll) {
        uint4 w[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = base + u * stride + lane;
            w[u] = v < nvec ? __ldg(x + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = base + u * stride + lane;
            const bool active = v < nvec;
            float f[8];
            unpack8(w[u], f);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
            for (int off = kTpg / 2; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
            const float s = group_scale(amax, kUe8m0);
            if constexpr (kE8) {
                // The warp's 32 / kTpg group bytes are consecutive in xe: lane 0
                // gathers them and stores them at once (8 or 2 bytes) when the
                // whole chunk is in range; a ragged last chunk stores per group.
                constexpr int kGroupsPerWarp = 32 / kTpg;
                const uint32_t e = __float_as_uint(s) >> 23;
                uint8_t* xe = static_cast<uint8_t*>(xs_out);
                const int64_t v0 = base + u * stride;
                if (v0 + 31 < nvec) {
                    // pack by halving: the leader of group j ends up with groups j, j+1, ...
                    uint32_t w = e & 0xFFu;
#pragma unroll
                    for (int d = kTpg, sh = 8; d < 32 && sh < 32; d *= 2, sh *= 2)
                        w |= __shfl_down_sync(0xFFFFFFFFu, w, d) << sh;
                    if (active) xq[v] = quantize8(f, s, kUe8m0);
                    if constexpr (kGroupsPerWarp == 8) {
                        const uint32_t hi = __shfl_sync(0xFFFFFFFFu, w, 16);   // groups 4 .. 7
                        if (lane == 0)
                            *reinterpret_cast<uint2*>(xe + v0 / kTpg) = make_uint2(w, hi);
                    } else {
                        if (lane == 0) *reinterpret_cast<uint16_t*>(xe + v0 / kTpg) = static_cast<uint16_t>(w);
                    }
                } else if (active) {
                    xq[v] = quantize8(f, s, kUe8m0);
                    if ((lane % kTpg) == 0) xe[v / kTpg] = static_cast<uint8_t>(e);
                }
            } else if constexpr (kGroup == 128) {
                // fp32 scales, group 128: the warp's two group scales go out as
                // one 8-byte store when the chunk is whole (measured 32.0 ->
                // 29.3 us at 8192 x 7168; for group 32 the eight shuffles cost
                // more than the per-group stores they replace).
                float* xs = static_cast<float*>(xs_out);
                const int64_t v0 = base + u * stride;
                if (v0 + 31 < nvec) {
                    const float s1 = __shfl_sync(0xFFFFFFFFu, s, kTpg);
                    if (active) xq[v] = quantize8(f, s, kUe8m0);
                    if (lane == 0) *reinterpret_cast<float2*>(xs + v0 / kTpg) = make_float2(s, s1);
                } else if (active) {
                    xq[v] = quantize8(f, s, kUe8m0);
                    if ((lane % kTpg) == 0) xs[v / kTpg] = s;
                }
            } else if (active) {
                xq[v] = quantize8(f, s, kUe8m0);
                if ((lane % kTpg) == 0) static_cast<float*>(xs_out)[v / kTpg] = s;
            }
        }
    }
}

// 32-byte accesses: one thread per 16 consecutive elements (one 256-bit load,
// one 16-byte code store), so a group spans kGroup / 16 lanes and its amax
// takes one shuffle step fewer than with 16-byte accesses.  Group 128: the
// warp's four group scales leave in one store; group 32: each group's first
// lane stores its scale (the warp's 16 scales are contiguous).  The same
// arithmetic per group as quant_token_group_kernel: the same codes and
// scales.  x must be 32-byte aligned (the host takes the 16-byte kernel
// otherwise).
template <int kGroup, bool kUe8m0, bool kE8 = false>
__global__ void __launch_bounds__(256, kGroup == 32 ? 2 : 3) quant_token_group_w_kernel(const uint4* __restrict__ x,
                                                                      uint4* __restrict__ xq,
                                                                      void* __restrict__ xs_out,
                                                                      int64_t nchunk) {
    static_assert(!kE8 || kUe8m0, "UE8M0 bytes need power-of-two scales");
    static_assert(kGroup == 32 || kGroup == 128, "group");
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    constexpr int kTpg = kGroup / 16;   // lanes per group
    constexpr int kUnroll = 4;    // 32-byte loads in flight per thread
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t stride = nwarps * 32;
    for (int64_t base = warp * 32; base < nchunk; base += stride * kUnroll) {
        uint32_t w[kUnroll][8];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v = base + u * stride + lane;
            if (v < nchunk) {
                asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                             : "=r"(w[u][0]), "=r"(w[u][1]), "=r"(w[u][2]), "=r"(w[u][3]), "=r"(w[u][4]),
                               "=r"(w[u][5]), "=r"(w[u][6]), "=r"(w[u][7])
                             : "l"(x + 2 * v));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[u][i] = 0u;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t v0 = base + u * stride, v = v0 + lane;
            const bool active = v < nchunk;
            float f0[8], f1[8];
            unpack8(make_uint4(w[u][0], w[u][1], w[u][2], w[u][3]), f0);
            unpack8(make_uint4(w[u][4], w[u][5], w[u][6], w[u][7]), f1);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(f0[i]), fabsf(f1[i])));
#pragma unroll
            for (int off = kTpg / 2; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
            const float s = group_scale(amax, kUe8m0);
            const uint2 q0 = quantize8(f0, s, kUe8m0), q1 = quantize8(f1, s, kUe8m0);
            if (active) xq[v] = make_uint4(q0.x, q0.y, q1.x, q1.y);
            if constexpr (kGroup == 32) {
                if (active && (lane % kTpg) == 0) {
                    if constexpr (kE8) static_cast<uint8_t*>(xs_out)[v / kTpg] = static_cast<uint8_t>(__float_as_uint(s) >> 23);
                    else static_cast<float*>(xs_out)[v / kTpg] = s;
                }
                continue;
            }
            // group 128: the scales of the warp's four groups (lanes 0, 8, 16, 24)
            const bool whole = v0 + 31 < nchunk;
            if constexpr (kE8) {
                uint8_t* xe = static_cast<uint8_t*>(xs_out);
                const uint32_t e = __float_as_uint(s) >> 23;
                uint32_t word = e & 0xFFu;
                word |= __shfl_down_sync(0xFFFFFFFFu, word, 8) << 8;
                word |= __shfl_down_sync(0xFFFFFFFFu, word, 16) << 16;
                if (whole) {
                    if (lane == 0) *reinterpret_cast<uint32_t*>(xe + v0 / kTpg) = word;
                } else if (active && (lane % kTpg) == 0) {
                    xe[v / kTpg] = static_cast<uint8_t>(e);
                }
            } else {
                float* xs = static_cast<float*>(xs_out);
                const float s1 = __shfl_sync(0xFFFFFFFFu, s, 8), s2 = __shfl_sync(0xFFFFFFFFu, s, 16),
                            s3 = __shfl_sync(0xFFFFFFFFu, s, 24);
                if (whole) {
                    if (lane == 0) *reinterpret_cast<float4*>(xs + v0 / kTpg) = make_float4(s, s1, s2, s3);
                } else if (active && (lane % kTpg) == 0) {
                    xs[v / kTpg] = s;
                }
            }
        }
    }
}

// One CTA per [blk_n, blk_k] weight tile: block-wide amax, then quantise.
template <int kBlkN, int kBlkK, bool kUe8m0>
__global__ void __launch_bounds__(256) quant_weight_block_kernel(const uint16_t* __restrict__ w,
                                                                 uint8_t* __restrict__ wq,
                                                                 float* __restrict__ ws, int64_t N,
                                                                 int64_t K) {
    constexpr int kVecPerRow = kBlkK / 8;
    constexpr int kVecs = kBlkN * kVecPerRow;
    constexpr int kPer = (kVecs + 255) / 256;
    __shared__ float red[8];
    const int64_t nb = blockIdx.y, kb = blockIdx.x;
    const int64_t KB = K / kBlkK;
    uint4 data[kPer];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int idx = threadIdx.x + i * 256;
        const int r = idx / kVecPerRow, c = idx % kVecPerRow;
        const int64_t n = nb * kBlkN + r;
        data[i] = make_uint4(0, 0, 0, 0);
        if (idx < kVecs && n < N)
            data[i] = __ldg(reinterpret_cast<const uint4*>(w + n * K + kb * kBlkK) + c);
        float f[8];
        unpack8(data[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float s = group_scale(amax, kUe8m0);
    if (threadIdx.x == 0) ws[nb * KB + kb] = s;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int idx = threadIdx.x + i * 256;
        const int r = idx / kVecPerRow, c = idx % kVecPerRow;
        const int64_t n = nb * kBlkN + r;
        if (idx < kVecs && n < N) {
            float f[8];
            unpack8(data[i], f);
            reinterpret_cast<uint2*>(wq + n * K + kb * kBlkK)[c] = quantize8(f, s, kUe8m0);
        }
    }
}

// ---------------------------------------------------------------------------
// V2 per-token-group quantisation ("Sgl project Sglang GEMM Interface",
// Quantization Routines: the V2 variant of sgl_per_token_group_quant_8bit with
// fused SiLU-and-mul and masked M).  x: bf16 [E, T, W] with W = 2H (rows
// [gate | up]) when fused, else H; the quantised value is silu(gate) * up (or
// x) in fp32.  Rows t >= masked_m[e] of expert e are skipped (not written).
// One thread per 8 outputs, kTpg = group/8 lanes per group as above; a
// warp's lanes never straddle a group (H % group == 0).
template <int kGroup, bool kUe8m0, bool kFuse>
__global__ void __launch_bounds__(256) quant_token_group_v2_kernel(const uint4* __restrict__ x,
                                                                   const int32_t* __restrict__ masked_m,
                                                                   uint2* __restrict__ xq, float* __restrict__ xs,
                                                                   int64_t nvec, int64_t vpr, int64_t T) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    constexpr int kTpg = kGroup / 8;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = warp * 32; base < nvec; base += nwarps * 32) {
        const int64_t v = base + lane;
        const int64_t row = v / vpr, c = v - row * vpr;
        bool active = v < nvec;
        if (active && masked_m != nullptr) {
            const int64_t e = row / T;
            active = row - e * T < static_cast<int64_t>(__ldg(masked_m + e));
        }
        float f[8];
        if (active) {
            if (kFuse) {
                float g[8], u[8];
                unpack8(__ldg(x + row * 2 * vpr + c), g);
                unpack8(__ldg(x + row * 2 * vpr + vpr + c), u);
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = qm::silu_mul(g[i], u[i]);
            } else {
                unpack8(__ldg(x + row * vpr + c), f);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = 0.0f;
        }
        float amax = qm::amax8(f);
#pragma unroll
        for (int off = kTpg / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        const float s = group_scale(amax, kUe8m0);
        if (active) {
            xq[v] = quantize8(f, s, kUe8m0);
            if ((lane % kTpg) == 0) xs[v / kTpg] = s;
        }
    }
}

// ---------------------------------------------------------------------------
// Per-token quantisation (sgl_per_token_quant_fp8, "Sgl project Sglang GEMM
// Interface", Quantization Routines): one scale per row, the group rule with
// the group spanning the whole row.  One CTA per row (grid-stride over rows):
// an amax pass over the row's 16-byte vectors, a block reduction, then a
// second pass that writes the codes.
constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    const int w = threadIdx.x >> 5;
    __syncthreads();   // red may still be read from the previous row
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float m = red[0];
#pragma unroll
    for (int i = 1; i < kRowThreads / 32; ++i) m = fmaxf(m, red[i]);
    return m;
}

// Rows of up to kRowThreads * kRowRegs vectors (K <= 8192) stay in registers
// between the two passes; longer rows are read a second time (from L1/L2).
// Six CTAs per SM keep about 80 KB of each SM's loads in flight.
constexpr int kRowRegs = 4;

__global__ void __launch_bounds__(kRowThreads, 6) quant_per_token_kernel(const uint4* __restrict__ x,
                                                                      uint2* __restrict__ xq,
                                                                      float* __restrict__ xs, int64_t M,
                                                                      int64_t vpr) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    __shared__ float red[kRowThreads / 32];
    const bool in_regs = vpr <= int64_t(kRowThreads) * kRowRegs;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint4* xr = x + m * vpr;
        float amax = 0.0f;
        uint4 w[kRowRegs];
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < kRowRegs; ++i) {   // all loads in flight before any use
                const int64_t v = threadIdx.x + int64_t(i) * kRowThreads;
                w[i] = v < vpr ? __ldg(xr + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < kRowRegs; ++i) {
                float f[8];
                unpack8(w[i], f);
                amax = fmaxf(amax, qm::amax8(f));
            }
        } else {
            for (int64_t v = threadIdx.x; v < vpr; v += kRowThreads) {
                float f[8];
                unpack8(__ldg(xr + v), f);
                amax = fmaxf(amax, qm::amax8(f));
            }
        }
        const float s = group_scale(block_max(amax, red), false);
        if (threadIdx.x == 0) xs[m] = s;
        if (in_regs) {
#pragma unroll
            for (int i = 0; i < kRowRegs; ++i) {
                const int64_t v = threadIdx.x + int64_t(i) * kRowThreads;
                if (v < vpr) {
                    float f[8];
                    unpack8(w[i], f);
                    xq[m * vpr + v] = quantize8(f, s, false);
                }
            }
        } else {
            for (int64_t v = threadIdx.x; v < vpr; v += kRowThreads) {
                float f[8];
                unpack8(__ldg(xr + v), f);
                xq[m * vpr + v] = quantize8(f, s, false);
            }
        }
    }
}

// Short rows (K <= 2048: at most 8 vectors per lane): one warp per row, the
// whole row in registers, a shuffle-only reduction, so a CTA has eight rows in
// flight instead of one.
constexpr int kWarpRowRegs = 8;

__global__ void __launch_bounds__(kRowThreads) quant_per_token_warp_kernel(const uint4* __restrict__ x,
                                                                           uint2* __restrict__ xq,
                                                                           float* __restrict__ xs, int64_t M,
                                                                           int64_t vpr) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nw = int64_t(gridDim.x) * (kRowThreads / 32);
    for (int64_t m = int64_t(blockIdx.x) * (kRowThreads / 32) + (threadIdx.x >> 5); m < M; m += nw) {
        const uint4* xr = x + m * vpr;
        uint4 w[kWarpRowRegs];
#pragma unroll
        for (int i = 0; i < kWarpRowRegs; ++i) {
            const int64_t v = lane + 32 * i;
            w[i] = v < vpr ? __ldg(xr + v) : make_uint4(0, 0, 0, 0);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kWarpRowRegs; ++i) {
            float f[8];
            unpack8(w[i], f);
            amax = fmaxf(amax, qm::amax8(f));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        const float s = group_scale(amax, false);
        if (lane == 0) xs[m] = s;
#pragma unroll
        for (int i = 0; i < kWarpRowRegs; ++i) {
            const int64_t v = lane + 32 * i;
            if (v < vpr) {
                float f[8];
                unpack8(w[i], f);
                xq[m * vpr + v] = quantize8(f, s, false);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Per-tensor quantisation (sgl_per_tensor_quant_fp8, same page: static or
// dynamic scaling).  Dynamic: the first kernel writes one amax per CTA to a
// fixed device array; the second kernel's CTAs each reduce those partials to
// the same scale (CTA 0 stores it) and quantise.  Static: only the second
// kernel, with the caller's scale.
constexpr int kAmaxParts = 1024;
__device__ float g_amax_parts[kAmaxParts];

__global__ void __launch_bounds__(kRowThreads) amax_partial_kernel(const uint4* __restrict__ x, int64_t nvec) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();
    __shared__ float red[kRowThreads / 32];
    float amax = 0.0f;
    for (int64_t v = blockIdx.x * int64_t(kRowThreads) + threadIdx.x; v < nvec;
         v += int64_t(gridDim.x) * kRowThreads) {
        float f[8];
        unpack8(__ldg(x + v), f);
        amax = fmaxf(amax, qm::amax8(f));
    }
    amax = block_max(amax, red);
    if (threadIdx.x == 0) g_amax_parts[blockIdx.x] = amax;
}

__global__ void __launch_bounds__(kRowThreads) quant_per_tensor_kernel(const uint4* __restrict__ x,
                                                                       uint2* __restrict__ xq, float* xs,
                                                                       int64_t nvec, int nparts, int is_static) {
    ptx::launch_dependents();
    ptx::grid_dependency_wait();   // the partials (or the caller's scale) are ready
    __shared__ float red[kRowThreads / 32];
    float s;
    if (is_static) {
        s = xs[0];
    } else {
        float amax = 0.0f;
        for (int i = threadIdx.x; i < nparts; i += kRowThreads) amax = fmaxf(amax, g_amax_parts[i]);
        s = group_scale(block_max(amax, red), false);
        if (blockIdx.x == 0 && threadIdx.x == 0) xs[0] = s;
    }
    for (int64_t v = blockIdx.x * int64_t(kRowThreads) + threadIdx.x; v < nvec;
         v += int64_t(gridDim.x) * kRowThreads) {
        float f[8];
        unpack8(__ldg(x + v), f);
        xq[v] = quantize8(f, s, false);
    }
}

template <int G, bool U, bool E8>
sgq_status launch_tgw(const void* x, int64_t M, int64_t K, void* xq, void* xs, cudaStream_t st) {
    const int64_t nchunk = M * K / 16;
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    static int resident[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    if (resident[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_token_group_w_kernel<G, U, E8>, 256, 0) !=
                cudaSuccess ||
            n < 1)
            return SGQ_ERR_CUDA;
        resident[dev] = n;
    }
    int64_t blocks = ((nchunk + 31) / 32 + 7) / 8;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * resident[dev];
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quant_token_group_w_kernel<G, U, E8>, static_cast<const uint4*>(x),
                           static_cast<uint4*>(xq), xs, nchunk) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

template <int G, bool U, bool E8 = false>
sgq_status launch_tg(const void* x, int64_t M, int64_t K, void* xq, void* xs, cudaStream_t st) {
    // Large x on a 32-byte boundary: 32-byte accesses (4096 x 7168: 0.87 ->
    // 0.99 of HBM at group 128, 0.86 -> 0.97 to UE8M0 bytes at group 32).
    // Decode-sized x keeps the 16-byte kernel, whose latency is lower there.
    if ((reinterpret_cast<uintptr_t>(x) & 31u) == 0 && M * K >= (int64_t(1) << 20))
        return launch_tgw<G, U, E8>(x, M, K, xq, xs, st);
    const int64_t nvec = M * K / 8;
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    // One wave of resident CTAs at most (grid-stride loop beyond that).
    static int resident[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    if (resident[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quant_token_group_kernel<G, U, E8>, 256, 0) != cudaSuccess ||
            n < 1)
            return SGQ_ERR_CUDA;
        resident[dev] = n;
    }
    const int64_t warps_needed = (nvec + 31) / 32;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(di.sm_count) * resident[dev];
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, quant_token_group_kernel<G, U, E8>, static_cast<const uint4*>(x),
                           static_cast<uint2*>(xq), xs, nvec) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

template <int BN, int BK, bool U>
sgq_status launch_wb(const void* w, int64_t N, int64_t K, void* wq, float* ws, cudaStream_t st) {
    dim3 grid(static_cast<unsigned>(K / BK), static_cast<unsigned>((N + BN - 1) / BN));
    quant_weight_block_kernel<BN, BK, U><<<grid, 256, 0, st>>>(
        static_cast<const uint16_t*>(w), static_cast<uint8_t*>(wq), ws, N, K);
    if (cudaGetLastError() != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, int blocks, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kRowThreads);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

sgq_status launch_quant_token_group(const void* x, int64_t M, int64_t K, int group, int ue8m0,
                                    void* xq, float* xs, cudaStream_t st) {
    if (group == 32) return ue8m0 ? launch_tg<32, true>(x, M, K, xq, xs, st)
                                  : launch_tg<32, false>(x, M, K, xq, xs, st);
    return ue8m0 ? launch_tg<128, true>(x, M, K, xq, xs, st)
                 : launch_tg<128, false>(x, M, K, xq, xs, st);
}

sgq_status launch_quant_token_group_e8(const void* x, int64_t M, int64_t K, int group, void* xq, uint8_t* xe,
                                       cudaStream_t st) {
    return group == 32 ? launch_tg<32, true, true>(x, M, K, xq, xe, st) : launch_tg<128, true, true>(x, M, K, xq, xe, st);
}

namespace {
// UE8M0 byte of a positive normal power of two: its biased exponent field;
// anything else -> 255 (the format's NaN) and a status bit.
__global__ void __launch_bounds__(256) scales_to_ue8m0_kernel(const float* __restrict__ s, int64_t n,
                                                              uint8_t* __restrict__ e, uint32_t* status) {
    uint32_t bad = 0;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const uint32_t b = __float_as_uint(__ldg(s + i));
        const uint32_t x = (b >> 23) & 0xFFu;
        const bool ok = (b & 0x807FFFFFu) == 0u && x >= 1u && x <= 254u;
        e[i] = static_cast<uint8_t>(ok ? x : 255u);
        bad |= ok ? 0u : 1u;
    }
    if (__any_sync(0xFFFFFFFFu, bad != 0u) && (threadIdx.x & 31) == 0) atomicOr(status, kStatusBadValue);
}
// fp32 value 2^(e - 127) of a UE8M0 byte (255 -> NaN), by its bits.
__global__ void __launch_bounds__(256) ue8m0_to_scales_kernel(const uint8_t* __restrict__ e, int64_t n,
                                                              float* __restrict__ s) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const uint32_t x = __ldg(e + i);
        s[i] = __uint_as_float(x == 255u ? 0x7FC00000u : (x == 0u ? 0x00400000u : x << 23));
    }
}
int elementwise_blocks(int64_t n) {
    DeviceInfo di;
    if (device_info(&di) != SGQ_OK) return 1;
    const int64_t want = (n + 255) / 256;
    const int64_t cap = int64_t(di.sm_count) * 8;
    return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}
}  // namespace

sgq_status launch_scales_to_ue8m0(const float* s, int64_t n, uint8_t* e, cudaStream_t st) {
    if (n == 0) return SGQ_OK;
    uint32_t* status = nullptr;
    const sgq_status rc = gemm::status_word(&status);
    if (rc != SGQ_OK) return rc;
    scales_to_ue8m0_kernel<<<elementwise_blocks(n), 256, 0, st>>>(s, n, e, status);
    if (cudaGetLastError() != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

sgq_status launch_ue8m0_to_scales(const uint8_t* e, int64_t n, float* s, cudaStream_t st) {
    if (n == 0) return SGQ_OK;
    ue8m0_to_scales_kernel<<<elementwise_blocks(n), 256, 0, st>>>(e, n, s);
    if (cudaGetLastError() != cudaSuccess) return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

sgq_status launch_quant_weight_block(const void* w, int64_t N, int64_t K, int blk_n, int blk_k,
                                     int ue8m0, void* wq, float* ws, cudaStream_t st) {
#define SGQ_WB(bn, bk)                                                               \
    if (blk_n == bn && blk_k == bk)                                                  \
        return ue8m0 ? launch_wb<bn, bk, true>(w, N, K, wq, ws, st)                  \
                     : launch_wb<bn, bk, false>(w, N, K, wq, ws, st);
    SGQ_WB(32, 32)
    SGQ_WB(32, 128)
    SGQ_WB(128, 32)
    SGQ_WB(128, 128)
#undef SGQ_WB
    return SGQ_ERR_INVALID_ARG;
}

sgq_status launch_quant_per_token(const void* x, int64_t M, int64_t K, void* xq, float* xs, cudaStream_t st) {
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    const int64_t vpr = K / 8;
    cudaLaunchAttribute attr[1];
    if (vpr <= 32 * kWarpRowRegs) {   // a warp per row
        const int64_t want = (M + kRowThreads / 32 - 1) / (kRowThreads / 32);
        const int64_t cap = int64_t(di.sm_count) * 8;
        cudaLaunchConfig_t cfg = pdl_config(attr, static_cast<int>(want < cap ? want : cap), st);
        if (cudaLaunchKernelEx(&cfg, quant_per_token_warp_kernel, static_cast<const uint4*>(x),
                               static_cast<uint2*>(xq), xs, M, vpr) != cudaSuccess)
            return SGQ_ERR_CUDA;
        note_launch();
        return SGQ_OK;
    }
    // one CTA per row (the hardware balances the waves), capped for huge M
    const int64_t cap = int64_t(1) << 20;
    const int blocks = static_cast<int>(M < cap ? M : cap);
    cudaLaunchConfig_t cfg = pdl_config(attr, blocks, st);
    if (cudaLaunchKernelEx(&cfg, quant_per_token_kernel, static_cast<const uint4*>(x), static_cast<uint2*>(xq), xs,
                           M, vpr) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

sgq_status launch_quant_per_tensor(const void* x, int64_t n, int is_static, void* xq, float* xs, cudaStream_t st) {
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    const int64_t nvec = n / 8;
    int64_t blocks = (nvec + kRowThreads - 1) / kRowThreads;
    const int64_t cap = int64_t(di.sm_count) * 4 < kAmaxParts ? int64_t(di.sm_count) * 4 : kAmaxParts;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr[1];
    if (!is_static) {
        cudaLaunchConfig_t cfg = pdl_config(attr, static_cast<int>(blocks), st);
        if (cudaLaunchKernelEx(&cfg, amax_partial_kernel, static_cast<const uint4*>(x), nvec) != cudaSuccess)
            return SGQ_ERR_CUDA;
        note_launch();
    }
    cudaLaunchConfig_t cfg = pdl_config(attr, static_cast<int>(blocks), st);
    if (cudaLaunchKernelEx(&cfg, quant_per_tensor_kernel, static_cast<const uint4*>(x), static_cast<uint2*>(xq), xs,
                           nvec, static_cast<int>(blocks), is_static) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}

namespace {
template <int G, bool U, bool F>
sgq_status launch_v2(const void* x, int64_t E, int64_t T, int64_t H, const int32_t* masked_m, void* xq, float* xs,
                     cudaStream_t st) {
    DeviceInfo di;
    sgq_status rc = device_info(&di);
    if (rc != SGQ_OK) return rc;
    const int64_t nvec = E * T * H / 8;
    int64_t blocks = (nvec + 255) / 256;
    const int64_t cap = int64_t(di.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(attr, static_cast<int>(blocks), st);
    cfg.blockDim = dim3(256);
    if (cudaLaunchKernelEx(&cfg, quant_token_group_v2_kernel<G, U, F>, static_cast<const uint4*>(x), masked_m,
                           static_cast<uint2*>(xq), xs, nvec, H / 8, T) != cudaSuccess)
        return SGQ_ERR_CUDA;
    note_launch();
    return SGQ_OK;
}
}  // namespace

sgq_status launch_quant_token_group_v2(const void* x, int64_t E, int64_t T, int64_t H, int group, int ue8m0,
                                       int fuse, const int32_t* masked_m, void* xq, float* xs, cudaStream_t st) {
#define SGQ_V2(g, u, f)                                                                  \
    if (group == g && (ue8m0 != 0) == u && (fuse != 0) == f)                            \
        return launch_v2<g, u, f>(x, E, T, H, masked_m, xq, xs, st);
    SGQ_V2(32, false, false) SGQ_V2(32, false, true) SGQ_V2(32, true, false) SGQ_V2(32, true, true)
    SGQ_V2(128, false, false) SGQ_V2(128, false, true) SGQ_V2(128, true, false) SGQ_V2(128, true, true)
#undef SGQ_V2
    return SGQ_ERR_INVALID_ARG;
}

}  // namespace sgq
