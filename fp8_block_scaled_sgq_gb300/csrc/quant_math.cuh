// Per-group quantisation arithmetic, shared by the stand-alone quantisation
// kernels (quant.cu) and the GEMM that quantises its activation tiles itself
// (gemm_kernel.cuh), so that both produce the same codes and scales.
//
// The rule ("Sgl project Sglang GEMM Interface", Quantization Routines:
// sgl_per_token_group_quant_8bit with group size, eps, fp8_min/fp8_max and
// the UE8M0 scale format; UE8M0 activation rounding from sglang PR #42604,
// Modifications) for each group:
//   s = max(amax, eps) / 448   (IEEE fp32 division), optionally rounded up to
//   a power of two; code = E4M3 RNE of clamp(x / s, -448, 448).
// The conversion instruction saturates to +-448, which is the clamp.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

namespace sgq {
namespace qm {

constexpr float kFp8Max = 448.0f;
constexpr float kEps = 1e-10f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// s = max(amax, eps) / 448, optionally rounded up to a power of two (by bits).
__device__ __forceinline__ float group_scale(float amax, bool ue8m0) {
    float s = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
    if (ue8m0) {
        uint32_t u = __float_as_uint(s);
        if (u & 0x7FFFFFu) u = (u & 0xFF800000u) + 0x800000u;
        s = __uint_as_float(u);
    }
    return s;
}

// x / s for all 8 values, then E4M3 with saturation, packed little-endian.
__device__ __forceinline__ uint2 quantize8(const float (&v)[8], float s, bool ue8m0) {
    float q[8];
    if (ue8m0) {
        // s = 2^e exactly, so 1/s = 2^-e is exact and x * (1/s) is the
        // correctly rounded x / s.
        const float r = __uint_as_float((254u - (__float_as_uint(s) >> 23)) << 23);
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(v[i], r);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(v[i], s);
    }
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_fp8x2_storage_t c =
            __nv_cvt_float2_to_fp8x2(make_float2(q[2 * i], q[2 * i + 1]), __NV_SATFINITE, __NV_E4M3);
        p[i] = static_cast<uint32_t>(c);
    }
    return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
    return a;
}

// exp(x) in fp32 by a textbook method, for the fused SiLU-and-mul: x = k ln2 + r
// with k = rint(x / ln2) and ln2 split into a short-mantissa high part and a low
// part (Cody & Waite's reduction), e^r from its Taylor series to degree 7
// (1/n! rounded to fp32) by Horner's scheme with fused multiply-adds, then
// times 2^k in two exponent-field steps.  Below -87.33 the result is 0, above
// 88.72 +inf.  Each step is one correctly rounded fp32 operation (explicit
// intrinsics: nothing contracted), so the value is reproducible bit for bit.
__device__ __forceinline__ float exp_tc(float x) {
    if (x > 88.72f) return __uint_as_float(0x7F800000u);
    if (x < -87.33f) return 0.0f;
    const float k = rintf(__fmul_rn(x, 1.44269504088896341f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);
    r = __fmaf_rn(-k, 1.42860682030941723e-6f, r);
    float p = static_cast<float>(1.0 / 5040.0);
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 720.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 120.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 24.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 6.0));
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ki = static_cast<int>(k);
    const int k1 = ki / 2, k2 = ki - k1;
    p = __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(k1 + 127) << 23));
    return __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(k2 + 127) << 23));
}

// silu(g) * u = (g / (1 + exp(-g))) * u, one fp32 operation per step.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp_tc(-g))), u);
}

}  // namespace qm
}  // namespace sgq
