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

}  // namespace qm
}  // namespace sgq
