/*
 * sgq_oracle.c -- plain, slow CPU oracle for the W8A8 FP8 block-scaled linear
 * layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header, table or constant
 * generator with the CUDA library; the two are compared against each other.
 *
 * What it computes, and where the pages define it:
 *
 *  - Per-token-group quantisation: "Sgl project Sglang GEMM Interface",
 *    Description / Quantization Routines (sgl_per_token_group_quant_8bit:
 *    group size, epsilon, clipping range, UE8M0 scale format) and its
 *    Signature section (input, output_q, output_s, group_size, eps, fp8_min,
 *    fp8_max, scale_ue8m0).  The UE8M0 rounding of activation scales is the
 *    "UE8M0 activation rounding" of sglang PR #42604 "[SM90] Use native
 *    block32 DeepGEMM for DeepSeek-V4.1", Modifications.
 *  - Weight block quantisation into [blk_n, blk_k] tiles with one scale per
 *    tile, stored [n_blocks, k_blocks]: the same PR, Motivation ([32,32] vs
 *    [128,128] blocks), and the vLLM "scaled_mm" API page,
 *    XPUFp8BlockScaledMMKernel.process_weights_after_loading ("[n_blocks,
 *    k_blocks] (one value per block tile)").
 *  - Per-token and per-tensor quantisation (sgl_per_token_quant_fp8,
 *    sgl_per_tensor_quant_fp8 with static or dynamic scaling: "Sgl project
 *    Sglang GEMM Interface", Quantization Routines and Signature) and the
 *    scaled GEMM fp8_scaled_mm (same page: per-tensor or per-row scale_a,
 *    per-tensor or per-column scale_b, optional bias, output dtype).
 *  - The V2 per-token-group quantiser's fused SiLU-and-mul and masked M (same
 *    page, Quantization Routines: "a V2 variant ... that adds fused
 *    SiLU-and-mul and masked M support"; Signature: fuse_silu_and_mul,
 *    masked_m).  Reading: input rows [gate | up] of width 2H, y = silu(gate) *
 *    up in fp32 with silu(g) = g / (1 + exp(-g)), quantised per group like x;
 *    for a [E, T, .] input, rows t >= masked_m[e] of expert e are left
 *    untouched.  exp is the Cody-Waite reduction with a degree-7 Taylor
 *    polynomial below, so that GPU and CPU produce the same fp32 value.
 *  - The GEMM: the vLLM "scaled_mm" API page,
 *    AiterInt8ScaledMMLinearKernel.apply_weights docstring: the output is
 *    mm(scale_a * a, scale_b * b) with numpy-style broadcasting of the scales,
 *    here with B given as [N, K] (the "_nt" form fp8_gemm_nt((Aq, As), (Wq,
 *    Ws), D, recipe) of the PR's Modifications).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - E4M3 is the OCP "E4M3FN" format: bias 7, no infinities, 0x7F/0xFF NaN,
 *    largest finite 448, subnormals k * 2^-9.  fp8_max = 448, fp8_min = -448.
 *  - eps = 1e-10 (fp32); scale = max(amax, eps) / 448 as a correctly rounded
 *    fp32 division; UE8M0 rounds that scale up to the next power of two.
 *  - codes = E4M3 round-to-nearest-even of clamp(x / scale, -448, 448), with
 *    x / scale a correctly rounded fp32 division; the sign of zero results is
 *    kept (-0 encodes as 0x80).
 *  - The GEMM is evaluated in fp64 on the dequantised operands.
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off [-fopenmp] (no fast-math:
 * the quantiser relies on IEEE fp32 division).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FP8_MAX 448.0f

static uint32_t orc_bits(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }
static float orc_float(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }

int sgqo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the parallel loops that follow (n < 1: all processors).  Timing
 * only: every loop computes each output on its own, so results do not depend
 * on it. */
void sgqo_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

/* bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits. */
float sgqo_bf16_to_f32(uint16_t h) { return orc_float((uint32_t)h << 16); }

/*
 * E4M3 encoder working only on the integer bits of the fp32 input.
 * Round-to-nearest-even at the E4M3 quantum of the input's binade, saturating
 * to +-448.  NaN inputs give 0x7F with the input's sign (outside the
 * contract; the quantiser never produces them from finite inputs).
 */
uint8_t sgqo_e4m3_encode(float v) {
    uint32_t u = orc_bits(v);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return (uint8_t)(sign | 0x7Fu);      /* NaN */
    if (mag >= orc_bits(ORC_FP8_MAX)) return (uint8_t)(sign | 0x7Eu); /* >= 448, inf */
    int e_field = (int)(mag >> 23);
    if (e_field == 0) return sign;   /* fp32 zero/subnormal: far below 2^-10 */
    /* value = sig * 2^(e - 23), sig in [2^23, 2^24) */
    uint32_t sig = (mag & 0x7FFFFFu) | 0x800000u;
    int e = e_field - 127;
    /* E4M3 quantum: 2^(e-3) in the normal range (e >= -6), else 2^-9. */
    int q_exp = (e >= -6) ? (e - 3) : -9;
    int shift = q_exp - (e - 23);      /* >= 20 */
    uint32_t n;
    if (shift >= 32) {
        n = 0;                         /* below half of the smallest subnormal */
    } else {
        n = sig >> shift;
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (n & 1u))) n += 1u;
    }
    /* value = n * 2^q_exp */
    if (n == 0) return sign;
    uint32_t code;
    if (q_exp == -9 && n < 8) {
        code = n;                                   /* subnormal: n * 2^-9 */
    } else if (n < 16) {
        code = ((uint32_t)(q_exp + 10) << 3) | (n - 8u);   /* (8+m) * 2^(E-10) */
    } else {                                        /* rounded up into next binade */
        code = ((uint32_t)(q_exp + 11) << 3);
    }
    if (code > 0x7Eu) code = 0x7Eu;                 /* saturate (cannot trigger below 448) */
    return (uint8_t)(sign | code);
}

void sgqo_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = sgqo_e4m3_encode(v[i]);
}

/* E4M3 decoder straight from the bit fields. */
double sgqo_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (E == 0xF && m == 7) return s ? -NAN : NAN;
    if (E == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), E - 10);
    return s ? -v : v;
}

/* Smallest power of two >= s, for positive normal s, by bits. */
float sgqo_ue8m0_ceil(float s) {
    uint32_t u = orc_bits(s);
    if (u & 0x7FFFFFu) u = (u & 0xFF800000u) + 0x800000u;
    return orc_float(u);
}

/* scale = max(amax, eps) / 448 (fp32, correctly rounded), optionally
 * rounded up to a power of two. */
float sgqo_group_scale(float amax, float eps, int ue8m0) {
    float a = amax > eps ? amax : eps;
    volatile float s = a / ORC_FP8_MAX;   /* volatile: keep it one fp32 division */
    float r = s;
    if (ue8m0) r = sgqo_ue8m0_ceil(r);
    return r;
}

/* One element: E4M3(clamp(x / s, -448, 448)). */
static uint8_t orc_quant_one(float x, float s) {
    volatile float q = x / s;
    float t = q;
    if (t > ORC_FP8_MAX) t = ORC_FP8_MAX;
    if (t < -ORC_FP8_MAX) t = -ORC_FP8_MAX;
    return sgqo_e4m3_encode(t);
}

/*
 * Per-token-group quantisation.  x: bf16 bits [M, K] row-major.
 * xq: E4M3 codes [M, K]; xs: fp32 [M, K / group] row-major.
 */
void sgqo_quant_token_group(const uint16_t* x, int64_t M, int64_t K, int group,
                            int ue8m0, float eps, uint8_t* xq, float* xs) {
    int64_t G = K / group;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = 0; j < G; ++j) {
            const uint16_t* xr = x + m * K + j * group;
            float amax = 0.0f;
            for (int i = 0; i < group; ++i) {
                float a = fabsf(sgqo_bf16_to_f32(xr[i]));
                if (a > amax) amax = a;
            }
            float s = sgqo_group_scale(amax, eps, ue8m0);
            xs[m * G + j] = s;
            for (int i = 0; i < group; ++i)
                xq[m * K + j * group + i] = orc_quant_one(sgqo_bf16_to_f32(xr[i]), s);
        }
    }
}

/*
 * Weight block quantisation.  w: bf16 bits [N, K].  One scale per
 * [blk_n, blk_k] tile; the last N-tile may be ragged and uses the rows that
 * exist.  wq: E4M3 codes [N, K]; ws: fp32 [ceil(N / blk_n), K / blk_k].
 */
void sgqo_quant_weight_block(const uint16_t* w, int64_t N, int64_t K, int blk_n,
                             int blk_k, int ue8m0, float eps, uint8_t* wq, float* ws) {
    int64_t NB = (N + blk_n - 1) / blk_n, KB = K / blk_k;
    for (int64_t nb = 0; nb < NB; ++nb) {
        int64_t n0 = nb * blk_n, n1 = n0 + blk_n < N ? n0 + blk_n : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t k0 = kb * blk_k;
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k0 + blk_k; ++k) {
                    float a = fabsf(sgqo_bf16_to_f32(w[n * K + k]));
                    if (a > amax) amax = a;
                }
            float s = sgqo_group_scale(amax, eps, ue8m0);
            ws[nb * KB + kb] = s;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = k0; k < k0 + blk_k; ++k)
                    wq[n * K + k] = orc_quant_one(sgqo_bf16_to_f32(w[n * K + k]), s);
        }
    }
}

/*
 * D[m, n] = sum_k (dec(Aq[m,k]) * As[m, k / a_group]) * (dec(Wq[n,k]) * Ws[n / blk_n, k / blk_k])
 * in fp64, and bound[m, n] = sum_k |a_deq| * |w_deq| (for the error bound).
 * Aq: [M, K]; As: [M, K / a_group]; Wq: [N, K]; Ws: [ceil(N/blk_n), K/blk_k].
 * Outputs are [M, N] row-major fp64.  bound may be NULL.
 */
void sgqo_gemm(const uint8_t* aq, const float* as, const uint8_t* wq, const float* ws,
               int64_t M, int64_t N, int64_t K, int a_group, int blk_n, int blk_k,
               double* d, double* bound) {
    int64_t AG = K / a_group, KB = K / blk_k;
    double* adeq = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            adeq[m * K + k] = sgqo_e4m3_decode(aq[m * K + k]) * (double)as[m * AG + k / a_group];
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double* wrow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k)
                wrow[k] = sgqo_e4m3_decode(wq[n * K + k]) * (double)ws[(n / blk_n) * KB + k / blk_k];
            for (int64_t m = 0; m < M; ++m) {
                const double* ar = adeq + m * K;
                double acc = 0.0, b = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    acc += ar[k] * wrow[k];
                    b += fabs(ar[k]) * fabs(wrow[k]);
                }
                d[m * N + n] = acc;
                if (bound) bound[m * N + n] = b;
            }
        }
        free(wrow);
    }
    free(adeq);
}

/*
 * Per-token quantisation (sgl_per_token_quant_fp8): one scale per row, the
 * group rule above with the group spanning the whole row.  The routine has no
 * UE8M0 option.  x: bf16 bits [M, K]; xq: [M, K]; xs: fp32 [M].
 */
void sgqo_quant_per_token(const uint16_t* x, int64_t M, int64_t K, float eps, uint8_t* xq, float* xs) {
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* xr = x + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(sgqo_bf16_to_f32(xr[k]));
            if (a > amax) amax = a;
        }
        float s = sgqo_group_scale(amax, eps, 0);
        xs[m] = s;
        for (int64_t k = 0; k < K; ++k) xq[m * K + k] = orc_quant_one(sgqo_bf16_to_f32(xr[k]), s);
    }
}

/*
 * Per-tensor quantisation (sgl_per_tensor_quant_fp8).  Dynamic (is_static =
 * 0): one scale max(amax over all n elements, eps) / 448, written to *s.
 * Static: *s is the caller's scale and only the codes are produced.
 */
void sgqo_quant_per_tensor(const uint16_t* x, int64_t n, int is_static, float eps, uint8_t* xq, float* s) {
    if (!is_static) {
        float amax = 0.0f;
        for (int64_t i = 0; i < n; ++i) {
            float a = fabsf(sgqo_bf16_to_f32(x[i]));
            if (a > amax) amax = a;
        }
        *s = sgqo_group_scale(amax, eps, 0);
    }
    float sc = *s;
    for (int64_t i = 0; i < n; ++i) xq[i] = orc_quant_one(sgqo_bf16_to_f32(x[i]), sc);
}

/*
 * Scaled GEMM (fp8_scaled_mm), B given as [N, K]:
 *   D[m, n] = (sum_k dec(Aq[m,k]) * dec(Wq[n,k])) * sa[m or 0] * sb[n or 0] + bias[n]
 * in fp64 (the scales broadcast numpy-style: sa has 1 or M values, sb 1 or N;
 * bias: bf16 bits [N] or NULL), and bound[m, n] = sum_k |a_deq| |w_deq| with the
 * scales applied.  Outputs [M, N] row-major fp64; bound may be NULL.
 */
void sgqo_scaled_mm(const uint8_t* aq, const float* sa, int64_t sa_n, const uint8_t* wq, const float* sb,
                    int64_t sb_n, const uint16_t* bias, int64_t M, int64_t N, int64_t K, double* d,
                    double* bound) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t n = 0; n < N; ++n) {
        const double bn = sb[sb_n == 1 ? 0 : n];
        const double bias_n = bias ? (double)sgqo_bf16_to_f32(bias[n]) : 0.0;
        for (int64_t m = 0; m < M; ++m) {
            const double am = sa[sa_n == 1 ? 0 : m];
            double acc = 0.0, b = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double av = sgqo_e4m3_decode(aq[m * K + k]), wv = sgqo_e4m3_decode(wq[n * K + k]);
                acc += av * wv;
                b += fabs(av) * fabs(wv);
            }
            d[m * N + n] = acc * am * bn + bias_n;
            if (bound) bound[m * N + n] = b * fabs(am * bn);
        }
    }
}

/*
 * exp(x) in fp32 by a textbook method: x = k ln2 + r with k = rint(x / ln2)
 * and ln2 split into a high part with a short mantissa and a low part (Cody &
 * Waite's reduction), |r| <= ln2/2; e^r from its Taylor series to degree 7
 * (1/n! rounded to fp32), Horner's scheme with fused multiply-adds; then
 * scaled by 2^k through the exponent field.  Below -87.3 the result is 0,
 * above 88.7 it is +inf.  Every step is one correctly rounded fp32 operation,
 * so any IEEE implementation of the same steps gives the same bits.
 */
float sgqo_exp_tc(float x) {
    if (x > 88.72f) return orc_float(0x7F800000u);
    if (x < -87.33f) return 0.0f;
    const float log2e = 1.44269504088896341f;
    const float ln2_hi = 0.693145751953125f;        /* 12 significant bits: k * ln2_hi is exact */
    const float ln2_lo = 1.42860682030941723e-6f;   /* ln2 - ln2_hi */
    volatile float kx = x * log2e;
    float k = rintf(kx);
    float r = fmaf(-k, ln2_hi, x);
    r = fmaf(-k, ln2_lo, r);
    const float c7 = (float)(1.0 / 5040.0), c6 = (float)(1.0 / 720.0), c5 = (float)(1.0 / 120.0);
    const float c4 = (float)(1.0 / 24.0), c3 = (float)(1.0 / 6.0), c2 = 0.5f;
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    /* p in [0.7, 1.42]: multiply by 2^k in two steps so that 2^k itself stays normal */
    int ki = (int)k;
    int k1 = ki / 2, k2 = ki - k1;
    volatile float q = p * orc_float((uint32_t)(k1 + 127) << 23);
    float res = q;
    volatile float q2 = res * orc_float((uint32_t)(k2 + 127) << 23);
    return q2;
}

/* y = silu(g) * u = (g / (1 + exp(-g))) * u, each step one fp32 operation. */
float sgqo_silu_mul(float g, float u) {
    volatile float den = 1.0f + sgqo_exp_tc(-g);
    volatile float s = g / den;
    volatile float y = s * u;
    return y;
}

/*
 * V2 per-token-group quantisation.  x: bf16 bits [E, T, W] with W = 2H when
 * fuse (rows [gate | up]) else W = H.  masked_m: int32 [E] or NULL (all T
 * rows).  xq: [E, T, H] codes; xs: fp32 [E, T, H / group].  Rows of expert e
 * from masked_m[e] on are not written.
 */
void sgqo_quant_token_group_v2(const uint16_t* x, int64_t E, int64_t T, int64_t H, int fuse,
                               const int32_t* masked_m, int group, int ue8m0, float eps, uint8_t* xq,
                               float* xs) {
    const int64_t W = fuse ? 2 * H : H, G = H / group;
    float* y = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
    for (int64_t e = 0; e < E; ++e) {
        int64_t rows = masked_m ? (int64_t)masked_m[e] : T;
        if (rows > T) rows = T;
        for (int64_t t = 0; t < rows; ++t) {
            const uint16_t* xr = x + (e * T + t) * W;
            for (int64_t k = 0; k < H; ++k)
                y[k] = fuse ? sgqo_silu_mul(sgqo_bf16_to_f32(xr[k]), sgqo_bf16_to_f32(xr[H + k]))
                            : sgqo_bf16_to_f32(xr[k]);
            const int64_t row = e * T + t;
            for (int64_t j = 0; j < G; ++j) {
                float amax = 0.0f;
                for (int i = 0; i < group; ++i) {
                    float a = fabsf(y[j * group + i]);
                    if (a > amax) amax = a;
                }
                float s = sgqo_group_scale(amax, eps, ue8m0);
                xs[row * G + j] = s;
                for (int i = 0; i < group; ++i) xq[row * H + j * group + i] = orc_quant_one(y[j * group + i], s);
            }
        }
    }
    free(y);
}
