// C-ABI entry points: argument validation, then the kernel launchers.
// Every check happens on the host before anything is enqueued; nothing
// aborts or falls back.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "sgq_internal.h"

namespace sgq {
namespace {

std::atomic<uint64_t> g_launches{0};
DeviceInfo g_dev[64];
bool g_dev_ok[64] = {};
std::mutex g_dev_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

void note_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

sgq_status device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ok[dev]) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return SGQ_ERR_CUDA;
        g_dev[dev] = d;
        g_dev_ok[dev] = true;
    }
    *out = g_dev[dev];
    return SGQ_OK;
}

}  // namespace sgq

using sgq::aligned16;

extern "C" {

sgq_status sgq_quant_token_group(const void* x, int64_t M, int64_t K, int group, int ue8m0, void* xq,
                                 float* xs, sgq_stream_t stream) {
    if (M < 0 || K <= 0 || (group != 32 && group != 128) || K % group != 0 || (ue8m0 != 0 && ue8m0 != 1))
        return SGQ_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) / 1 || M * K > (int64_t(1) << 40)) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!x || !xq || !xs) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xs)) return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_token_group(x, M, K, group, ue8m0, xq, xs,
                                         reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_quant_token_group_ue8m0(const void* x, int64_t M, int64_t K, int group, void* xq, uint8_t* xe,
                                       sgq_stream_t stream) {
    if (M < 0 || K <= 0 || (group != 32 && group != 128) || K % group != 0) return SGQ_ERR_INVALID_ARG;
    if (M > (int64_t(1) << 31) / 1 || M * K > (int64_t(1) << 40)) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!x || !xq || !xe) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xe)) return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_token_group_e8(x, M, K, group, xq, xe, reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_scales_to_ue8m0(const float* s, int64_t n, uint8_t* e, sgq_stream_t stream) {
    if (n < 0 || n > (int64_t(1) << 40)) return SGQ_ERR_INVALID_ARG;
    if (n == 0) return SGQ_OK;
    if (!s || !e) return SGQ_ERR_INVALID_ARG;
    return sgq::launch_scales_to_ue8m0(s, n, e, reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_quant_weight_block(const void* w, int64_t N, int64_t K, int blk_n, int blk_k, int ue8m0,
                                  void* wq, float* ws, sgq_stream_t stream) {
    if (N < 0 || K <= 0 || (blk_n != 32 && blk_n != 128) || (blk_k != 32 && blk_k != 128) ||
        K % blk_k != 0 || (ue8m0 != 0 && ue8m0 != 1))
        return SGQ_ERR_INVALID_ARG;
    if ((N + blk_n - 1) / blk_n > 65535 || K / blk_k > (int64_t(1) << 31) - 1) return SGQ_ERR_INVALID_ARG;
    if (N == 0) return SGQ_OK;
    if (!w || !wq || !ws) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(wq) || !aligned16(ws)) return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_weight_block(w, N, K, blk_n, blk_k, ue8m0, wq, ws,
                                          reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_fp8_block_gemm_ex(const void* Aq, const float* As, const void* Wq, const float* Ws, void* D,
                                 int64_t M, int64_t N, int64_t K, int blk_n, int blk_k, uint32_t flags,
                                 sgq_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || (blk_n != 32 && blk_n != 128) || (blk_k != 32 && blk_k != 128) ||
        K % blk_k != 0 || N % 8 != 0 ||
        (flags & ~uint32_t(SGQ_GEMM_FORCE_PROMOTE | SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE |
                           SGQ_GEMM_TEST_TIMEOUT | SGQ_GEMM_SCALES_POW2)) != 0 ||
        (flags & (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE)) == (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE))
        return SGQ_ERR_INVALID_ARG;
    // int32 indexing inside the kernel
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!Aq || !As || !Wq || !Ws || !D) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(As) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(D))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_fp8_block_gemm(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, flags,
                                      reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_fp8_block_gemm(const void* Aq, const float* As, const void* Wq, const float* Ws, void* D,
                              int64_t M, int64_t N, int64_t K, int blk_n, int blk_k, sgq_stream_t stream) {
    return sgq_fp8_block_gemm_ex(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, SGQ_GEMM_DEFAULT, stream);
}

sgq_status sgq_fp8_block_gemm_ue8m0(const void* Aq, const uint8_t* Ae, const void* Wq, const uint8_t* We, void* D,
                                    int64_t M, int64_t N, int64_t K, int blk_n, int blk_k, uint32_t flags,
                                    sgq_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || (blk_n != 32 && blk_n != 128) || (blk_k != 32 && blk_k != 128) ||
        K % blk_k != 0 || N % 8 != 0 ||
        (flags & ~uint32_t(SGQ_GEMM_FORCE_PROMOTE | SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE |
                           SGQ_GEMM_SCALES_POW2)) != 0 ||
        (flags & (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE)) == (SGQ_GEMM_ISSUE_ALT | SGQ_GEMM_ISSUE_SINGLE))
        return SGQ_ERR_INVALID_ARG;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!Aq || !Ae || !Wq || !We || !D) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(Ae) || !aligned16(Wq) || !aligned16(We) || !aligned16(D))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_fp8_block_gemm_ue8m0(Aq, Ae, Wq, We, D, M, N, K, blk_n, blk_k, flags,
                                            reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_fp8_block_gemm_noalloc(const void* Aq, const float* As, const void* Wq, const float* Ws,
                                      void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                      sgq_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || (blk_n != 32 && blk_n != 128) || (blk_k != 32 && blk_k != 128) ||
        K % blk_k != 0 || N % 8 != 0)
        return SGQ_ERR_INVALID_ARG;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!Aq || !As || !Wq || !Ws || !D) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(As) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(D))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_fp8_block_gemm_noalloc(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k,
                                              reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_quant_token_group_v2(const void* x, int64_t E, int64_t T, int64_t H, int group, int ue8m0,
                                    int fuse_silu_and_mul, const int32_t* masked_m, void* xq, float* xs,
                                    sgq_stream_t stream) {
    if (E < 0 || T < 0 || H <= 0 || (group != 32 && group != 128) || H % group != 0 ||
        (ue8m0 != 0 && ue8m0 != 1) || (fuse_silu_and_mul != 0 && fuse_silu_and_mul != 1))
        return SGQ_ERR_INVALID_ARG;
    if (E >= (int64_t(1) << 31) || T >= (int64_t(1) << 31) || E * T * H > (int64_t(1) << 40))
        return SGQ_ERR_INVALID_ARG;
    if (E == 0 || T == 0) return SGQ_OK;
    if (!x || !xq || !xs) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xs) || (masked_m && !aligned16(masked_m)))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_token_group_v2(x, E, T, H, group, ue8m0, fuse_silu_and_mul, masked_m, xq, xs,
                                            reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_quant_per_token(const void* x, int64_t M, int64_t K, void* xq, float* xs, sgq_stream_t stream) {
    if (M < 0 || K <= 0 || K % 16 != 0 || M >= (int64_t(1) << 31) || M * K > (int64_t(1) << 40))
        return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!x || !xq || !xs) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xs)) return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_per_token(x, M, K, xq, xs, reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_quant_per_tensor(const void* x, int64_t n, int is_static, void* xq, float* xs, sgq_stream_t stream) {
    if (n < 0 || n % 16 != 0 || n > (int64_t(1) << 40) || (is_static != 0 && is_static != 1))
        return SGQ_ERR_INVALID_ARG;
    if (n == 0) return SGQ_OK;
    if (!x || !xq || !xs) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xs)) return SGQ_ERR_MISALIGNED;
    return sgq::launch_quant_per_tensor(x, n, is_static, xq, xs, reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_fp8_scaled_mm(const void* Aq, const float* sa, int64_t sa_n, const void* Wq, const float* sb,
                             int64_t sb_n, const void* bias, void* D, int64_t M, int64_t N, int64_t K,
                             sgq_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || K % 32 != 0 || N % 8 != 0) return SGQ_ERR_INVALID_ARG;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return SGQ_ERR_INVALID_ARG;
    if ((sa_n != 1 && sa_n != M) || (sb_n != 1 && sb_n != N)) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!Aq || !sa || !Wq || !sb || !D) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(Aq) || !aligned16(sa) || !aligned16(Wq) || !aligned16(sb) || !aligned16(D) ||
        (bias && !aligned16(bias)))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_fp8_scaled_mm(Aq, sa, sa_n, Wq, sb, sb_n, bias, D, M, N, K,
                                     reinterpret_cast<cudaStream_t>(stream));
}

sgq_status sgq_fp8_block_linear(const void* x, int ue8m0, const void* Wq, const float* Ws, void* D, int64_t M,
                                int64_t N, int64_t K, int blk_n, int blk_k, void* xq, float* xs,
                                sgq_stream_t stream) {
    if (M < 0 || N <= 0 || K <= 0 || (blk_n != 32 && blk_n != 128) || (blk_k != 32 && blk_k != 128) ||
        K % blk_k != 0 || N % 8 != 0 || (ue8m0 != 0 && ue8m0 != 1))
        return SGQ_ERR_INVALID_ARG;
    if (M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return SGQ_ERR_INVALID_ARG;
    if ((xq == nullptr) != (xs == nullptr)) return SGQ_ERR_INVALID_ARG;
    if (M == 0) return SGQ_OK;
    if (!x || !Wq || !Ws || !D) return SGQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wq) || !aligned16(Ws) || !aligned16(D) || (xq && !aligned16(xq)) ||
        (xs && !aligned16(xs)))
        return SGQ_ERR_MISALIGNED;
    return sgq::launch_fp8_block_linear(x, ue8m0, Wq, Ws, D, M, N, K, blk_n, blk_k, xq, xs,
                                        reinterpret_cast<cudaStream_t>(stream));
}

const char* sgq_status_string(sgq_status s) {
    switch (s) {
        case SGQ_OK: return "SGQ_OK";
        case SGQ_ERR_INVALID_ARG: return "SGQ_ERR_INVALID_ARG";
        case SGQ_ERR_UNSUPPORTED: return "SGQ_ERR_UNSUPPORTED";
        case SGQ_ERR_MISALIGNED: return "SGQ_ERR_MISALIGNED";
        case SGQ_ERR_CUDA: return "SGQ_ERR_CUDA";
        case SGQ_ERR_TIMEOUT: return "SGQ_ERR_TIMEOUT";
    }
    return "SGQ_ERR_UNKNOWN";
}

sgq_status sgq_device_status(sgq_stream_t stream) {
    return sgq::read_and_clear_device_status(reinterpret_cast<cudaStream_t>(stream));
}

uint64_t sgq_launch_count(void) { return sgq::g_launches.load(std::memory_order_relaxed); }

uint64_t sgq_allocated_bytes(void) { return sgq::allocated_bytes(); }

sgq_status sgq_gemm_plan(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int32_t* out) {
    if (out == nullptr || M < 1 || N < 1 || K < 1 || (blk_k != 32 && blk_k != 128) || sm_count < 1)
        return SGQ_ERR_INVALID_ARG;
    return sgq::gemm_plan_query(M, N, K, blk_k, sm_count, out);
}

sgq_status sgq_gemm_plan_pow2(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int e8, int32_t* out) {
    if (out == nullptr || M < 1 || N < 1 || K < 1 || (blk_k != 32 && blk_k != 128) || sm_count < 2 ||
        (e8 != 0 && e8 != 1))
        return SGQ_ERR_INVALID_ARG;
    return sgq::gemm_plan_pow2_query(M, N, K, blk_k, sm_count, e8, out);
}

int sgq_version(void) { return 104; }

}  // extern "C"
