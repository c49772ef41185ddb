// Internal host-side interface between the C-ABI layer and the kernel files.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/sgq.h"

namespace sgq {

// Per-device facts, queried once.
struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};
sgq_status device_info(DeviceInfo* out);

// Count of kernel launches made by the library (for benchmarks).
void note_launch(int n = 1);

sgq_status launch_quant_token_group(const void* x, int64_t M, int64_t K, int group,
                                    int ue8m0, void* xq, float* xs, cudaStream_t stream);
sgq_status launch_quant_token_group_e8(const void* x, int64_t M, int64_t K, int group, void* xq, uint8_t* xe,
                                       cudaStream_t stream);
// fp32 power-of-two scales -> UE8M0 bytes (255 and a device status for others).
sgq_status launch_scales_to_ue8m0(const float* s, int64_t n, uint8_t* e, cudaStream_t stream);
// UE8M0 bytes -> fp32 scales 2^(e - 127).
sgq_status launch_ue8m0_to_scales(const uint8_t* e, int64_t n, float* s, cudaStream_t stream);
sgq_status launch_fp8_block_gemm_ue8m0(const void* Aq, const uint8_t* Ae, const void* Wq, const uint8_t* We,
                                       void* D, int64_t M, int64_t N, int64_t K, int blk_n, int blk_k,
                                       uint32_t flags, cudaStream_t stream);
sgq_status launch_quant_weight_block(const void* w, int64_t N, int64_t K, int blk_n,
                                     int blk_k, int ue8m0, void* wq, float* ws,
                                     cudaStream_t stream);
sgq_status launch_quant_token_group_v2(const void* x, int64_t E, int64_t T, int64_t H, int group, int ue8m0,
                                       int fuse, const int32_t* masked_m, void* xq, float* xs,
                                       cudaStream_t stream);
sgq_status launch_quant_per_token(const void* x, int64_t M, int64_t K, void* xq, float* xs,
                                  cudaStream_t stream);
sgq_status launch_quant_per_tensor(const void* x, int64_t n, int is_static, void* xq, float* xs,
                                   cudaStream_t stream);
sgq_status launch_fp8_block_gemm(const void* Aq, const float* As, const void* Wq,
                                 const float* Ws, void* D, int64_t M, int64_t N, int64_t K,
                                 int blk_n, int blk_k, uint32_t flags, cudaStream_t stream);
sgq_status launch_fp8_block_gemm_noalloc(const void* Aq, const float* As, const void* Wq,
                                         const float* Ws, void* D, int64_t M, int64_t N, int64_t K,
                                         int blk_n, int blk_k, cudaStream_t stream);
sgq_status launch_fp8_block_linear(const void* x, int ue8m0, const void* Wq, const float* Ws, void* D,
                                   int64_t M, int64_t N, int64_t K, int blk_n, int blk_k, void* xq,
                                   float* xs, cudaStream_t stream);
sgq_status launch_fp8_scaled_mm(const void* Aq, const float* sa, int64_t sa_n, const void* Wq,
                                const float* sb, int64_t sb_n, const void* bias, void* D, int64_t M,
                                int64_t N, int64_t K, cudaStream_t stream);
// The GEMM's launch plan for a device with sm_count SMs (host only):
// out[0..7] = swap-AB, BN, K splits, work items, grid, alternating issuers,
// cluster split-K, CTA pairs.
sgq_status gemm_plan_query(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int32_t* out);
sgq_status gemm_plan_pow2_query(int64_t M, int64_t N, int64_t K, int blk_k, int sm_count, int e8, int32_t* out);
// Bytes of device memory the library has allocated on the current device.
uint64_t allocated_bytes();
// The device status word of the current device (kernels atomicOr bits into
// it: 1 a bounded wait ran out, 2 a scale broke its power-of-two promise or
// could not be expressed as UE8M0).
namespace gemm {
sgq_status status_word(uint32_t** out);
}
constexpr uint32_t kStatusBadValue = 2u;
// Reads and clears the device status word of the current device (after a sync).
sgq_status read_and_clear_device_status(cudaStream_t stream);

}  // namespace sgq
