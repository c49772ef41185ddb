// Instantiates the block-scaled GEMM for the [32,32] weight-block recipe
// (activation groups of 32).
#include "gemm_kernel.cuh"

namespace sgq {
namespace gemm {
sgq_status dispatch_32_32(bool swap, bool pair, int bn, bool scale_tma, const CUtensorMap* maps, const GemmArgs& a,
                           int grid, cudaStream_t st) {
    return dispatch<32, 32>(swap, pair, bn, scale_tma, maps, a, grid, st);
}
}  // namespace gemm
}  // namespace sgq
