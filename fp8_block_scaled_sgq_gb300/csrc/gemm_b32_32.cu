// Instantiates the block-scaled GEMM for the [32,32] weight-block recipe
// (activation groups of 32).
#include "gemm_kernel.cuh"

namespace sgq {
namespace gemm {
sgq_status dispatch_32_32(const Variant& v, const CUtensorMap* maps, const GemmArgs& a, const ExtArgs& fz, int grid,
                           cudaStream_t st) {
    return dispatch<32, 32>(v, maps, a, fz, grid, st);
}
}  // namespace gemm
}  // namespace sgq
