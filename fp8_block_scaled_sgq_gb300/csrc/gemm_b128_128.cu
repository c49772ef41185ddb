// Instantiates the block-scaled GEMM for the [128,128] weight-block recipe
// (activation groups of 128).
#include "gemm_kernel.cuh"

namespace sgq {
namespace gemm {
sgq_status dispatch_128_128(const Variant& v, const CUtensorMap* maps, const GemmArgs& a, const ExtArgs& fz, int grid,
                           cudaStream_t st) {
    return dispatch<128, 128>(v, maps, a, fz, grid, st);
}
}  // namespace gemm
}  // namespace sgq
