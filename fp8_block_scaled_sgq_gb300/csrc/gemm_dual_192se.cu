// Instantiates the two-accumulator prefill GEMM (power-of-two scales) with
// tiles of 192 weight rows, K split over several CTAs per tile, UE8M0 scale bytes, for the four weight-block
// recipes.
#include "gemm_dual.cuh"

namespace sgq {
namespace dual {
sgq_status dispatch_192_split_e8(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a,
                  int grid, cudaStream_t st) {
    return dispatch_bn<192, true, false, true>(blk_n, blk_k, tmA, tmB, a, grid, st);
}
}  // namespace dual
}  // namespace sgq
