// Instantiates the two-accumulator prefill GEMM (power-of-two scales) with
// tiles of 192 weight rows, one CTA per tile, fp32 scales, for the four weight-block
// recipes.
#include "gemm_dual.cuh"

namespace sgq {
namespace dual {
sgq_status dispatch_192(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a,
                  int grid, cudaStream_t st) {
    return dispatch_bn<192, false, false, false>(blk_n, blk_k, tmA, tmB, a, grid, st);
}
}  // namespace dual
}  // namespace sgq
