// Instantiates the two-accumulator prefill GEMM (power-of-two scales) for
// CTA pairs: tiles of 512 activation rows x 192 weight rows over a cluster of
// two, for the four weight-block recipes.
#include "gemm_dual.cuh"

namespace sgq {
namespace dual {
sgq_status dispatch_192_pair(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const DualArgs& a, int grid, cudaStream_t st) {
    return dispatch_bn<192, false, true>(blk_n, blk_k, tmA, tmB, a, grid, st);
}
}  // namespace dual
}  // namespace sgq
