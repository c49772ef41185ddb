// Instantiates the two-accumulator prefill GEMM (power-of-two scales) for the
// four weight-block recipes.
#include "gemm_dual.cuh"

namespace sgq {
namespace dual {
sgq_status dispatch(int blk_n, int blk_k, const CUtensorMap& tmA, const CUtensorMap& tmB, const DualArgs& a,
                    int grid, cudaStream_t st) {
    if (blk_n == 32) {
        return blk_k == 32 ? run<kBN, 32, 32>(tmA, tmB, a, grid, st) : run<kBN, 32, 128>(tmA, tmB, a, grid, st);
    }
    return blk_k == 32 ? run<kBN, 128, 32>(tmA, tmB, a, grid, st) : run<kBN, 128, 128>(tmA, tmB, a, grid, st);
}
}  // namespace dual
}  // namespace sgq
