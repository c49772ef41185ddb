// Instantiates the decode-sized GEMM for weight blocks 128 rows wide
// ([128,128] and [128,32] recipes).
#include "gemm_decode.cuh"

namespace sgq {
namespace dec {
sgq_status dispatch_n128(int blk_k, int bn, bool quant, const CUtensorMap& tmW, const DecArgs& a, int grid,
                         cudaStream_t st) {
    return blk_k == 32 ? dispatch<128, 32>(bn, quant, tmW, a, grid, st)
                       : dispatch<128, 128>(bn, quant, tmW, a, grid, st);
}
}  // namespace dec
}  // namespace sgq
