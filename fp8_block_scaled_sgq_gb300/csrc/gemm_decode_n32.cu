// Instantiates the decode-sized GEMM for weight blocks 32 rows wide
// ([32,32] and [32,128] recipes).
#include "gemm_decode.cuh"

namespace sgq {
namespace dec {
sgq_status dispatch_n32(int blk_k, int bn, bool quant, const CUtensorMap& tmW, const DecArgs& a, int grid,
                        cudaStream_t st) {
    return blk_k == 32 ? dispatch<32, 32>(bn, quant, tmW, a, grid, st) : dispatch<32, 128>(bn, quant, tmW, a, grid, st);
}
}  // namespace dec
}  // namespace sgq
