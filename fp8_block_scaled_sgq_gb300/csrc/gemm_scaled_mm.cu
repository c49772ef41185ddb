// Instantiates the GEMM for per-channel scaling (fp8_scaled_mm): per-tensor or
// per-row A scales, per-tensor or per-column B scales, applied once in the
// epilogue; the MMAs run unscaled over the whole K range.  The block recipe
// template arguments are unused here.
#include "gemm_kernel.cuh"

namespace sgq {
namespace gemm {
sgq_status dispatch_chan(const Variant& v, const CUtensorMap* maps, const GemmArgs& a, const ExtArgs& fz, int grid,
                         cudaStream_t st) {
    if (!v.swap) return run<256, 4, false, 1, 128, 128, false, false, false, false, true>(maps, a, fz, grid, st);
    switch (v.bn) {
        case 16: return run<16, 8, true, 2, 128, 128, false, false, false, false, true>(maps, a, fz, grid, st);
        case 32: return run<32, 8, true, 2, 128, 128, false, false, false, false, true>(maps, a, fz, grid, st);
        default: return run<64, 7, true, 2, 128, 128, false, false, false, false, true>(maps, a, fz, grid, st);
    }
}
}  // namespace gemm
}  // namespace sgq
