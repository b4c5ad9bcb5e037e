// gemm_forward.cu -- the forward pass's two GEMM instantiations
// (rows operand K-major, columns operand MN-major).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_column_gelu(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_BIAS_GELU, true>(a, b, g, grid, st);
    return launch_gemm<false, true, EPI_BIAS_GELU, false>(a, b, g, grid, st);
}

cudaError_t launch_row_sum(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_BIAS_RESIDUAL, true>(a, b, g, grid, st);
    return launch_gemm<false, true, EPI_BIAS_RESIDUAL, false>(a, b, g, grid, st);
}

}  // namespace tpmlp
