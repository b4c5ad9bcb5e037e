// gemm_forward.cu -- the forward pass's two GEMM instantiations
// (rows operand K-major, columns operand MN-major).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_column_gelu(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_BIAS_GELU, true>(m, g, grid, st);
    return launch_gemm<false, true, EPI_BIAS_GELU, false>(m, g, grid, st);
}

cudaError_t launch_row_sum(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_BIAS_RESIDUAL, true>(m, g, grid, st);
    return launch_gemm<false, true, EPI_BIAS_RESIDUAL, false>(m, g, grid, st);
}

cudaError_t launch_column_bias(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                               cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_BIAS, true>(m, g, grid, st);
    return launch_gemm<false, true, EPI_BIAS, false>(m, g, grid, st);
}

cudaError_t launch_row_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                               cudaStream_t st) {
    if (pair) return launch_gemm<false, true, EPI_PARTIAL, true>(m, g, grid, st);
    return launch_gemm<false, true, EPI_PARTIAL, false>(m, g, grid, st);
}

}  // namespace tpmlp
