// gemm_backward_weight.cu -- the weight-gradient GEMMs dA = X^T dZ and
// dB = H^T dY (both operands MN-major: the token dimension is the reduction),
// whole or as fp32 partial sums over k-range splits.
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_weight_grad(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<true, true, EPI_STORE, true>(m, g, grid, st);
    return launch_gemm<true, true, EPI_STORE, false>(m, g, grid, st);
}

cudaError_t launch_weight_grad_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                                       cudaStream_t st) {
    if (pair) return launch_gemm<true, true, EPI_PARTIAL, true>(m, g, grid, st);
    return launch_gemm<true, true, EPI_PARTIAL, false>(m, g, grid, st);
}

}  // namespace tpmlp
