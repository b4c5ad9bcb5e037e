// gemm_backward_weight.cu -- the weight-gradient GEMMs dA = X^T dZ and
// dB = H^T dY (both operands MN-major: the token dimension is the reduction).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_weight_grad(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<true, true, EPI_STORE, true>(m, g, grid, st);
    return launch_gemm<true, true, EPI_STORE, false>(m, g, grid, st);
}

}  // namespace tpmlp
