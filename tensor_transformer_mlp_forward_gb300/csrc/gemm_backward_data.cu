// gemm_backward_data.cu -- the backward GEMMs of the activation path, dZ and
// dX (both operands K-major).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_dgelu(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, false, EPI_DGELU, true>(a, b, g, grid, st);
    return launch_gemm<false, false, EPI_DGELU, false>(a, b, g, grid, st);
}

cudaError_t launch_dx(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair) return launch_gemm<false, false, EPI_STORE, true>(a, b, g, grid, st);
    return launch_gemm<false, false, EPI_STORE, false>(a, b, g, grid, st);
}

}  // namespace tpmlp
