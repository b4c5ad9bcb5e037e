// gemm_backward_data.cu -- the backward GEMMs of the activation path, dZ and
// dX (both operands K-major).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_dgelu(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                         cudaStream_t st) {
    return launch_gemm<false, false, EPI_DGELU>(a, b, g, grid, st);
}

cudaError_t launch_dx(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                      cudaStream_t st) {
    return launch_gemm<false, false, EPI_STORE>(a, b, g, grid, st);
}

}  // namespace tpmlp
