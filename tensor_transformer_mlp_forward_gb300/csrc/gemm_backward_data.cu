// gemm_backward_data.cu -- the backward GEMMs of the activation path, dZ and
// dX (both operands K-major).
#include "kernels.h"

namespace tpmlp {

cudaError_t launch_dgelu(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (g.epi_warps == 8) {
        if (pair) return launch_gemm<false, false, EPI_DGELU, true, 8>(m, g, grid, st);
        return launch_gemm<false, false, EPI_DGELU, false, 8>(m, g, grid, st);
    }
    if (pair) return launch_gemm<false, false, EPI_DGELU, true>(m, g, grid, st);
    return launch_gemm<false, false, EPI_DGELU, false>(m, g, grid, st);
}

cudaError_t launch_dx(const GemmMaps& m, const GemmArgs& g, int grid,
                        bool pair, cudaStream_t st) {
    if (pair && g.tile_n == 2 * BN)
        return launch_gemm<false, false, EPI_STORE, true, 4, 2 * BN>(m, g, grid, st);
    if (pair) return launch_gemm<false, false, EPI_STORE, true>(m, g, grid, st);
    return launch_gemm<false, false, EPI_STORE, false>(m, g, grid, st);
}

cudaError_t launch_dx_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                               cudaStream_t st) {
    if (pair) return launch_gemm<false, false, EPI_PARTIAL, true>(m, g, grid, st);
    return launch_gemm<false, false, EPI_PARTIAL, false>(m, g, grid, st);
}

}  // namespace tpmlp
