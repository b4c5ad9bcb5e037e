// kernels.h -- host-side launchers of the library's kernels (one per GEMM
// variant and reduction), shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm.cuh"

namespace tpmlp {

// A K-major, B MN-major: the forward GEMMs.
cudaError_t launch_column_gelu(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g,
                               int grid, cudaStream_t st);
cudaError_t launch_row_sum(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g,
                           int grid, cudaStream_t st);
// A K-major, B K-major: dZ and dX.
cudaError_t launch_dgelu(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                         cudaStream_t st);
cudaError_t launch_dx(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                      cudaStream_t st);
// A MN-major, B MN-major: the weight gradients.
cudaError_t launch_weight_grad(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g,
                               int grid, cudaStream_t st);

template <bool A_MN, bool B_MN, int EPI>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int grid,
                        cudaStream_t st) {
    auto kern = tcgen05_gemm_kernel<A_MN, B_MN, EPI>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(a, b, g);
    return cudaGetLastError();
}

}  // namespace tpmlp
