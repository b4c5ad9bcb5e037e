// kernels.h -- host-side launchers of the library's kernels (one per GEMM
// variant and reduction), shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm.cuh"

#include <utility>

namespace tpmlp {

// Whether the library's kernels are launched as programmatic dependents of
// the kernel before them on the stream (tpmlp_set_dependent_launch).
bool dependent_launch();

// Launches `kern` with the programmatic stream serialization attribute when
// dependent launch is on, else as a plain launch.  Every kernel launched
// this way calls pdl_wait() before its first global memory access, so it may
// be scheduled (and run its set-up) while the previous kernel finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (dependent_launch()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// The four tensor maps of one GEMM: operands A and B, output o0 (and o1, the
// second output of the bias + GeLU epilogue; a copy of o0 otherwise).
struct GemmMaps {
    CUtensorMap a, b, o0, o1;
};

// Each launcher runs the CTA-pair kernel when `pair` is set (grid even,
// launched as clusters of 2), else the single-CTA kernel; where the
// epilogue has an eight-warp form, g.epi_warps (4 or 8) picks it.
// A K-major, B MN-major: the forward GEMMs.
cudaError_t launch_column_gelu(const GemmMaps& m, const GemmArgs& g,
                               int grid, bool pair, cudaStream_t st);
cudaError_t launch_row_sum(const GemmMaps& m, const GemmArgs& g,
                           int grid, bool pair, cudaStream_t st);
// Column GEMM with + bias only (the attention block's Q/K/V projection).
cudaError_t launch_column_bias(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                               cudaStream_t st);
// The same two GEMMs with a split reduction: fp32 partials per k-range split.
cudaError_t launch_row_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                               cudaStream_t st);
// A K-major, B K-major: dZ and dX.
cudaError_t launch_dgelu(const GemmMaps& m, const GemmArgs& g, int grid,
                         bool pair, cudaStream_t st);
cudaError_t launch_dx(const GemmMaps& m, const GemmArgs& g, int grid,
                      bool pair, cudaStream_t st);
cudaError_t launch_dx_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                              cudaStream_t st);
// A MN-major, B MN-major: the weight gradients read from X, dZ, H and dY in
// place (their K-major form from the transposes runs launch_dx).
cudaError_t launch_weight_grad(const GemmMaps& m, const GemmArgs& g,
                               int grid, bool pair, cudaStream_t st);
// The same with a split reduction: fp32 partials per k-range split.
cudaError_t launch_weight_grad_partial(const GemmMaps& m, const GemmArgs& g, int grid, bool pair,
                                       cudaStream_t st);

// out[c * ld_out + r] = in[r * cols + c], bf16, with each output row zeroed
// from `rows` to the next multiple of 8 (transpose.cu).  cols % 8 == 0,
// ld_out % 8 == 0, ld_out >= rows rounded up to 8, 16-byte aligned pointers.
cudaError_t launch_transpose(const __nv_bfloat16* in, int rows, int cols, __nv_bfloat16* out,
                             int ld_out, cudaStream_t st, int* launches);

// Column sums db[j] = sum_{r < T} G[r * n + j] of a bf16 [T, n] matrix in
// fp32 (colsum.cu).  With colsum_chunks(T, n) > 1 row chunks the chunks'
// partial rows go to `partial` (colsum_workspace_floats(T, n) floats,
// 16-byte aligned, any contents) and a second kernel adds them in chunk
// order; with one chunk db is written directly.  T == 0 or n == 0 launches
// nothing.
int colsum_chunks(int T, int n);
size_t colsum_workspace_floats(int T, int n);
cudaError_t launch_colsum(const __nv_bfloat16* G, int T, int n, float* db, float* partial,
                          cudaStream_t st, int* launches);
// out[j] = sum_{i < rows} P[i * n + j] for an fp32 [rows, n] matrix (colsum.cu).
cudaError_t launch_rowsum_f32(const float* P, int rows, int n, float* out, cudaStream_t st,
                              int* launches);

// Residual add + LayerNorm (layernorm.cu).  `launches` is incremented per
// kernel launched.
cudaError_t launch_ln_forward(const __nv_bfloat16* a, const __nv_bfloat16* r,
                              const __nv_bfloat16* gamma, const __nv_bfloat16* beta, int T, int h,
                              float eps, __nv_bfloat16* X, __nv_bfloat16* s, float* mean,
                              float* rstd, cudaStream_t st, int* launches);
cudaError_t launch_ln_backward(const __nv_bfloat16* dX, const __nv_bfloat16* dres,
                               const __nv_bfloat16* a, const __nv_bfloat16* r,
                               const __nv_bfloat16* gamma, const float* mean, const float* rstd,
                               int T, int h, __nv_bfloat16* ds, float* dgamma, float* dbeta,
                               float* partial, cudaStream_t st, int* launches);
// Row chunks of the dgamma / dbeta partial sums (partial = 2 * chunks * h floats).
int ln_param_chunks(int T, int h);

// Causal attention of every (sequence, head) (attention.cu).  Head dims
// d in {64, 96, 128, 160}.  QKV [T, 3h] is read through 3-D tensor maps
// {3h, s, nb} with 64 x 128-row (qkv128) or 64 x 64-row (qkv64) boxes, dO
// [T, h] likewise; T = nb * s.
struct AttnParams {
    int nb, s, h, nh;
    __nv_bfloat16* O;            // forward: output [T, h]
    float* lse;                  // forward: log2-domain log-sum-exp [nh, T]
    const __nv_bfloat16* O_in;   // backward: the forward's O
    const __nv_bfloat16* dO;     // backward: gradient at O [T, h]
    const float* lse_in;         // backward: the forward's lse
    float* delta_out;            // backward: rowsum(dO * O) scratch [nh, T]
    __nv_bfloat16* dqkv;         // backward: output [T, 3h]
    unsigned int* work;          // item counters of the persistent kernels (forward 1 word,
                                 // backward 2), caller memory, cleared by the launcher
    int* status;
};
cudaError_t launch_attn_forward(const CUtensorMap& tm_qkv128, const CUtensorMap& tm_qkv64, int d,
                                const AttnParams& p, cudaStream_t st, int* launches);
cudaError_t launch_attn_backward(const CUtensorMap& tm_qkv128, const CUtensorMap& tm_qkv64,
                                 const CUtensorMap& tm_do128, const CUtensorMap& tm_do64, int d,
                                 const AttnParams& p, cudaStream_t st, int* launches);

// `grid` is the number of work units wanted (CTAs, or CTA pairs when PAIR).
// With static units it is clipped to what can be resident at once, so the
// persistent loop never waits for a second wave of CTAs; with dynamic units
// (g.dynamic_tiles) it is one CTA (pair) per unit and the running ones take
// over the launches of the others.
template <bool A_MN, bool B_MN, int EPI, bool PAIR, int EW = 4, int TN = BN>
cudaError_t launch_gemm(const GemmMaps& m, const GemmArgs& g, int grid,
                        cudaStream_t st) {
    auto kern = tcgen05_gemm_kernel<A_MN, B_MN, EPI, PAIR, EW, TN>;
    constexpr int smem = Geometry<PAIR, EW, TN>::SMEM_BYTES;
    constexpr int threads = Geometry<PAIR, EW, TN>::THREADS;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    if (PAIR) {
        static int resident_clusters = 0;  // same for every device of this build's target
        if (resident_clusters == 0) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2 * static_cast<unsigned>(grid));
            q.blockDim = dim3(threads);
            q.dynamicSmemBytes = smem;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 2;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &q);
            if (e != cudaSuccess) return e;
            resident_clusters = n > 0 ? n : 1;
        }
        // persistent: no more pairs than can be resident; with dynamic units
        // one pair per unit, the ones that do not fit wait to be cancelled
        grid = 2 * (g.dynamic_tiles || grid < resident_clusters ? grid : resident_clusters);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (PAIR) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (g.dependent_launch) {  // may begin before the previous kernel ends (pdl_wait inside)
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, m.a, m.b, m.o0, m.o1, g);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tpmlp
