// colsum.cu -- column sums of a bf16 matrix in fp32: the bias gradients of
// the tensor-parallel MLP block ("Megatron-LM: Tensor Model Parallel",
// Figure 3(a): db2 is the sum of dY over the tokens, since the row-parallel
// GEMM's output bias is added once after the g all-reduce) and of the
// attention block (dbo from dY, dbqkv from dQKV), and the final sum of
// per-tile column partials (db1 from the dZ GEMM's epilogue).
//
//   db[j] = sum_{r < T} G[r * n + j]
//
// HBM-bound: 2 bytes read per element.  A 2-D grid of 64-column blocks x
// row chunks (about 640 CTAs) writes one fp32 partial row per chunk; a
// second kernel adds the chunks' rows in chunk order, so the result does not
// depend on which CTA runs when.  Both are launched as programmatic
// dependents: each may be scheduled while the kernel before it finishes, so
// the second launch costs no gap, and no counter or cleared scratch word is
// needed.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kernels.h"

namespace tpmlp {
namespace {

long long cdiv_ll(long long a, long long b) { return (a + b - 1) / b; }

constexpr int kColBlock = 64;   // columns per CTA: 8 lanes x 8 bf16 (16 B each)
constexpr int kSumThreads = 256;
constexpr int kSumBatch = 8;    // 16-byte loads a thread keeps in flight
constexpr int kTargetCtas = 640;

// Partial column sums of G [T, n] over one chunk of rows.  A warp covers
// 64 columns and 4 rows per step (lanes 8j..8j+7 read row 4k+j, 16 B each),
// the CTA 32 rows per step.  Each thread issues the loads of kSumBatch steps
// before it adds any of them (rows past the chunk count as zero), so that
// 32 KiB per CTA are in flight; the adds stay in row order.  The 4 row
// phases meet by warp shuffle, the 8 warps in shared memory, in a fixed
// order.  Writes out[blockIdx.y * n + col].
__global__ void __launch_bounds__(kSumThreads)
    colsum_partial_kernel(const __nv_bfloat16* __restrict__ G, int T, int n, int rows_per_chunk,
                          float* __restrict__ out) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // G is written by the kernel before this one
    __shared__ float part[kSumThreads / 32][kColBlock];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * kColBlock + (lane & 7) * 8;
    const int r0 = blockIdx.y * rows_per_chunk;
    const int r1 = min(T, r0 + rows_per_chunk);
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    const int rt = r0 + warp * 4 + (lane >> 3);  // this thread's first row
    if (col0 + 8 <= n) {
        const __nv_bfloat16* base = G + col0;
        for (int r = rt; r < r1; r += 32 * kSumBatch) {
            // every load is issued (a row past the chunk re-reads its last
            // row) and its words are zeroed afterwards: no branch between
            // the loads
            uint4 u[kSumBatch];
#pragma unroll
            for (int k = 0; k < kSumBatch; ++k) {
                const int rk = min(r + 32 * k, r1 - 1);
                u[k] = __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(rk) * n));
            }
#pragma unroll
            for (int k = 0; k < kSumBatch; ++k) {
                const uint32_t keep = r + 32 * k < r1 ? 0xFFFFFFFFu : 0u;
                const uint32_t w[4] = {u[k].x & keep, u[k].y & keep, u[k].z & keep, u[k].w & keep};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[2 * j] += __uint_as_float(w[j] << 16);
                    acc[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
                }
            }
        }
    } else {
        for (int r = rt; r < r1; r += 32) {
            const __nv_bfloat16* row = G + static_cast<long long>(r) * n + col0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (col0 + i < n) acc[i] += __bfloat162float(row[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], 8);
        acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], 16);
    }
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) part[warp][lane * 8 + i] = acc[i];
    }
    __syncthreads();
    if (threadIdx.x < kColBlock) {
        const int col = blockIdx.x * kColBlock + threadIdx.x;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kSumThreads / 32; ++w) s += part[w][threadIdx.x];
        if (col < n) out[static_cast<long long>(blockIdx.y) * n + col] = s;
    }
}

// out[j] = sum_{i < rows} P[i * n + j].  A 256-thread CTA covers 32 columns:
// the warp g sums rows g, g + 8, g + 16, ... in order (4 loads in flight a
// thread), then thread j of warp 0 adds the 8 warps' sums in warp order.
constexpr int kRowsumCols = 32;
constexpr int kRowsumGroups = 8;

__global__ void __launch_bounds__(kRowsumCols * kRowsumGroups)
    rowsum_kernel(const float* __restrict__ P, int rows, int n, float* __restrict__ out) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // P is written by the kernel before this one
    __shared__ float part[kRowsumGroups][kRowsumCols];
    const int g = threadIdx.x / kRowsumCols, c = threadIdx.x % kRowsumCols;
    const int j = blockIdx.x * kRowsumCols + c;
    float s = 0.0f;
    if (j < n) {
#pragma unroll 4
        for (int i = g; i < rows; i += kRowsumGroups) s += __ldg(P + static_cast<long long>(i) * n + j);
    }
    part[g][c] = s;
    __syncthreads();
    if (g == 0 && j < n) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kRowsumGroups; ++w) t += part[w][c];
        out[j] = t;
    }
}

}  // namespace

int colsum_chunks(int T, int n) {
    const long long col_blocks = cdiv_ll(n, kColBlock);
    long long r = cdiv_ll(kTargetCtas, col_blocks);
    r = std::min<long long>(r, std::max<long long>(1, cdiv_ll(T, 32)));
    return static_cast<int>(std::max<long long>(1, r));
}

size_t colsum_workspace_floats(int T, int n) {
    return static_cast<size_t>(colsum_chunks(T, n)) * static_cast<size_t>(n);
}

cudaError_t launch_rowsum_f32(const float* P, int rows, int n, float* out, cudaStream_t st,
                              int* launches) {
    if (n == 0) return cudaSuccess;
    cudaError_t e = launch_dependent(rowsum_kernel,
                                     dim3(static_cast<unsigned>(cdiv_ll(n, kRowsumCols))),
                                     dim3(kRowsumCols * kRowsumGroups), 0, st, P, rows, n, out);
    if (launches) ++*launches;
    return e;
}

// T == 0 or n == 0 launches nothing and leaves db as it was.
cudaError_t launch_colsum(const __nv_bfloat16* G, int T, int n, float* db, float* partial,
                          cudaStream_t st, int* launches) {
    if (T == 0 || n == 0) return cudaSuccess;
    const int chunks = colsum_chunks(T, n);
    const int rows_per_chunk = static_cast<int>(cdiv_ll(T, chunks));
    const dim3 grid(static_cast<unsigned>(cdiv_ll(n, kColBlock)), static_cast<unsigned>(chunks));
    // one chunk: its partial row is the result
    cudaError_t e = launch_dependent(colsum_partial_kernel, grid, dim3(kSumThreads), 0, st, G, T, n,
                                     rows_per_chunk, chunks == 1 ? db : partial);
    if (launches) ++*launches;
    if (e != cudaSuccess || chunks == 1) return e;
    return launch_rowsum_f32(partial, chunks, n, db, st, launches);
}

}  // namespace tpmlp
