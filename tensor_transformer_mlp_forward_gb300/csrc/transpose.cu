// transpose.cu -- bf16 matrix transpose: the layout change that lets the
// weight-gradient GEMMs dA_i = X^T dZ_i and dB_i = H_i^T dY read both operands
// K-major ("Megatron-LM: Tensor Model Parallel", Figure 3(a): the backward
// pass of the column- and row-parallel GEMMs takes X, dZ_i, H_i and dY with
// the token dimension as the reduction).
//
//   out[c * ld_out + r] = in[r * cols + c]      r < rows, c < cols
//
// and out[c * ld_out + r] = 0 for rows <= r < rows rounded up to a multiple of
// 8, so that every output row's written part ends on a 16-byte boundary;
// nothing further right is touched.
//
// HBM-bound: 2 bytes read and 2 written per element, no arithmetic.  A
// 256-thread CTA moves one 64 x 64 tile through 8 KiB of shared memory:
//  - coalesced 16-byte loads of two adjacent input rows r, r + 1;
//  - element pairs (in[r][c], in[r+1][c]) packed into the 32-bit word r / 2
//    of output row c;
//  - the word index XOR-swizzled by 4 * ((c / 8) % 8), which makes both the
//    word stores (8 columns x 4 row pairs per warp) and the 16-byte reads
//    (4 output rows x 128 bytes per warp) bank-conflict free;
//  - coalesced 16-byte stores.
// Eight CTAs fit an SM: 64 KiB of loads in flight per SM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace tpmlp {
namespace {

constexpr int kTile = 64;
constexpr int kTransposeThreads = 256;

__global__ void __launch_bounds__(kTransposeThreads)
    transpose_bf16_kernel(const uint16_t* __restrict__ in, int rows, int cols,
                          uint16_t* __restrict__ out, int ld_out, int col_tiles) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // `in` comes from the kernel before this one
    __shared__ __align__(16) uint32_t sT[kTile * kTile / 2];  // [output row c][word]
    const int tid = threadIdx.x;
    const int tr = static_cast<int>(blockIdx.x / col_tiles);
    const int r0 = tr * kTile;
    const int c0 = static_cast<int>(blockIdx.x - static_cast<unsigned>(tr) * col_tiles) * kTile;

    // ---- load: rows r0 + 2 rp and r0 + 2 rp + 1, columns c0 + 8 cc .. + 7
    {
        const int rp = tid >> 3, cc = tid & 7;
        const int r = r0 + 2 * rp, c = c0 + 8 * cc;
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (c < cols) {
            const uint16_t* p = in + static_cast<long long>(r) * cols + c;
            if (r < rows) a = __ldg(reinterpret_cast<const uint4*>(p));
            if (r + 1 < rows) b = __ldg(reinterpret_cast<const uint4*>(p + cols));
        }
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
        const int word = rp ^ (4 * cc);  // output rows 8 cc .. 8 cc + 7 share the swizzle
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t lo = (k & 1) ? (wa[k >> 1] >> 16) : (wa[k >> 1] & 0xFFFFu);
            const uint32_t hi = (k & 1) ? (wb[k >> 1] & 0xFFFF0000u) : (wb[k >> 1] << 16);
            sT[(8 * cc + k) * (kTile / 2) + word] = lo | hi;
        }
    }
    __syncthreads();
    // ---- store: output row c0 + c, columns r0 + 8 q .. + 7
    const int rows8 = (rows + 7) & ~7;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = tid + i * kTransposeThreads;
        const int c = idx >> 3, q = idx & 7;
        const int oc = c0 + c, orow = r0 + 8 * q;
        const uint4 v = *reinterpret_cast<const uint4*>(
            &sT[c * (kTile / 2) + 4 * (q ^ ((c >> 3) & 7))]);
        if (oc < cols && orow < rows8)
            *reinterpret_cast<uint4*>(out + static_cast<long long>(oc) * ld_out + orow) = v;
    }
}

}  // namespace

cudaError_t launch_transpose(const __nv_bfloat16* in, int rows, int cols, __nv_bfloat16* out,
                             int ld_out, cudaStream_t st, int* launches) {
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int col_tiles = (cols + kTile - 1) / kTile;
    const long long tiles = static_cast<long long>((rows + kTile - 1) / kTile) * col_tiles;
    if (tiles > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    cudaError_t e = launch_dependent(transpose_bf16_kernel, dim3(static_cast<unsigned>(tiles)),
                                     dim3(kTransposeThreads), 0, st,
                                     reinterpret_cast<const uint16_t*>(in), rows, cols,
                                     reinterpret_cast<uint16_t*>(out), ld_out, col_tiles);
    if (launches) ++*launches;
    return e;
}

}  // namespace tpmlp
