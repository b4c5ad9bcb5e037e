// layernorm.cu -- residual add + LayerNorm producing the MLP block's input X
// ("Megatron-DeepSpeed to ZeRO-3", seekfood.cn, section 4.3: a fused
// LayerNorm + residual kernel; "Megatron-LM: Tensor Model Parallel",
// Figure 2: layer normalization and the residual connection around the MLP).
//
// Per row of h values:
//   s = a + r ; mu = mean(s) ; var = mean((s - mu)^2) ; rstd = 1/sqrt(var+eps)
//   X = (s - mu) * rstd * gamma + beta
// and its backward pass (dres: the gradient reaching s directly):
//   xhat = (s - mu) rstd ; g = dX * gamma
//   ds = rstd (g - mean(g) - xhat mean(g xhat)) + dres
//   dgamma = sum_rows dX xhat ; dbeta = sum_rows dX
// The work is a few reads and writes per element: HBM-bound, so these are
// plain CUDA-core kernels with 16-byte accesses; statistics in fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "kernels.h"

namespace tpmlp {
namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(w[j] << 16);
        v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    return u;
}

// Sum over the block (blockDim.x a multiple of 32, at most 1024); every
// thread receives the total.  `scratch` holds 32 floats.
__device__ __forceinline__ float block_sum(float x, float* scratch) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();  // scratch may still be read by a previous call
    if (lane == 0) scratch[warp] = x;
    __syncthreads();
    float t = lane < nw ? scratch[lane] : 0.0f;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
    return t;
}

// One CTA per row; s is staged in dynamic shared memory as fp32.
__global__ void __launch_bounds__(512)
    ln_forward_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ r,
                      const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ beta,
                      int h, float eps, __nv_bfloat16* __restrict__ X,
                      __nv_bfloat16* __restrict__ s_out, float* __restrict__ mean,
                      float* __restrict__ rstd) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    extern __shared__ float srow[];
    __shared__ float scratch[32];
    const long long base = static_cast<long long>(blockIdx.x) * h;
    const int nvec = h >> 3;
    float sum = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float x[8], y[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + base) + v), x);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(r + base) + v), y);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x[j] += y[j];
            sum += x[j];
            srow[8 * v + j] = x[j];
        }
        if (s_out != nullptr) reinterpret_cast<uint4*>(s_out + base)[v] = f32_to_bf16x8(x);
    }
    const float mu = block_sum(sum, scratch) / static_cast<float>(h);
    float sq = 0.0f;
    for (int i = threadIdx.x; i < h; i += blockDim.x) {
        const float c = srow[i] - mu;
        sq += c * c;
    }
    const float rs = rsqrtf(block_sum(sq, scratch) / static_cast<float>(h) + eps);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float g[8], b[8], o[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(gamma) + v), g);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(beta) + v), b);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] = (srow[8 * v + j] - mu) * rs * g[j] + b[j];
        reinterpret_cast<uint4*>(X + base)[v] = f32_to_bf16x8(o);
    }
    if (threadIdx.x == 0) {
        mean[blockIdx.x] = mu;
        rstd[blockIdx.x] = rs;
    }
}

// One CTA per row: ds = rstd (g - mean(g) - xhat mean(g xhat)) + dres.  The
// row is read twice (the second pass hits L1/L2).
__global__ void __launch_bounds__(512)
    ln_backward_rows_kernel(const __nv_bfloat16* __restrict__ dX,
                            const __nv_bfloat16* __restrict__ dres,
                            const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ r,
                            const __nv_bfloat16* __restrict__ gamma, const float* __restrict__ mean,
                            const float* __restrict__ rstd, int h, __nv_bfloat16* __restrict__ ds) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    __shared__ float scratch[32];
    const long long base = static_cast<long long>(blockIdx.x) * h;
    const int nvec = h >> 3;
    const float mu = mean[blockIdx.x], rs = rstd[blockIdx.x];
    float mg = 0.0f, mgx = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float x[8], y[8], d[8], g[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + base) + v), x);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(r + base) + v), y);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(dX + base) + v), d);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(gamma) + v), g);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float gj = d[j] * g[j];
            mg += gj;
            mgx += gj * (x[j] + y[j] - mu) * rs;
        }
    }
    mg = block_sum(mg, scratch) / static_cast<float>(h);
    mgx = block_sum(mgx, scratch) / static_cast<float>(h);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        float x[8], y[8], d[8], g[8], e[8], o[8];
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + base) + v), x);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(r + base) + v), y);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(dX + base) + v), d);
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(gamma) + v), g);
        if (dres != nullptr) {
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(dres + base) + v), e);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float xh = (x[j] + y[j] - mu) * rs;
            o[j] = rs * (d[j] * g[j] - mg - xh * mgx) + e[j];
        }
        reinterpret_cast<uint4*>(ds + base)[v] = f32_to_bf16x8(o);
    }
}

// Column partial sums of dX * xhat and dX over one chunk of rows (64-column
// blocks; a warp takes 4 rows x 64 columns per step, 16 B per lane; the four
// row phases meet by shuffle and the 8 warps in shared memory, in a fixed
// order).  Writes pg/pb[blockIdx.y * h + col].
__global__ void __launch_bounds__(256)
    ln_param_grad_kernel(const __nv_bfloat16* __restrict__ dX, const __nv_bfloat16* __restrict__ a,
                         const __nv_bfloat16* __restrict__ r, const float* __restrict__ mean,
                         const float* __restrict__ rstd, int T, int h, int rows_per_chunk,
                         float* __restrict__ pg, float* __restrict__ pb) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    __shared__ float part[2][8][64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 64 + (lane & 7) * 8;
    const int r0 = blockIdx.y * rows_per_chunk;
    const int r1 = min(T, r0 + rows_per_chunk);
    float sg[8], sb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sg[i] = sb[i] = 0.0f;
    if (col0 < h) {
        for (int row = r0 + warp * 4 + (lane >> 3); row < r1; row += 32) {
            const long long off = static_cast<long long>(row) * h + col0;
            float x[8], y[8], d[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + off)), x);
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(r + off)), y);
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(dX + off)), d);
            const float mu = __ldg(mean + row), rs = __ldg(rstd + row);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                sg[i] += d[i] * (x[i] + y[i] - mu) * rs;
                sb[i] += d[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        sg[i] += __shfl_xor_sync(0xFFFFFFFFu, sg[i], 8);
        sg[i] += __shfl_xor_sync(0xFFFFFFFFu, sg[i], 16);
        sb[i] += __shfl_xor_sync(0xFFFFFFFFu, sb[i], 8);
        sb[i] += __shfl_xor_sync(0xFFFFFFFFu, sb[i], 16);
    }
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            part[0][warp][lane * 8 + i] = sg[i];
            part[1][warp][lane * 8 + i] = sb[i];
        }
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int which = threadIdx.x >> 6, c = threadIdx.x & 63;
        const int col = blockIdx.x * 64 + c;
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += part[which][w][c];
        if (col < h) (which == 0 ? pg : pb)[static_cast<long long>(blockIdx.y) * h + col] = t;
    }
}

// ------------------------------------------------ register-resident rows
// For h <= 8 * 8 * LN_THREADS each thread holds VPT vectors of 8 values of
// the row (vector k of thread t: columns 8 (t + k LN_THREADS) .. +7), so all
// of a row's loads are in flight at once.

constexpr int LN_THREADS = 512;

template <int VPT>
__global__ void __launch_bounds__(LN_THREADS)
    ln_forward_reg_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ r,
                          const __nv_bfloat16* __restrict__ gamma,
                          const __nv_bfloat16* __restrict__ beta, int h, float eps,
                          __nv_bfloat16* __restrict__ X, __nv_bfloat16* __restrict__ s_out,
                          float* __restrict__ mean, float* __restrict__ rstd) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    __shared__ float scratch[32];
    const long long base = static_cast<long long>(blockIdx.x) * h;
    const int nvec = h >> 3;
    float v[VPT][8];
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int vi = threadIdx.x + k * LN_THREADS;
        if (vi < nvec) {
            float y[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(a + base) + vi), v[k]);
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(r + base) + vi), y);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[k][j] += y[j];
                sum += v[k][j];
            }
            if (s_out != nullptr) reinterpret_cast<uint4*>(s_out + base)[vi] = f32_to_bf16x8(v[k]);
        }
    }
    const float mu = block_sum(sum, scratch) / static_cast<float>(h);
    float sq = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        if (threadIdx.x + k * LN_THREADS < nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j) sq += (v[k][j] - mu) * (v[k][j] - mu);
        }
    }
    const float rs = rsqrtf(block_sum(sq, scratch) / static_cast<float>(h) + eps);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int vi = threadIdx.x + k * LN_THREADS;
        if (vi < nvec) {
            float g[8], b[8], o[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(gamma) + vi), g);
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(beta) + vi), b);
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = (v[k][j] - mu) * rs * g[j] + b[j];
            reinterpret_cast<uint4*>(X + base)[vi] = f32_to_bf16x8(o);
        }
    }
    if (threadIdx.x == 0) {
        mean[blockIdx.x] = mu;
        rstd[blockIdx.x] = rs;
    }
}

// out[j] = sum_{i < rows} P[i * n + j], in row order.
__global__ void __launch_bounds__(256)
    ln_rowsum_kernel(const float* __restrict__ P, int rows, int n, float* __restrict__ out) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    float s = 0.0f;
    for (int i = 0; i < rows; ++i) s += P[static_cast<long long>(i) * n + j];
    out[j] = s;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

int ln_threads(int h) {
    const int nvec = h >> 3;
    int t = 32;
    while (t < nvec && t < 512) t <<= 1;
    return t;
}

// Register-resident forward for h <= 8 * 8 * LN_THREADS = 32768.
constexpr int LN_REG_MAX_H = 8 * 8 * LN_THREADS;

int ln_vpt(int h) { return ceil_div(h >> 3, LN_THREADS); }

template <typename Fn>
cudaError_t dispatch_vpt(int vpt, Fn&& fn) {
    switch (vpt) {
        case 1: return fn(std::integral_constant<int, 1>{});
        case 2: return fn(std::integral_constant<int, 2>{});
        case 3: return fn(std::integral_constant<int, 3>{});
        case 4: return fn(std::integral_constant<int, 4>{});
        case 5: return fn(std::integral_constant<int, 5>{});
        case 6: return fn(std::integral_constant<int, 6>{});
        case 7: return fn(std::integral_constant<int, 7>{});
        default: return fn(std::integral_constant<int, 8>{});
    }
}

}  // namespace

int ln_param_chunks(int T, int h) {
    const long long col_blocks = (h + 63) / 64;
    long long c = (640 + col_blocks - 1) / col_blocks;
    const long long most = (T + 31) / 32;
    if (c > most) c = most;
    return static_cast<int>(c < 1 ? 1 : c);
}

cudaError_t launch_ln_forward(const __nv_bfloat16* a, const __nv_bfloat16* r,
                              const __nv_bfloat16* gamma, const __nv_bfloat16* beta, int T, int h,
                              float eps, __nv_bfloat16* X, __nv_bfloat16* s, float* mean,
                              float* rstd, cudaStream_t st, int* launches) {
    ++*launches;
    if (h <= LN_REG_MAX_H) {
        return dispatch_vpt(ln_vpt(h), [&](auto vpt) {
            ln_forward_reg_kernel<decltype(vpt)::value>
                <<<T, LN_THREADS, 0, st>>>(a, r, gamma, beta, h, eps, X, s, mean, rstd);
            return cudaGetLastError();
        });
    }
    const size_t smem = sizeof(float) * static_cast<size_t>(h);
    cudaError_t e = cudaFuncSetAttribute(ln_forward_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    ln_forward_kernel<<<T, ln_threads(h), smem, st>>>(a, r, gamma, beta, h, eps, X, s, mean, rstd);
    return cudaGetLastError();
}

cudaError_t launch_ln_backward(const __nv_bfloat16* dX, const __nv_bfloat16* dres,
                               const __nv_bfloat16* a, const __nv_bfloat16* r,
                               const __nv_bfloat16* gamma, const float* mean, const float* rstd,
                               int T, int h, __nv_bfloat16* ds, float* dgamma, float* dbeta,
                               float* partial, cudaStream_t st, int* launches) {
    // The row kernel reads each row twice (the second pass hits L1/L2): its
    // small register footprint keeps several rows in flight per SM, which
    // measured faster than holding the row in registers at one row per SM.
    ln_backward_rows_kernel<<<T, ln_threads(h), 0, st>>>(dX, dres, a, r, gamma, mean, rstd, h, ds);
    ++*launches;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int chunks = ln_param_chunks(T, h);
    const int rows_per_chunk = ceil_div(T, chunks);
    float* pg = partial;
    float* pb = partial + static_cast<size_t>(chunks) * h;
    ln_param_grad_kernel<<<dim3(ceil_div(h, 64), chunks), 256, 0, st>>>(dX, a, r, mean, rstd, T, h,
                                                                        rows_per_chunk, pg, pb);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ln_rowsum_kernel<<<ceil_div(h, 256), 256, 0, st>>>(pg, chunks, h, dgamma);
    ln_rowsum_kernel<<<ceil_div(h, 256), 256, 0, st>>>(pb, chunks, h, dbeta);
    *launches += 2;
    return cudaGetLastError();
}

}  // namespace tpmlp
