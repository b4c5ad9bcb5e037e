// philox.cuh -- the Philox4x32 counter-based generator with 10 rounds (J. K.
// Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel Random Numbers:
// As Easy as 1, 2, 3", SC'11), and the dropout keep decision built on it.
//
// Dropout before the residual add is outside the model-parallel region, so
// every shard must draw the same pattern ("Megatron-LM: Tensor Model
// Parallel", section "Hybrid MP + DP"): the keep bit of element e of the
// [T, h] output depends only on (seed, offset + e):
//   g = offset + e ; w = Philox(counter = (lo g/4, hi g/4, 0, 0),
//                               key = (lo seed, hi seed))[g % 4]
//   keep = w >= threshold      (threshold = floor(p * 2^32))
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tpmlp {

// One block: 10 rounds of the multiply-hi/lo bijection (multiplier
// 0xD2511F53 on word 0, 0xCD9E8D57 on word 2); between rounds the key
// advances by the Weyl increments 0x9E3779B9, 0xBB67AE85.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Keep bits of the four elements g0 .. g0+3 (g0 a multiple of 4), bit j for
// element g0 + j.
__device__ __forceinline__ uint32_t dropout_keep4(uint64_t seed, uint64_t g0, uint32_t threshold) {
    const uint64_t blk = g0 >> 2;
    const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(blk),
                                             static_cast<uint32_t>(blk >> 32), 0u, 0u),
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    return (w.x >= threshold ? 1u : 0u) | (w.y >= threshold ? 2u : 0u) |
           (w.z >= threshold ? 4u : 0u) | (w.w >= threshold ? 8u : 0u);
}

// Dropout parameters of the bias-dropout-add epilogue.
struct Dropout {
    uint32_t threshold;  // floor(p * 2^32); 0 = no dropout
    float scale;         // 1 / (1 - p)
    uint64_t seed;
    uint64_t offset;     // counter of element (0, 0); a multiple of 4
};

}  // namespace tpmlp
