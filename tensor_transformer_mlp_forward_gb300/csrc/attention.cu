// attention.cu -- the core of the head-parallel self-attention block on
// tcgen05 tensor cores: causal softmax attention of every (sequence, head),
// forward and backward.
//
// "Megatron-LM: Tensor Model Parallel" (charles2530.github.io), section
// "Attention: split Q/K/V by head" (Figure 3b): the Q, K and V projections
// are split by columns so that each rank owns a group of heads, and each
// head's scores, softmax and value sum are computed where the head lives.
// On one GPU the heads of every shard are work items of the same kernels;
// the shard count only decides which rank a head would belong to and
// changes nothing here.
//
// Layout: QKV [T, 3h] bf16 (row = token n*s + pos; columns [Q | K | V], head
// j at columns j*d .. j*d+d-1 of each part), O and dO [T, h], dQKV [T, 3h],
// lse and delta fp32 [nh, T].  Scores are scaled by 1/sqrt(d) and causal
// (a token sees itself and the earlier tokens of its own sequence).
//
//   S = Q_j K_j^T / sqrt(d) (masked) ; P = softmax_rows(S) ; O_j = P V_j
//   backward: dV = P^T dO ; dP = dO V^T ; dS = P * (dP - delta),
//             delta = rowsum(dO * O) ; dQ = dS K / sqrt(d) ; dK = dS^T Q / sqrt(d)
//
// The softmax runs in the log2 domain: with c = log2(e)/sqrt(d) each score is
// taken as u = c * (q . k), P = 2^(u - m) / l, and lse = m + log2(l) is saved
// per (head, token) so that the backward pass rebuilds P = 2^(u - lse) without
// a second normalisation pass.
//
// Kernels (softmax warps own one query or key row per thread and TMEM lane; a
// producer warp issues the TMA loads; one thread of the MMA warp allocates
// TMEM and issues every MMA).  The three tensor-core kernels are persistent:
// one CTA per SM takes work items in turn from an atomic counter, heaviest
// first, so that one item's loads and read-out overlap its neighbours' MMAs.
//   attn_fwd_kernel     items: pairs of 128-query tiles of a (sequence, head);
//                       two softmax warpgroups in ping-pong; S and the output
//                       O of each tile in TMEM; P written back into TMEM over
//                       S and used there as the A operand of P V.
//   attn_delta_kernel   delta = rowsum(dO * O) per (token, head).
//   attn_bwd_dq_kernel  items: (128 queries, head, sequence); 64-key tiles:
//                       S and dP in TMEM (double-buffered), dS written back
//                       over S and used there as the A operand of dS K, dQ
//                       accumulated in TMEM.
//   attn_bwd_dkdv_kernel items: (128 keys, head, sequence); 64-query tiles:
//                       S^T and dP^T in TMEM, P^T and dS^T written back over
//                       them and used there as the A operands of P^T dO and
//                       dS^T Q, dV and dK accumulated in TMEM.
// Keeping P, dS, P^T and dS^T in tensor memory keeps shared-memory traffic
// (K, V, Q, dO operands and the TMA writes) within what shared memory
// delivers per clock.
// dQ and dK/dV are separate kernels so that every gradient is written once,
// in a fixed summation order, with no atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace tpmlp {
namespace {

constexpr int kAttnThreads = 192;
constexpr int kRowBytes = 128;  // one 64-column bf16 box row (the swizzle width)

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 values in one 64-bit register, for the paired fp32 instructions
// (one issue slot for two FMAs or two adds).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of UMMA k-step kk (16 elements) inside a K-major operand tile
// of R rows stored as 64-column boxes (R x 128 B each): box kk/4, 32 B a step.
template <int R>
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
    return static_cast<uint32_t>((kk >> 2) * (R * kRowBytes) + (kk & 3) * 32);
}

// Byte offset of UMMA k-step kk of an MN-major operand whose K runs along the
// box rows: 16 rows of 128 B.
__device__ __forceinline__ uint32_t mnmajor_step(int kk) {
    return static_cast<uint32_t>(kk * 16 * kRowBytes);
}

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

// Stores 32 consecutive 32-bit TMEM columns of this thread's lane (same
// lane quadrant rule as tmem_ld32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16,"
        " %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 x bf16 -> f32: the A operand (128
// rows = TMEM lanes, 16 k values packed two bf16 to a 32-bit column, low
// half first) is read from tensor memory.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
        " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// tcgen05 MMA chain D (+)= A B^T with A in tensor memory (k-step kk reads the
// 8 columns a_tmem + 8 kk) and B MN-major along d in shared memory (the value
// or query/key tile as the N operand, N = d): the N extent is issued as a
// multiple of 64 (whole swizzle atoms, `box_bytes` apart) plus a 32-wide
// tail, so that no MMA spans part of an atom.  The tail (d % 64 == 32) goes
// to columns d_tail (d_tmem + the whole atoms' width unless given).
template <int D, int KSTEPS>
__device__ __forceinline__ void mma_ts_n_is_d(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t box_bytes, bool accumulate_first,
                                              uint32_t d_tail = 0xFFFFFFFFu) {
    constexpr int N1 = (D / 64) * 64;
    constexpr int N2 = D - N1;
    constexpr uint32_t id1 = idesc_bf16_f32(128, N1 > 0 ? N1 : 64, false, true);
    constexpr uint32_t id2 = idesc_bf16_f32(128, N2 > 0 ? N2 : 32, false, true);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint32_t acc = (accumulate_first || kk > 0) ? 1u : 0u;
        const uint64_t bd = desc_add(b_desc, mnmajor_step(kk));
        if constexpr (N1 > 0) tc_mma_f16_ts(d_tmem, a_tmem + 8 * kk, bd, id1, acc);
        if constexpr (N2 > 0)
            tc_mma_f16_ts(d_tail == 0xFFFFFFFFu ? d_tmem + N1 : d_tail, a_tmem + 8 * kk,
                          desc_add(bd, (N1 / 64) * box_bytes), id2, acc);
    }
}

// ---------------------------------------------------------------- forward

struct AttnArgs {
    int nb, s, h, nh;
    long long T;
    int q_tiles;     // work tiles along the sequence (forward: pairs of 128-row tiles)
    unsigned int* work;  // this launch's item counter, zero at launch (caller memory)
    float scale2;    // log2(e) / sqrt(d)
    float scale;     // 1 / sqrt(d)
    __nv_bfloat16* O;        // forward output [T, h]
    float* lse;              // forward output [nh, T]
    const float* lse_in;     // backward input [nh, T]
    const float* delta;      // backward input [nh, T]
    __nv_bfloat16* dqkv;     // backward output [T, 3h]
    int* status;
};

// The forward CTA owns two adjacent 128-query tiles of one (sequence, head),
// A = rows q0..q0+127 and B = q0+128..q0+255, which share every K/V tile.
// Each has its own softmax warpgroup (A: warps 0-3, B: warps 4-7) and its own
// S and O accumulators in TMEM.  P goes back into TMEM, packed bf16 over the
// first columns of S, and is the A operand of P V from there.  The MMA warp
// alternates between the tiles (ping-pong): while warpgroup A turns S_A into
// P_A, the tensor cores run B's P V and next S, and the other way round.
// Key tiles are 128 keys for d <= 128 and 64 keys for d = 160, whose two
// output accumulators (2 x 160 columns) leave room for only 64 columns of S
// per tile.
constexpr int kFwdThreads = 320;  // 8 softmax warps, producer, MMA
constexpr float kRescaleLog2 = 8.0f;  // keep a stale row max while it is within 2^8

template <int D>
struct FwdCfg {
    static constexpr int NB = (D + 63) / 64;            // 64-column boxes per row
    static constexpr int BKV = D <= 128 ? 128 : 64;     // keys per K/V tile
    static constexpr int QTILE = NB * 128 * kRowBytes;  // 128 query rows x D (box-padded)
    static constexpr int KVTILE = NB * BKV * kRowBytes;
    static constexpr int FIXED = 2 * QTILE;
    static constexpr int STAGES_FIT = (225 * 1024 - FIXED) / KVTILE;
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int SMEM = 1024 + FIXED + STAGES * KVTILE + 256;
    // TMEM columns of tile x.  d <= 128: S at 256 x, O at 256 x + 128 (its
    // 32-wide tail, d = 96, right after).  d = 160: S at 64 x, the 128-column
    // part of O at 128 + 128 x and its 32-column tail at 384 + 32 x, so that
    // every N >= 128 accumulator part starts on a multiple of 128.
    static constexpr uint32_t s_col(int x) { return D <= 128 ? 256u * x : 64u * x; }
    static constexpr uint32_t o_col(int x) { return D <= 128 ? 256u * x + 128u : 128u + 128u * x; }
    static constexpr uint32_t o_tail(int x) {
        return D <= 128 ? o_col(x) + (D / 64) * 64 : 384u + 32u * x;
    }
    // column of 32-column chunk c of O_x
    static constexpr uint32_t o_chunk(int x, int c) {
        return c < (D / 64) * 2 ? o_col(x) + 32u * c : o_tail(x) + 32u * (c - (D / 64) * 2);
    }
};

// Work counters of the persistent kernels: CTAs take work items one at a
// time from the launch's counter (atomicAdd) until it runs past the last
// item.  The counter is a word of the caller's workspace that the launcher
// clears on the stream first, so no two calls share one.

// Work items of the forward kernel: (pair of 128-query tiles, sequence,
// head), heaviest (most key tiles) first.

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q128,  // QKV, 128-row boxes (Q)
                    const __grid_constant__ CUtensorMap tm_kv,    // QKV, BKV-row boxes (K, V)
                    const AttnArgs a) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    using C = FwdCfg<D>;
    constexpr int S = C::STAGES;
    constexpr int BKV = C::BKV;
    constexpr int SCH = BKV / 32;  // 32-key chunks of S per key tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sQ = smem;                   // Q_A, Q_B
    uint8_t* ring = smem + 2 * C::QTILE;  // K_0, V_0, K_1, V_1, ... of every item in turn
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + S * C::KVTILE);
    uint64_t* q_full = bars;              // the item's Q tiles have landed
    uint64_t* q_empty = bars + 1;         // the item's last S MMAs have read them
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = kv_full + S;
    uint64_t* s_full = kv_empty + S;      // [tile]
    uint64_t* p_full = s_full + 2;        // [tile]
    uint64_t* pv_done = p_full + 2;       // [tile]
    uint64_t* o_free = pv_done + 2;       // [tile] the softmax warps have read O_x out
    uint64_t* item_full = o_free + 2;     // [2]
    uint64_t* item_empty = item_full + 2; // [2]
    uint64_t* drain = item_empty + 2;
    int* items = reinterpret_cast<int*>(drain + 1);  // [2]
    uint32_t* misc = reinterpret_cast<uint32_t*>(items + 2);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = a.nb * a.nh;
    const int total = a.q_tiles * per;
    struct Item {
        int q0, n, head, n_kv;
        bool has_b;
        int last[2];  // last key tile each query tile sees
    };
    auto decode = [&](int item) {
        Item it;
        const int g = item / per;
        const int rem = item - g * per;
        it.n = rem / a.nh;
        it.head = rem - it.n * a.nh;
        it.q0 = (a.q_tiles - 1 - g) * 256;
        it.has_b = it.q0 + 128 < a.s;
        it.last[0] = (it.q0 + 127) / BKV;
        it.last[1] = (it.q0 + 255) / BKV;
        it.n_kv = it.has_b ? it.last[1] + 1 : it.last[0] + 1;
        return it;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);  // one arrival per warp of the tile's warpgroup
            mbar_init(&pv_done[x], 1);
            mbar_init(&o_free[x], 4);
            mbar_init(&item_full[x], 1);
            mbar_init(&item_empty[x], 9);  // the MMA thread and the 8 softmax warps
        }
        mbar_init(drain, 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 8) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_q128);
            prefetch_tmap(&tm_kv);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            int q_loads = 0;
            bool ok = true;
            for (int k = 0;; ++k) {
                const int slot = k & 1;
                if (k >= 2 && !wait_bounded(&item_empty[slot], static_cast<uint32_t>((k - 2) >> 1) & 1u,
                                            abort_flag, a.status, 0x111))
                    ok = false;
                int item = -1;
                if (ok) {
                    item = static_cast<int>(atomicAdd(a.work, 1u));
                    if (item >= total) item = -1;
                }
                items[slot] = item;
                mbar_arrive(&item_full[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                const int qcol = it.head * D, kcol = a.h + it.head * D, vcol = 2 * a.h + it.head * D;
                // the previous item's S MMAs are done with the Q tiles
                if (k >= 1 && !wait_bounded(q_empty, static_cast<uint32_t>(k - 1) & 1u, abort_flag,
                                            a.status, 0x112))
                    break;
                mbar_arrive_expect_tx(q_full, (it.has_b ? 2 : 1) * C::QTILE);
                for (int x = 0; x < (it.has_b ? 2 : 1); ++x)
                    for (int b = 0; b < C::NB; ++b)
                        tma_load_3d(&tm_q128, smem_u32(q_full),
                                    smem_u32(sQ) + x * C::QTILE + b * 128 * kRowBytes, qcol + 64 * b,
                                    it.q0 + 128 * x, it.n);
                ++q_loads;
                for (int idx = 0; idx < 2 * it.n_kv; ++idx) {  // K_j = 2j, V_j = 2j + 1
                    if (!wait_bounded(&kv_empty[stage], phase ^ 1u, abort_flag, a.status, 0x101)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&kv_full[stage], C::KVTILE);
                    const uint32_t dst = smem_u32(ring) + stage * C::KVTILE;
                    const int col = (idx & 1) ? vcol : kcol;
                    for (int b = 0; b < C::NB; ++b)
                        tma_load_3d(&tm_kv, smem_u32(&kv_full[stage]), dst + b * BKV * kRowBytes,
                                    col + 64 * b, (idx >> 1) * BKV, it.n);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (q_loads > 0) wait_drain(q_full, static_cast<uint32_t>(q_loads - 1) & 1u, a.status, 0x102);
            for (int i = 0; i < S; ++i)
                if (issued & (1u << i)) wait_drain(&kv_full[i], (issued_phase >> i) & 1u, a.status, 0x103);
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, BKV, false, false);
            bool ok = true;
            int rstage = 0;  // ring entries are taken in order, across items
            uint32_t rphase = 0;
            int gx[2] = {0, 0};  // S / P V MMAs of each tile over the items so far
            int cx[2] = {0, 0};  // items each tile has taken part in
            // wait for the next ring entry; returns its stage
            auto acquire = [&](int site) -> int {
                const int stage = rstage;
                if (ok && !wait_bounded(&kv_full[stage], rphase, abort_flag, a.status, site)) ok = false;
                tc_fence_after();
                if (++rstage == S) {
                    rstage = 0;
                    rphase ^= 1u;
                }
                return stage;
            };
            int s_left = 0;  // S MMAs of the item still to issue
            auto issue_s = [&](int x, int stage) {  // S_x = Q_x K^T
                const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ) + x * C::QTILE, 16, 1024);
                const uint64_t kdesc = smem_desc_sw128(smem_u32(ring) + stage * C::KVTILE, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_f16(tmem + C::s_col(x), desc_add(qdesc, kmajor_step<128>(kk)),
                               desc_add(kdesc, kmajor_step<BKV>(kk)), id_s, kk > 0 ? 1u : 0u);
                tc_commit(&s_full[x]);
                // the item's last S: once done, the Q tiles may be replaced
                if (--s_left == 0) tc_commit(q_empty);
            };
            auto issue_pv = [&](int x, int j, int stage) {  // O_x (+)= P_x V
                // the first P V of an item overwrites the previous item's O_x
                if (ok && j == 0 && cx[x] >= 1 &&
                    !wait_bounded(&o_free[x], static_cast<uint32_t>(cx[x] - 1) & 1u, abort_flag, a.status,
                                  0x113 + x))
                    ok = false;
                if (ok && !wait_bounded(&p_full[x], static_cast<uint32_t>(gx[x] + j) & 1u, abort_flag,
                                        a.status, 0x105 + x))
                    ok = false;
                if (!ok) return;
                tc_fence_after();
                // O_x (+)= P_x V: A = P_x from TMEM (packed over S_x's first
                // columns), B = V (MN-major: d along the rows, keys down the box)
                const uint64_t vdesc =
                    smem_desc_sw128(smem_u32(ring) + stage * C::KVTILE, BKV * kRowBytes, 1024);
                mma_ts_n_is_d<D, BKV / 16>(tmem + C::o_col(x), tmem + C::s_col(x), vdesc,
                                           BKV * kRowBytes, j > 0, tmem + C::o_tail(x));
                tc_commit(&pv_done[x]);
            };
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                  a.status, 0x115))
                    break;
                const int item = *reinterpret_cast<volatile int*>(&items[slot]);
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                if (!wait_bounded(q_full, static_cast<uint32_t>(k) & 1u, abort_flag, a.status, 0x104)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                s_left = it.last[0] + 1 + (it.has_b ? it.last[1] + 1 : 0);
                // S of both tiles for key tile 0
                int ks = acquire(0x107);
                if (ok) {
                    issue_s(0, ks);
                    if (it.has_b) issue_s(1, ks);
                    tc_commit(&kv_empty[ks]);
                }
                for (int j = 0; j < it.n_kv && ok; ++j) {
                    const int vs = acquire(0x108);
                    const bool more = j + 1 < it.n_kv;
                    int kn = -1;
                    if (j <= it.last[0]) {
                        issue_pv(0, j, vs);
                        if (ok && j + 1 <= it.last[0]) {
                            kn = acquire(0x109);
                            if (ok) issue_s(0, kn);
                        }
                    }
                    if (it.has_b && ok) {
                        issue_pv(1, j, vs);
                        if (ok) tc_commit(&kv_empty[vs]);
                        if (ok && more) {
                            if (kn < 0) kn = acquire(0x10A);
                            if (ok) issue_s(1, kn);
                        }
                    } else if (ok) {
                        tc_commit(&kv_empty[vs]);
                    }
                    if (ok && kn >= 0) tc_commit(&kv_empty[kn]);
                }
                gx[0] += it.last[0] + 1;
                cx[0] += 1;
                if (it.has_b) {
                    gx[1] += it.last[1] + 1;
                    cx[1] += 1;
                }
            }
            tc_commit(drain);
            wait_drain(drain, 0, a.status, 0x10B);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------- softmax warps
        const int x = warp >> 2;               // tile: 0 = A, 1 = B
        const int r = threadIdx.x & 127;       // row of the tile = TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t s_addr = lane_addr + C::s_col(x);
        int gxl = 0;  // this tile's S / P V MMAs over the items so far
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            if (!warp_wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                   a.status, 0x116))
                break;
            const int item = *reinterpret_cast<volatile int*>(&items[slot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Item it = decode(item);
            if (x == 1 && !it.has_b) continue;  // no B tile in this item
            const int q = it.q0 + 128 * x + r;
            const int jl = it.last[x];
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j <= jl; ++j) {
                if (!warp_wait_bounded(&s_full[x], static_cast<uint32_t>(gxl + j) & 1u, abort_flag,
                                       a.status, 0x10C + x)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[SCH][32];
#pragma unroll
                for (int c = 0; c < SCH; ++c) tmem_ld32(s_addr + c * 32, v[c]);
                tmem_wait_ld();
                // causal mask where this key tile reaches past the row's query
                const int k0 = j * BKV;
                if (k0 + BKV - 1 > q) {
#pragma unroll
                    for (int c = 0; c < SCH; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (k0 + c * 32 + i > q) v[c][i] = __float_as_uint(-INFINITY);
                }
                // eight independent max / sum chains: the row is one thread's
                // work, so its reductions must not be one serial chain
                float mx8[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mx8[kk] = -INFINITY;
#pragma unroll
                for (int c = 0; c < SCH; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(v[c][i]));
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                // the reference max only moves when the row max outgrows it by
                // more than 2^8, so the O rescale below is rare.  A row whose
                // keys in this tile are all masked (rows past the sequence end
                // in a 64-key tile) keeps its reference.
                const float m_new = fmaxf(m, mx * a.scale2);
                const bool move = (j == 0 && m_new > -INFINITY) || m_new > m + kRescaleLog2;
                const float alpha = move ? ex2(m - m_new) : 1.0f;
                if (move) m = m_new;
                uint64_t rs2[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) rs2[kk] = 0ull;  // (0.0f, 0.0f)
                const uint64_t scale2 = f32x2(a.scale2, a.scale2), neg_m = f32x2(-m, -m);
                uint32_t pk[SCH][16];
#pragma unroll
                for (int c = 0; c < SCH; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        // masked scores are -inf: 2^-inf = 0
                        float x0, x1;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(v[c][2 * i]), __uint_as_float(v[c][2 * i + 1])),
                                              scale2, neg_m), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        rs2[i & 3] = add_f32x2(rs2[i & 3], f32x2(p0, p1));
                        pk[c][i] = pack_bf16x2(p0, p1);
                    }
                float rsv[8];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) f32x2_split(rs2[kk], rsv[2 * kk], rsv[2 * kk + 1]);
                const float rs = ((rsv[0] + rsv[1]) + (rsv[2] + rsv[3])) + ((rsv[4] + rsv[5]) + (rsv[6] + rsv[7]));
                l = fmaf(l, alpha, rs);
                // S_x(j) was issued after P_x V of the previous key tile, and the
                // commit that signalled S_x covers every earlier MMA: that P V
                // has finished, so O_x is final and P_x's columns are free
                if (j >= 1) {
                    if (__any_sync(0xFFFFFFFFu, move)) {
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(lane_addr + C::o_chunk(x, c), o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(lane_addr + C::o_chunk(x, c), o);
                        }
                        tmem_wait_st();
                    }
                }
                // P_x, packed bf16, over the first columns of S_x (already read)
#pragma unroll
                for (int c = 0; c < SCH; ++c) tmem_st16(s_addr + 16 * c, pk[c]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[x]);
            }
            if (!ok || !warp_wait_bounded(&pv_done[x], static_cast<uint32_t>(gxl + jl) & 1u, abort_flag,
                                          a.status, 0x110 + x)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = 1.0f / l;
            const bool q_ok = q < a.s;
            const long long tok = static_cast<long long>(it.n) * a.s + q;
            uint4* dst = reinterpret_cast<uint4*>(a.O + tok * a.h + it.head * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_addr + C::o_chunk(x, c), o);  // every lane: warp-collective
                tmem_wait_ld();
                if (q_ok) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(o[8 * i]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
                        u.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
                        u.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
                        u.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
                        dst[c * 4 + i] = u;
                    }
                }
            }
            if (q_ok) a.lse[it.head * a.T + tok] = m + lg2(l);
            // O_x is in registers or on its way to memory: the MMA may reuse it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[x]);
            gxl += jl + 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------ delta

// delta[head, tok] = sum_c dO[tok, head*d + c] * O[tok, head*d + c], fp32.
// The (token, head) segments of d elements lie end to end in dO and O, d/8
// 16-byte chunks each.  A CTA takes kDeltaSegs(d) whole segments (at most
// 2048 chunks): its 256 threads read the chunks coalesced (chunk base + tid +
// 256 k, all loads issued before any product), each chunk's 8 products are
// summed and parked in shared memory, and one thread per segment adds its
// chunks in order.
constexpr int kDeltaChunks = 2048;
constexpr int kDeltaThreads = 256;
template <int D>
constexpr int delta_segs() { return kDeltaChunks / (D / 8); }

template <int D>
__global__ void __launch_bounds__(kDeltaThreads)
    attn_delta_kernel(const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ O,
                      long long T, int nh, float* __restrict__ delta) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    constexpr int CH = D / 8;                 // chunks per segment
    constexpr int SEGS = delta_segs<D>();     // segments per CTA
    constexpr int PER = (SEGS * CH + kDeltaThreads - 1) / kDeltaThreads;
    __shared__ float part[SEGS * CH];
    const long long seg0 = static_cast<long long>(blockIdx.x) * SEGS;
    const long long segs_total = T * nh;
    const int segs = static_cast<int>(segs_total - seg0 < SEGS ? segs_total - seg0 : SEGS);
    const int chunks = segs * CH;
    const uint4* g = reinterpret_cast<const uint4*>(dO) + seg0 * CH;
    const uint4* o = reinterpret_cast<const uint4*>(O) + seg0 * CH;
    uint4 gu[PER], ou[PER];
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int c = threadIdx.x + k * kDeltaThreads;
        if (c < chunks) {
            gu[k] = __ldg(g + c);
            ou[k] = __ldg(o + c);
        }
    }
#pragma unroll
    for (int k = 0; k < PER; ++k) {
        const int c = threadIdx.x + k * kDeltaThreads;
        if (c < chunks) {
            const uint32_t gw[4] = {gu[k].x, gu[k].y, gu[k].z, gu[k].w};
            const uint32_t ow[4] = {ou[k].x, ou[k].y, ou[k].z, ou[k].w};
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc = fmaf(__uint_as_float(gw[j] << 16), __uint_as_float(ow[j] << 16), acc);
                acc = fmaf(__uint_as_float(gw[j] & 0xFFFF0000u), __uint_as_float(ow[j] & 0xFFFF0000u), acc);
            }
            part[c] = acc;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < segs; t += kDeltaThreads) {
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < CH; ++i) sum += part[t * CH + i];
        const long long sg = seg0 + t;
        const long long tok = sg / nh;
        const long long head = sg - tok * nh;
        delta[head * T + tok] = sum;
    }
}

// ------------------------------------------------------------- dQ

template <int D>
struct DqCfg {
    static constexpr int NB = (D + 63) / 64;
    static constexpr int ROW_TILE = NB * 128 * kRowBytes;  // Q or dO: 128 rows
    static constexpr int KV_TILE = NB * 64 * kRowBytes;    // K or V: 64 rows
    static constexpr int FIXED = 2 * ROW_TILE;
    static constexpr int STAGES_FIT = (225 * 1024 - FIXED) / (2 * KV_TILE);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int SMEM = 1024 + FIXED + STAGES * 2 * KV_TILE + 256;
};

// Work items of the dQ kernel: (128 queries, sequence, head), heaviest
// (most key tiles) first, taken in turn from the launch's item counter.

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q128,  // QKV, 128-row boxes
                       const __grid_constant__ CUtensorMap tm_kv64,  // QKV, 64-row boxes
                       const __grid_constant__ CUtensorMap tm_do128, // dO, 128-row boxes
                       const AttnArgs a) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    using C = DqCfg<D>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sQ = smem;
    uint8_t* sdO = sQ + C::ROW_TILE;
    uint8_t* ring = sdO + C::ROW_TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + S * 2 * C::KV_TILE);
    uint64_t* q_full = bars;             // the item's Q and dO have landed
    uint64_t* q_empty = bars + 1;        // the item's last S and dP MMAs have read them
    uint64_t* kv_full = bars + 2;
    uint64_t* kv_empty = kv_full + S;
    uint64_t* sdp_full = kv_empty + S;   // [2]
    uint64_t* ds_full = sdp_full + 2;    // [2]
    // dQ accumulators: two for d <= 128 (TMEM columns 256 and 384), so that
    // item k's dQ is read out while item k + 1's MMAs run; one for d = 160
    constexpr int NDQ = D <= 128 ? 2 : 1;
    uint64_t* dq_done = ds_full + 2;     // [NDQ] the item's dQ is complete in TMEM
    uint64_t* dq_free = dq_done + NDQ;   // [NDQ] the softmax warps have read it out
    uint64_t* item_full = dq_free + NDQ; // [2] items[slot] holds the next item
    uint64_t* item_empty = item_full + 2;  // [2] every consumer has read it
    uint64_t* drain = item_empty + 2;
    int* items = reinterpret_cast<int*>(drain + 1);  // [2]
    uint32_t* misc = reinterpret_cast<uint32_t*>(items + 2);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_qt = a.nb * a.nh;
    const int total = a.q_tiles * per_qt;
    struct Item {
        int q0, n, head, n_kv;
    };
    auto decode = [&](int item) {
        Item it;
        const int qt = a.q_tiles - 1 - item / per_qt;
        const int rem = item - (a.q_tiles - 1 - qt) * per_qt;
        it.n = rem / a.nh;
        it.head = rem - it.n * a.nh;
        it.q0 = qt * 128;
        // 64-key tiles holding keys <= the tile's last valid query
        it.n_kv = min(it.q0 + 127, a.s - 1) / 64 + 1;
        return it;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sdp_full[b], 1);
            mbar_init(&ds_full[b], 4);
            mbar_init(&item_full[b], 1);
            mbar_init(&item_empty[b], 5);  // the MMA thread and the 4 softmax warps
        }
        for (int b = 0; b < NDQ; ++b) {
            mbar_init(&dq_done[b], 1);
            mbar_init(&dq_free[b], 4);
        }
        mbar_init(drain, 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // TMEM columns: S[b] at 64 b, dP[b] at 128 + 64 b, dQ[x] at 256 + 128 x
    constexpr uint32_t kS = 0, kDP = 128, kDQ = 256;

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tm_q128);
            prefetch_tmap(&tm_kv64);
            prefetch_tmap(&tm_do128);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            int q_loads = 0;  // Q/dO loads issued (q_full's completed phases)
            bool ok = true;
            for (int k = 0;; ++k) {
                const int slot = k & 1;
                // the slot's item k - 2 has been read by every consumer
                if (k >= 2 && !wait_bounded(&item_empty[slot], static_cast<uint32_t>((k - 2) >> 1) & 1u,
                                            abort_flag, a.status, 0x20B))
                    ok = false;
                int item = -1;
                if (ok) {
                    item = static_cast<int>(atomicAdd(a.work, 1u));
                    if (item >= total) item = -1;
                }
                items[slot] = item;
                mbar_arrive(&item_full[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                const int qcol = it.head * D, kcol = a.h + it.head * D, vcol = 2 * a.h + it.head * D;
                // Q and dO: the previous item's S and dP MMAs are done with them
                if (k >= 1 && !wait_bounded(q_empty, static_cast<uint32_t>(k - 1) & 1u, abort_flag,
                                            a.status, 0x20C))
                    break;
                mbar_arrive_expect_tx(q_full, 2 * C::ROW_TILE);
                for (int b = 0; b < C::NB; ++b) {
                    tma_load_3d(&tm_q128, smem_u32(q_full), smem_u32(sQ) + b * 128 * kRowBytes,
                                qcol + 64 * b, it.q0, it.n);
                    tma_load_3d(&tm_do128, smem_u32(q_full), smem_u32(sdO) + b * 128 * kRowBytes,
                                qcol + 64 * b, it.q0, it.n);
                }
                ++q_loads;
                for (int j = 0; j < it.n_kv && ok; ++j) {
                    if (!wait_bounded(&kv_empty[stage], phase ^ 1u, abort_flag, a.status, 0x201)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&kv_full[stage], 2 * C::KV_TILE);
                    const uint32_t dst = smem_u32(ring) + stage * 2 * C::KV_TILE;
                    for (int b = 0; b < C::NB; ++b) {
                        tma_load_3d(&tm_kv64, smem_u32(&kv_full[stage]), dst + b * 64 * kRowBytes,
                                    kcol + 64 * b, j * 64, it.n);
                        tma_load_3d(&tm_kv64, smem_u32(&kv_full[stage]),
                                    dst + C::KV_TILE + b * 64 * kRowBytes, vcol + 64 * b, j * 64, it.n);
                    }
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // every copy this thread started lands before the CTA may exit
            if (q_loads > 0) wait_drain(q_full, static_cast<uint32_t>(q_loads - 1) & 1u, a.status, 0x202);
            for (int i = 0; i < S; ++i)
                if (issued & (1u << i)) wait_drain(&kv_full[i], (issued_phase >> i) & 1u, a.status, 0x203);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16_f32(128, 64, false, false);
            const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dodesc = smem_desc_sw128(smem_u32(sdO), 16, 1024);
            int stage = 0, g = 0;  // g: tiles of every item so far (S/dP buffer index)
            uint32_t phase = 0;
            bool ok = true;
            // dQ += dS K for tile i of item k (global tile gi), K in ring stage st
            auto issue_dq = [&](int i, int gi, int st, int k) {
                if (!ok) return;
                // the first dQ MMA of an item overwrites the dQ of item k - NDQ
                if (i == 0 && k >= NDQ &&
                    !wait_bounded(&dq_free[k % NDQ], static_cast<uint32_t>((k - NDQ) / NDQ) & 1u,
                                  abort_flag, a.status, 0x20D)) {
                    ok = false;
                    return;
                }
                if (!wait_bounded(&ds_full[gi & 1], static_cast<uint32_t>(gi >> 1) & 1u, abort_flag,
                                  a.status, 0x205)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                // A = dS from TMEM (the softmax threads wrote it, packed bf16,
                // over the first 32 columns of the S buffer), B = K (MN-major:
                // d along the rows, keys down the 64-row box)
                const uint64_t kdesc = smem_desc_sw128(smem_u32(ring) + st * 2 * C::KV_TILE,
                                                       64 * kRowBytes, 1024);
                mma_ts_n_is_d<D, 64 / 16>(tmem + kDQ + 128u * static_cast<uint32_t>(k % NDQ),
                                          tmem + kS + 64 * (gi & 1), kdesc, 64 * kRowBytes, i > 0);
                tc_commit(&kv_empty[st]);
            };
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                  a.status, 0x20E))
                    break;
                const int item = *reinterpret_cast<volatile int*>(&items[slot]);
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                if (!wait_bounded(q_full, static_cast<uint32_t>(k) & 1u, abort_flag, a.status, 0x204)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                int prev_stage = 0;
                for (int j = 0; j < it.n_kv && ok; ++j, ++g) {
                    if (!wait_bounded(&kv_full[stage], phase, abort_flag, a.status, 0x206)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kv = smem_u32(ring) + stage * 2 * C::KV_TILE;
                    const uint64_t kdesc = smem_desc_sw128(kv, 16, 1024);
                    const uint64_t vdesc = smem_desc_sw128(kv + C::KV_TILE, 16, 1024);
                    const uint32_t b = static_cast<uint32_t>(g & 1);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        tc_mma_f16(tmem + kS + 64 * b, desc_add(qdesc, kmajor_step<128>(kk)),
                                   desc_add(kdesc, kmajor_step<64>(kk)), id_s, kk > 0 ? 1u : 0u);
                        tc_mma_f16(tmem + kDP + 64 * b, desc_add(dodesc, kmajor_step<128>(kk)),
                                   desc_add(vdesc, kmajor_step<64>(kk)), id_s, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&sdp_full[b]);
                    // the item's last S and dP have been issued: once they are
                    // done, Q and dO may be replaced by the next item's
                    if (j == it.n_kv - 1) tc_commit(q_empty);
                    if (j >= 1) issue_dq(j - 1, g - 1, prev_stage, k);
                    prev_stage = stage;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                issue_dq(it.n_kv - 1, g - 1, prev_stage, k);
                if (ok) tc_commit(&dq_done[k % NDQ]);
            }
            tc_commit(drain);
            wait_drain(drain, 0, a.status, 0x207);
        }
        __syncwarp();
    } else {
        const int r = threadIdx.x;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bool ok = true;
        int g = 0;
        // An item whose dQ is complete but not yet read out: with two dQ
        // accumulators, item k's is read out after item k + 1's second key
        // tile (its first, when it has one), while the MMA works on item
        // k + 1; with one, at the end of item k.
        struct Pending {
            int k;
            long long tok;
            bool q_ok;
            int head;
        };
        Pending pend{-1, 0, false, 0};
        auto readout = [&](const Pending& pd) -> bool {
            if (!warp_wait_bounded(&dq_done[pd.k % NDQ], static_cast<uint32_t>(pd.k / NDQ) & 1u,
                                   abort_flag, a.status, 0x20A))
                return false;
            tc_fence_after();
            // tcgen05.ld is warp-collective (.sync.aligned): every lane loads,
            // only rows inside the sequence are stored
            uint4* dst = reinterpret_cast<uint4*>(a.dqkv + pd.tok * 3 * a.h + pd.head * D);
            const uint32_t col = kDQ + 128u * static_cast<uint32_t>(pd.k % NDQ);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_addr + col + c * 32, v);
                tmem_wait_ld();
                if (pd.q_ok) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 u;
                        u.x = pack_bf16x2(__uint_as_float(v[8 * i]) * a.scale, __uint_as_float(v[8 * i + 1]) * a.scale);
                        u.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]) * a.scale, __uint_as_float(v[8 * i + 3]) * a.scale);
                        u.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]) * a.scale, __uint_as_float(v[8 * i + 5]) * a.scale);
                        u.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]) * a.scale, __uint_as_float(v[8 * i + 7]) * a.scale);
                        dst[c * 4 + i] = u;
                    }
                }
            }
            // dQ is in registers or on its way to memory: the MMA may reuse it
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(&dq_free[pd.k % NDQ]);
            return true;
        };
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            if (!warp_wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                   a.status, 0x20F))
                break;
            const int item = *reinterpret_cast<volatile int*>(&items[slot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Item it = decode(item);
            const int q = it.q0 + r;
            const bool q_ok = q < a.s;
            const long long tok = static_cast<long long>(it.n) * a.s + q;
            const float lse = q_ok ? __ldg(a.lse_in + it.head * a.T + tok) : 0.0f;
            const float dlt = q_ok ? __ldg(a.delta + it.head * a.T + tok) : 0.0f;
            for (int j = 0; j < it.n_kv; ++j, ++g) {
                const uint32_t b = static_cast<uint32_t>(g & 1);
                // S(g) was issued after dQ(g-2), which read this buffer's
                // previous dS, so once it is here the buffer is free
                if (!warp_wait_bounded(&sdp_full[b], static_cast<uint32_t>(g >> 1) & 1u, abort_flag,
                                       a.status, 0x208)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t sv[32], pv[32];
                    tmem_ld32(lane_addr + kS + 64 * b + c * 32, sv);
                    tmem_ld32(lane_addr + kDP + 64 * b + c * 32, pv);
                    tmem_wait_ld();
                    const int key0 = j * 64 + c * 32;
                    // causal mask (keys after the query), only where this chunk
                    // reaches past the row's query; a masked score of -inf gives
                    // P = 0.  Rows past the sequence read zero Q and dO rows and
                    // are never stored, so they need no mask.
                    if (key0 + 31 > q) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (key0 + i > q) sv[i] = __float_as_uint(-INFINITY);
                    }
                    uint32_t dd[16];
                    const uint64_t scale2 = f32x2(a.scale2, a.scale2), neg_lse = f32x2(-lse, -lse),
                                   neg_dlt = f32x2(-dlt, -dlt);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0, x1, d0, d1;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])),
                                              scale2, neg_lse), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        f32x2_split(mul_f32x2(f32x2(p0, p1),
                                              add_f32x2(f32x2(__uint_as_float(pv[2 * i]),
                                                              __uint_as_float(pv[2 * i + 1])), neg_dlt)), d0, d1);
                        dd[i] = pack_bf16x2(d0, d1);
                    }
                    // dS, packed, over the S columns this thread has read
                    tmem_st16(lane_addr + kS + 64 * b + 16 * c, dd);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ds_full[b]);
                if (NDQ == 2 && pend.k >= 0 && j == (it.n_kv > 1 ? 1 : 0)) {
                    if (!readout(pend)) {
                        ok = false;
                        break;
                    }
                    pend.k = -1;
                }
            }
            if (!ok) break;
            if constexpr (NDQ == 1) {
                if (!readout(Pending{k, tok, q_ok, it.head})) {
                    ok = false;
                    break;
                }
            } else {
                pend = Pending{k, tok, q_ok, it.head};
            }
        }
        if (ok && pend.k >= 0) readout(pend);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------- dK, dV

template <int D>
struct DkvCfg {
    static constexpr int NB = (D + 63) / 64;
    static constexpr int KEY_TILE = NB * 128 * kRowBytes;  // K or V: 128 rows
    static constexpr int Q_TILE = NB * 64 * kRowBytes;     // Q or dO: 64 rows
    static constexpr int FIXED = 2 * KEY_TILE;
    static constexpr int STAGES_FIT = (225 * 1024 - FIXED) / (2 * Q_TILE);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int SMEM = 1024 + FIXED + STAGES * 2 * Q_TILE + 256;
};

// Work items of the dK/dV kernel: (128 keys, sequence, head), the first key
// tiles (most queries after them) first, taken in turn from the launch's item counter.

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k128,  // QKV, 128-row boxes
                         const __grid_constant__ CUtensorMap tm_q64,    // QKV, 64-row boxes
                         const __grid_constant__ CUtensorMap tm_do64,   // dO, 64-row boxes
                         const AttnArgs a) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    using C = DkvCfg<D>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* sK = smem;
    uint8_t* sV = sK + C::KEY_TILE;
    uint8_t* ring = sV + C::KEY_TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring + S * 2 * C::Q_TILE);
    uint64_t* kv_full = bars;            // the item's K and V have landed
    uint64_t* kv_empty = bars + 1;       // the item's last S^T and dP^T MMAs have read them
    uint64_t* q_full = bars + 2;
    uint64_t* q_empty = q_full + S;
    uint64_t* st_full = q_empty + S;     // [2]
    uint64_t* pds_full = st_full + 2;    // [2]
    uint64_t* grad_done = pds_full + 2;  // the item's dV and dK are complete in TMEM
    uint64_t* grad_free = grad_done + 1; // the softmax warps have read them out
    uint64_t* item_full = grad_free + 1;     // [2]
    uint64_t* item_empty = item_full + 2;    // [2]
    uint64_t* drain = item_empty + 2;
    int* items = reinterpret_cast<int*>(drain + 1);  // [2]
    uint32_t* misc = reinterpret_cast<uint32_t*>(items + 2);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per_kt = a.nb * a.nh;
    const int total = ((a.s + 127) / 128) * per_kt;
    struct Item {
        int k0, n, head, i0, nq;
    };
    auto decode = [&](int item) {
        Item it;
        const int kt = item / per_kt;
        const int rem = item - kt * per_kt;
        it.n = rem / a.nh;
        it.head = rem - it.n * a.nh;
        it.k0 = kt * 128;
        it.i0 = it.k0 / 64;                  // first 64-query tile with a query >= k0
        it.nq = (a.s + 63) / 64 - it.i0;     // query tiles to visit
        return it;
    };

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st_full[b], 1);
            mbar_init(&pds_full[b], 4);
            mbar_init(&item_full[b], 1);
            mbar_init(&item_empty[b], 5);  // the MMA thread and the 4 softmax warps
        }
        mbar_init(grad_done, 1);
        mbar_init(grad_free, 4);
        mbar_init(drain, 1);
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // TMEM columns.  d <= 128: S^T[b] at 64 b, dP^T[b] at 128 + 64 b (two
    // buffers, so the next tile's S^T / dP^T run during this tile's softmax),
    // dV at 256, dK at the next multiple of 64 after dV.  d = 160: one buffer
    // (S^T at 0, dP^T at 64), the 128-column parts of dV and dK at 128 and 256
    // and their 32-column tails at 384 and 416.  Every N >= 128 accumulator
    // part starts on a multiple of 128.
    constexpr int NBUF = D <= 128 ? 2 : 1;
    constexpr uint32_t kST = 0, kDPT = NBUF == 2 ? 128 : 64;
    constexpr uint32_t kDV = NBUF == 2 ? 256 : 128;
    constexpr uint32_t kDK = NBUF == 2 ? 256 + ((D + 63) / 64) * 64 : 256;
    constexpr uint32_t kDVt = NBUF == 2 ? kDV + (D / 64) * 64 : 384;
    constexpr uint32_t kDKt = NBUF == 2 ? kDK + (D / 64) * 64 : 416;
    // column of 32-column chunk c of an accumulator with parts at main / tail
    auto acc_col = [](uint32_t main, uint32_t tail, int c) -> uint32_t {
        return c < D / 64 * 2 ? main + 32 * c : tail + 32 * (c - D / 64 * 2);
    };

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tm_k128);
            prefetch_tmap(&tm_q64);
            prefetch_tmap(&tm_do64);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_phase = 0;
            int kv_loads = 0;  // K/V loads issued (kv_full's completed phases)
            bool ok = true;
            for (int k = 0;; ++k) {
                const int slot = k & 1;
                // the slot's item k - 2 has been read by every consumer
                if (k >= 2 && !wait_bounded(&item_empty[slot], static_cast<uint32_t>((k - 2) >> 1) & 1u,
                                            abort_flag, a.status, 0x30B))
                    ok = false;
                int item = -1;
                if (ok) {
                    item = static_cast<int>(atomicAdd(a.work, 1u));
                    if (item >= total) item = -1;
                }
                items[slot] = item;
                mbar_arrive(&item_full[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                const int qcol = it.head * D, kcol = a.h + it.head * D, vcol = 2 * a.h + it.head * D;
                // K and V: the previous item's S^T and dP^T MMAs are done with them
                if (k >= 1 && !wait_bounded(kv_empty, static_cast<uint32_t>(k - 1) & 1u, abort_flag,
                                            a.status, 0x30C))
                    break;
                mbar_arrive_expect_tx(kv_full, 2 * C::KEY_TILE);
                for (int b = 0; b < C::NB; ++b) {
                    tma_load_3d(&tm_k128, smem_u32(kv_full), smem_u32(sK) + b * 128 * kRowBytes,
                                kcol + 64 * b, it.k0, it.n);
                    tma_load_3d(&tm_k128, smem_u32(kv_full), smem_u32(sV) + b * 128 * kRowBytes,
                                vcol + 64 * b, it.k0, it.n);
                }
                ++kv_loads;
                for (int i = 0; i < it.nq && ok; ++i) {
                    if (!wait_bounded(&q_empty[stage], phase ^ 1u, abort_flag, a.status, 0x301)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&q_full[stage], 2 * C::Q_TILE);
                    const uint32_t dst = smem_u32(ring) + stage * 2 * C::Q_TILE;
                    const int qrow = (it.i0 + i) * 64;
                    for (int b = 0; b < C::NB; ++b) {
                        tma_load_3d(&tm_q64, smem_u32(&q_full[stage]), dst + b * 64 * kRowBytes,
                                    qcol + 64 * b, qrow, it.n);
                        tma_load_3d(&tm_do64, smem_u32(&q_full[stage]),
                                    dst + C::Q_TILE + b * 64 * kRowBytes, qcol + 64 * b, qrow, it.n);
                    }
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // every copy this thread started lands before the CTA may exit
            if (kv_loads > 0) wait_drain(kv_full, static_cast<uint32_t>(kv_loads - 1) & 1u, a.status, 0x302);
            for (int i = 0; i < S; ++i)
                if (issued & (1u << i)) wait_drain(&q_full[i], (issued_phase >> i) & 1u, a.status, 0x303);
        }
        __syncwarp();
    } else if (warp == 5) {
        if (lane == 0) {
            constexpr uint32_t id_st = idesc_bf16_f32(128, 64, false, false);
            const uint64_t kdesc = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t vdesc = smem_desc_sw128(smem_u32(sV), 16, 1024);
            int stage = 0, g = 0;  // g: query tiles of every item so far
            uint32_t phase = 0;
            bool ok = true;
            // dV / dK of tile i of item k (global tile gi), Q/dO in ring stage st
            auto issue_grads = [&](int i, int gi, int st, int k) {
                if (!ok) return;
                // the first dV / dK MMAs of an item overwrite the previous item's
                if (i == 0 && k >= 1 &&
                    !wait_bounded(grad_free, static_cast<uint32_t>(k - 1) & 1u, abort_flag, a.status, 0x30D)) {
                    ok = false;
                    return;
                }
                if (!wait_bounded(&pds_full[NBUF == 2 ? (gi & 1) : 0],
                                  static_cast<uint32_t>(NBUF == 2 ? (gi >> 1) : gi) & 1u, abort_flag,
                                  a.status, 0x305)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                const uint32_t qd = smem_u32(ring) + st * 2 * C::Q_TILE;
                // dV += P^T dO and dK += dS^T Q: A = P^T / dS^T from TMEM (the
                // softmax threads wrote them, packed bf16, over the first 32
                // columns of the S^T / dP^T buffer), B = dO / Q (MN-major: d
                // along the rows, queries down the 64-row box)
                const uint64_t dodesc = smem_desc_sw128(qd + C::Q_TILE, 64 * kRowBytes, 1024);
                const uint64_t qdesc = smem_desc_sw128(qd, 64 * kRowBytes, 1024);
                const uint32_t b = NBUF == 2 ? static_cast<uint32_t>(gi & 1) : 0u;
                mma_ts_n_is_d<D, 64 / 16>(tmem + kDV, tmem + kST + 64 * b, dodesc, 64 * kRowBytes, i > 0,
                                          tmem + kDVt);
                mma_ts_n_is_d<D, 64 / 16>(tmem + kDK, tmem + kDPT + 64 * b, qdesc, 64 * kRowBytes, i > 0,
                                          tmem + kDKt);
                tc_commit(&q_empty[st]);
            };
            for (int k = 0; ok; ++k) {
                const int slot = k & 1;
                if (!wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                  a.status, 0x30E))
                    break;
                const int item = *reinterpret_cast<volatile int*>(&items[slot]);
                mbar_arrive(&item_empty[slot]);
                if (item < 0) break;
                const Item it = decode(item);
                if (!wait_bounded(kv_full, static_cast<uint32_t>(k) & 1u, abort_flag, a.status, 0x304)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                int prev_stage = 0;
                for (int i = 0; i < it.nq && ok; ++i, ++g) {
                    if (!wait_bounded(&q_full[stage], phase, abort_flag, a.status, 0x306)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t qd = smem_u32(ring) + stage * 2 * C::Q_TILE;
                    const uint64_t qdesc = smem_desc_sw128(qd, 16, 1024);
                    const uint64_t dodesc = smem_desc_sw128(qd + C::Q_TILE, 16, 1024);
                    const uint32_t b = NBUF == 2 ? static_cast<uint32_t>(g & 1) : 0u;
                    // S^T = K Q^T and dP^T = V dO^T (M = 128 keys, N = 64 queries, K = d)
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        tc_mma_f16(tmem + kST + 64 * b, desc_add(kdesc, kmajor_step<128>(kk)),
                                   desc_add(qdesc, kmajor_step<64>(kk)), id_st, kk > 0 ? 1u : 0u);
                        tc_mma_f16(tmem + kDPT + 64 * b, desc_add(vdesc, kmajor_step<128>(kk)),
                                   desc_add(dodesc, kmajor_step<64>(kk)), id_st, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&st_full[b]);
                    // the item's last S^T and dP^T have been issued: once they are
                    // done, K and V may be replaced by the next item's
                    if (i == it.nq - 1) tc_commit(kv_empty);
                    if constexpr (NBUF == 2) {
                        // the previous tile's dV / dK run while this tile is softmaxed
                        if (i >= 1) issue_grads(i - 1, g - 1, prev_stage, k);
                    } else {
                        // one buffer: this tile's dV / dK before the next S^T
                        issue_grads(i, g, stage, k);
                    }
                    prev_stage = stage;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if constexpr (NBUF == 2) issue_grads(it.nq - 1, g - 1, prev_stage, k);
                if (ok) tc_commit(grad_done);
            }
            tc_commit(drain);
            wait_drain(drain, 0, a.status, 0x307);
        }
        __syncwarp();
    } else {
        const int r = threadIdx.x;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bool ok = true;
        int g = 0;
        for (int k = 0; ok; ++k) {
            const int slot = k & 1;
            if (!warp_wait_bounded(&item_full[slot], static_cast<uint32_t>(k >> 1) & 1u, abort_flag,
                                   a.status, 0x30F))
                break;
            const int item = *reinterpret_cast<volatile int*>(&items[slot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&item_empty[slot]);
            if (item < 0) break;
            const Item it = decode(item);
            const int i0 = it.i0, nq = it.nq, n = it.n, head = it.head;
            const int key = it.k0 + r;
            const float* lse_seq = a.lse_in + head * a.T + static_cast<long long>(n) * a.s;
            const float* dlt_seq = a.delta + head * a.T + static_cast<long long>(n) * a.s;
            // lse and delta of a 64-query tile: lane l holds queries l and 32 + l
            // (lse +inf and delta 0 past the sequence, so P = 0 there); the
            // next tile's are loaded while this one is computed, and each chunk
            // reads them by warp shuffle
            auto fetch = [&](int i, float (&lv)[2], float (&dv)[2]) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int qq = (i0 + i) * 64 + 32 * h2 + lane;
                    const bool in = i < nq && qq < a.s;
                    lv[h2] = in ? -__ldg(lse_seq + qq) : -INFINITY;  // held negated
                    dv[h2] = in ? -__ldg(dlt_seq + qq) : -0.0f;
                }
            };
            float lse_c[2], dlt_c[2];
            fetch(0, lse_c, dlt_c);
            for (int i = 0; i < nq; ++i, ++g) {
                const uint32_t b = NBUF == 2 ? static_cast<uint32_t>(g & 1) : 0u;
                float lse_n[2], dlt_n[2];
                fetch(i + 1, lse_n, dlt_n);
                // S^T(g) was issued after the dV / dK that last read this buffer's
                // P^T / dS^T, so once it is here the buffer is free
                if (!warp_wait_bounded(&st_full[b], static_cast<uint32_t>(NBUF == 2 ? (g >> 1) : g) & 1u,
                                       abort_flag, a.status, 0x308)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int qa = (i0 + i) * 64 + c * 32;  // first query of this chunk
                    uint32_t sv[32], pv[32];
                    tmem_ld32(lane_addr + kST + 64 * b + c * 32, sv);
                    tmem_ld32(lane_addr + kDPT + 64 * b + c * 32, pv);
                    tmem_wait_ld();
                    // causal mask: queries before this row's key
                    if (qa < key) {
#pragma unroll
                        for (int v = 0; v < 32; ++v)
                            if (qa + v < key) sv[v] = __float_as_uint(-INFINITY);
                    }
                    uint32_t pp[16], dd[16];
                    const uint64_t scale2 = f32x2(a.scale2, a.scale2);
#pragma unroll
                    for (int v = 0; v < 16; ++v) {
                        const uint64_t neg_lq = f32x2(__shfl_sync(0xFFFFFFFFu, lse_c[c], 2 * v),
                                                      __shfl_sync(0xFFFFFFFFu, lse_c[c], 2 * v + 1));
                        const uint64_t neg_dq = f32x2(__shfl_sync(0xFFFFFFFFu, dlt_c[c], 2 * v),
                                                      __shfl_sync(0xFFFFFFFFu, dlt_c[c], 2 * v + 1));
                        float x0, x1, d0, d1;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(sv[2 * v]), __uint_as_float(sv[2 * v + 1])),
                                              scale2, neg_lq), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        f32x2_split(mul_f32x2(f32x2(p0, p1),
                                              add_f32x2(f32x2(__uint_as_float(pv[2 * v]),
                                                              __uint_as_float(pv[2 * v + 1])), neg_dq)), d0, d1);
                        pp[v] = pack_bf16x2(p0, p1);
                        dd[v] = pack_bf16x2(d0, d1);
                    }
                    // P^T and dS^T, packed, over the columns this thread has read
                    tmem_st16(lane_addr + kST + 64 * b + 16 * c, pp);
                    tmem_st16(lane_addr + kDPT + 64 * b + 16 * c, dd);
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    lse_c[h2] = lse_n[h2];
                    dlt_c[h2] = dlt_n[h2];
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&pds_full[b]);
            }
            if (!ok || !warp_wait_bounded(grad_done, static_cast<uint32_t>(k) & 1u, abort_flag, a.status,
                                          0x30A)) {
                ok = false;
                break;
            }
            {
                tc_fence_after();
                // tcgen05.ld is warp-collective (.sync.aligned): every lane loads,
                // only keys inside the sequence are stored
                const bool key_ok = key < a.s;
                const long long tok = static_cast<long long>(n) * a.s + key;
                uint4* dk = reinterpret_cast<uint4*>(a.dqkv + tok * 3 * a.h + a.h + head * D);
                uint4* dv = reinterpret_cast<uint4*>(a.dqkv + tok * 3 * a.h + 2 * a.h + head * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32], k[32];
                    tmem_ld32(lane_addr + acc_col(kDV, kDVt, c), v);
                    tmem_ld32(lane_addr + acc_col(kDK, kDKt, c), k);
                    tmem_wait_ld();
                    if (key_ok) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint4 u, w;
                            u.x = pack_bf16x2(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1]));
                            u.y = pack_bf16x2(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3]));
                            u.z = pack_bf16x2(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5]));
                            u.w = pack_bf16x2(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7]));
                            w.x = pack_bf16x2(__uint_as_float(k[8 * i]) * a.scale, __uint_as_float(k[8 * i + 1]) * a.scale);
                            w.y = pack_bf16x2(__uint_as_float(k[8 * i + 2]) * a.scale, __uint_as_float(k[8 * i + 3]) * a.scale);
                            w.z = pack_bf16x2(__uint_as_float(k[8 * i + 4]) * a.scale, __uint_as_float(k[8 * i + 5]) * a.scale);
                            w.w = pack_bf16x2(__uint_as_float(k[8 * i + 6]) * a.scale, __uint_as_float(k[8 * i + 7]) * a.scale);
                            dv[c * 4 + i] = u;
                            dk[c * 4 + i] = w;
                        }
                    }
                }
            }
            // dV and dK are in registers or on their way to memory: the MMA may reuse them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(grad_free);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// ------------------------------------------------------------- launchers

namespace {
// CTAs of a persistent attention kernel: one per SM at most.
unsigned persistent_grid(unsigned items) {
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return items < static_cast<unsigned>(sms) ? items : static_cast<unsigned>(sms);
}
}  // namespace

cudaError_t launch_attn_forward(const CUtensorMap& tm_qkv128, const CUtensorMap& tm_qkv64, int d,
                                const AttnParams& p, cudaStream_t st, int* launches) {
    AttnArgs a{};
    a.nb = p.nb; a.s = p.s; a.h = p.h; a.nh = p.nh;
    a.T = static_cast<long long>(p.nb) * p.s;
    a.q_tiles = (p.s + 255) / 256;  // pairs of 128-query tiles
    a.scale = 1.0f / sqrtf(static_cast<float>(d));
    a.scale2 = 1.4426950408889634f * a.scale;
    a.O = p.O;
    a.lse = p.lse;
    a.status = p.status;
    // persistent: items (query-tile pairs x sequences x heads) taken in turn
    const unsigned grid = persistent_grid(static_cast<unsigned>(a.q_tiles * p.nb * p.nh));
    a.work = p.work;
    cudaError_t e = cudaMemsetAsync(p.work, 0, sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
#define TPMLP_ATTN_FWD(DD)                                                                        \
    if (d == DD) {                                                                                \
        auto kern = attn_fwd_kernel<DD>;                                                          \
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<DD>::SMEM); \
        if (e == cudaSuccess)                                                                     \
            kern<<<grid, kFwdThreads, FwdCfg<DD>::SMEM, st>>>(                                    \
                tm_qkv128, FwdCfg<DD>::BKV == 128 ? tm_qkv128 : tm_qkv64, a);                     \
    }
    TPMLP_ATTN_FWD(64)
    TPMLP_ATTN_FWD(96)
    TPMLP_ATTN_FWD(128)
    TPMLP_ATTN_FWD(160)
#undef TPMLP_ATTN_FWD
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e == cudaSuccess) ++*launches;
    return e;
}

cudaError_t launch_attn_backward(const CUtensorMap& tm_qkv128, const CUtensorMap& tm_qkv64,
                                 const CUtensorMap& tm_do128, const CUtensorMap& tm_do64, int d,
                                 const AttnParams& p, cudaStream_t st, int* launches) {
    AttnArgs a{};
    a.nb = p.nb; a.s = p.s; a.h = p.h; a.nh = p.nh;
    a.T = static_cast<long long>(p.nb) * p.s;
    a.scale = 1.0f / sqrtf(static_cast<float>(d));
    a.scale2 = 1.4426950408889634f * a.scale;
    a.lse_in = p.lse_in;
    a.dqkv = p.dqkv;
    a.status = p.status;
    // delta = rowsum(dO * O)
    {
        const long long items = a.T * p.nh;  // (token, head) segments
        auto blocks = [&](int segs) { return static_cast<unsigned>((items + segs - 1) / segs); };
        if (d == 64)
            attn_delta_kernel<64><<<blocks(delta_segs<64>()), kDeltaThreads, 0, st>>>(
                p.dO, p.O_in, a.T, p.nh, p.delta_out);
        if (d == 96)
            attn_delta_kernel<96><<<blocks(delta_segs<96>()), kDeltaThreads, 0, st>>>(
                p.dO, p.O_in, a.T, p.nh, p.delta_out);
        if (d == 128)
            attn_delta_kernel<128><<<blocks(delta_segs<128>()), kDeltaThreads, 0, st>>>(
                p.dO, p.O_in, a.T, p.nh, p.delta_out);
        if (d == 160)
            attn_delta_kernel<160><<<blocks(delta_segs<160>()), kDeltaThreads, 0, st>>>(
                p.dO, p.O_in, a.T, p.nh, p.delta_out);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        ++*launches;
    }
    a.delta = p.delta_out;
    cudaError_t e = cudaSuccess;
    const int q_tiles = (p.s + 127) / 128;
    AttnArgs aq = a;
    aq.q_tiles = q_tiles;
    aq.work = p.work;      // the dQ kernel's item counter
    a.work = p.work + 1;   // the dK/dV kernel's
    e = cudaMemsetAsync(p.work, 0, 2 * sizeof(unsigned int), st);
    if (e != cudaSuccess) return e;
    // the dQ and dK/dV kernels are persistent: one CTA per SM at most, items
    // taken in turn (both have q_tiles x nb x nh items)
    const unsigned dq_grid = persistent_grid(static_cast<unsigned>(q_tiles * p.nb * p.nh));
#define TPMLP_ATTN_BWD(DD)                                                                          \
    if (d == DD) {                                                                                  \
        auto kq = attn_bwd_dq_kernel<DD>;                                                           \
        e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<DD>::SMEM); \
        if (e == cudaSuccess) {                                                                     \
            kq<<<dq_grid, kAttnThreads, DqCfg<DD>::SMEM, st>>>(tm_qkv128, tm_qkv64, tm_do128, aq);  \
            e = cudaGetLastError();                                                                 \
        }                                                                                           \
        if (e == cudaSuccess) {                                                                     \
            ++*launches;                                                                            \
            auto kk = attn_bwd_dkdv_kernel<DD>;                                                     \
            e = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvCfg<DD>::SMEM); \
            if (e == cudaSuccess) {                                                                 \
                kk<<<dq_grid, kAttnThreads, DkvCfg<DD>::SMEM, st>>>(tm_qkv128, tm_qkv64, tm_do64, a); \
                e = cudaGetLastError();                                                             \
            }                                                                                       \
            if (e == cudaSuccess) ++*launches;                                                      \
        }                                                                                           \
    }
    TPMLP_ATTN_BWD(64)
    TPMLP_ATTN_BWD(96)
    TPMLP_ATTN_BWD(128)
    TPMLP_ATTN_BWD(160)
#undef TPMLP_ATTN_BWD
    return e;
}

}  // namespace tpmlp
