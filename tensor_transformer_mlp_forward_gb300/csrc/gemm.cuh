// gemm.cuh -- persistent tcgen05/TMEM bf16 GEMM for sm_103a with the MLP
// block's fused epilogues.
//
//   D[m, n] = sum_k A[m, k] * B[n, k]        (fp32 accumulation in TMEM)
//
// A is the "rows" operand ([M, K] logically) and B the "columns" operand
// ([N, K] logically); each is stored K-major (k contiguous) or MN-major
// (m / n contiguous), chosen per GEMM so that every product of the block's
// forward and backward pass reads the row-major tensors in place, with no
// transpose kernel.
//
// Shards.  The block's t shards are index ranges of one tensor.  Each
// operand is addressed through a 3-D tensor map whose middle or outer
// dimension is the shard index, so a tile never crosses a shard boundary
// and the tensor memory accelerator zero-fills each shard's ragged tail:
//   SHARD_N  output columns split (column-parallel GEMM): tiles enumerate
//            (shard, m tile, n tile inside the shard);
//   SHARD_M  output rows split (the dB GEMM);
//   SHARD_K  reduction split (row-parallel GEMM): each output tile walks
//            shard 0's K range, then shard 1's, ..., accumulating into the
//            same TMEM accumulator -- the in-device g / f operator sum.
//
// CTA layout (32 (EW + 2) threads, one CTA per SM, persistent over tiles):
//   warps 0..EW-1  epilogue: TMEM -> registers -> fused math -> global
//                  memory; warp w reads TMEM lane quadrant w % 4
//                  (accumulator rows 32 (w % 4) ..) and, with EW = 8, the
//                  half w / 4 of the 256 columns;
//   warp EW        TMA producer (one thread) feeding a STAGES-deep smem ring;
//   warp EW + 1    TMEM owner and MMA issuer (one thread).
// Two 128x256 fp32 accumulators (all 512 TMEM columns) let the epilogue of
// tile i overlap the mainloop of tile i+1.  With a short reduction a tile's
// mainloop is short too (16 k-blocks at K = 1024), and four epilogue warps,
// one per scheduler, may not hide their own load and store latencies behind
// it; EW = 8 puts two epilogue warps on every scheduler, each with half of
// the columns, at the price of one pipeline stage (its staging buffers).
// The dZ GEMM, whose epilogue is the heaviest, is built in both forms.
//
// PAIR variant (cluster of 2 CTAs on neighbouring SMs, tcgen05 cta_group::2):
// the pair computes a 256 x 256 tile.  Each CTA loads its own 128 rows of A
// and 128 of the 256 B rows; the leader CTA's single thread issues
// M=256 x N=256 MMAs that read both CTAs' shared memory and write 128
// accumulator rows into each CTA's TMEM.  Per flop this halves the B traffic
// into each SM (shared memory and L2), and leaves room for 7 stages.
//
// The producer and MMA loops are single threads whose per-k-block latency
// decides how much of the TMA latency the ring hides, so they carry no
// divisions and no descriptor construction: shard and k advance by
// counters, descriptors by adding offsets to precomputed bases.
#pragma once

#include "philox.cuh"
#include "ptx.cuh"

namespace tpmlp {

constexpr int BM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;  // accumulator columns (one TMEM accumulator)
constexpr int BK = 64;   // 64 bf16 = one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int MN_ATOM_BYTES = 64 * BK * 2;  // one 64-wide MN-major box: 8 KiB
constexpr int TMEM_COLS = 512;
constexpr int BAR_BYTES = 512;
constexpr int kTileSlots = 4;  // responses of the dynamic tile scheduler in flight
// Epilogue staging: per epilogue warp two buffers, each a 32-row x 64-column
// bf16 block (rows 128 B apart, 128-byte swizzle) stored by one TMA store.
constexpr int EPI_BUF_BYTES = 32 * 128;

// Per-variant geometry.  Single CTA: a 128 x 256 tile, stages of
// A 128x64 + B 256x64 (48 KiB).  CTA pair (cluster of 2, cta_group::2): a
// 256 x 256 tile, each CTA holding 128 rows of A and 128 rows of B per stage
// (32 KiB).  Wide pair (TN = 512): a 256 x 512 tile computed as two N = 256
// MMAs that share the A stage, each CTA holding 128 rows of A and 256 of B
// (48 KiB, four stages), the whole of TMEM one accumulator: a quarter fewer
// operand bytes from L2 per flop, no second accumulator for the epilogue to
// drain while the next tile runs.  EW epilogue warps with two staging
// buffers each; the stages fill what is left of the 227 KiB of shared
// memory.
template <bool PAIR, int EW = 4, int TN = BN>
struct Geometry {
    static constexpr bool WIDE = TN == 2 * BN;
    static constexpr int TILE_M = PAIR ? 2 * BM : BM;
    static constexpr int TILE_N = TN;
    static constexpr int ACCS = WIDE ? 1 : 2;             // TMEM accumulators
    static constexpr int B_ROWS = PAIR ? TN / 2 : BN;  // B rows in this CTA's smem
    static constexpr int STAGES = WIDE ? 4 : PAIR ? (EW == 8 ? 5 : 6) : (EW == 8 ? 3 : 4);
    static constexpr int THREADS = 32 * (EW + 2);
    static constexpr int A_STAGE_BYTES = BM * BK * 2;
    static constexpr int B_STAGE_BYTES = B_ROWS * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGING_BYTES = EW * 2 * EPI_BUF_BYTES;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
    static_assert(EW == 4 || EW == 8, "four or eight epilogue warps");
    static_assert(TN == BN || (PAIR && EW == 4 && TN == 2 * BN), "wide tiles: CTA pairs, 4 warps");
    static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");
};

enum ShardMode { SHARD_NONE = 0, SHARD_N = 1, SHARD_M = 2, SHARD_K = 3 };
// Where an operand's tensor map carries the shard index.
enum ShardOn { ON_NONE = 0, ON_CONTIG = 1, ON_ROWS = 2 };
// EPI_PARTIAL: split reduction -- the fp32 accumulator of k-range split ks is
// stored as is into plane ks of an fp32 [splits, M, N] workspace.
// EPI_BIAS: + bias only (the attention block's Q/K/V projection).
enum Epilogue {
    EPI_BIAS_GELU = 0,
    EPI_BIAS_RESIDUAL = 1,
    EPI_DGELU = 2,
    EPI_STORE = 3,
    EPI_PARTIAL = 4,
    EPI_BIAS = 5
};

struct GemmArgs {
    int M, N;            // output extent of one shard (SHARD_M: M per shard; SHARD_N: N per shard)
    int shards;          // t
    int shard_mode;      // ShardMode
    int a_on, b_on;      // ShardOn of each operand's tensor map
    int m_tiles;         // m tiles (TILE_M rows) per shard (SHARD_M) or in total
    int n_tiles;         // n tiles per shard (SHARD_N) or in total
    int mt_total, nt_total;
    int k_blocks;        // BK blocks per shard (SHARD_K) or in total
    int num_tiles;       // work units: output tiles x k_splits
    int base_tiles;      // output tiles (mt_total * nt_total)
    int k_splits;        // contiguous k-block ranges per output tile (EPI_PARTIAL)
    int raster_m_fastest;
    int band;            // tiles per band along the fast dimension (see decode_tile)
    int o_on;             // ShardOn of the output tensor maps (Z and H, Y, dZ, dX, dA or dB)
    const __nv_bfloat16* bias;  // b1 or b2, indexed by global output column
    const __nv_bfloat16* aux;   // residual (EPI_BIAS_RESIDUAL) or Z (EPI_DGELU)
    long long ld_aux;
    int skip_o0;    // EPI_BIAS_GELU: 1 = H only, Z is not stored (recomputed later)
    Dropout drop;   // EPI_BIAS_RESIDUAL: bias-dropout-add (drop.threshold 0: none)
    float* colsum;  // EPI_DGELU: column sums per 32-row block, [4 * mt_total][ld_colsum]
    long long ld_colsum;
    int* status;    // device status word
    // This launch covers output tiles [tile_offset, tile_offset + base_tiles)
    // of the raster order (decode_tile); 0 and all tiles by default.
    int tile_offset;
    // EPI_PARTIAL: 1 = the partial sums of work unit u go to slot u of a
    // compact [units, TILE_M, BN] fp32 map (tile-local coordinates) instead
    // of split ks of a [splits, M, N] map.
    int partial_compact;
    int epi_warps;  // host side: 4 or 8 epilogue warps (the kernel variant launched)
    int dependent_launch;  // host side: launched with programmatic stream serialization
    // 1: the grid holds one CTA (pair) per work unit and a running CTA (pair)
    // takes the next unit by cancelling the launch of a pending one (cluster
    // launch control), so the units in flight are always a contiguous run of
    // the raster order; 0: a persistent grid, CTA (pair) u takes units
    // u, u + units, ...
    int dynamic_tiles;
    // MN-major operands whose tensor map is the 4-D view {64, k, mn / 64,
    // shard} (a_mn4 for A, b_mn4 for B): the operand's whole part of a
    // stage (ROWS / 64 atoms of 64 x BK) is one box.
    int a_mn4, b_mn4;
    int tile_n;  // host side: output columns of a CTA pair's tile, BN or 2 BN (wide)
};

struct TileCoord {
    int m0, n0, s;
    int ks;    // k-range split of this work unit (0 unless the reduction is split)
    int slot;  // the work unit's index in this launch
};

template <int TILE_M, int TILE_N = BN>
__device__ __forceinline__ TileCoord decode_tile(int tile, const GemmArgs& p) {
    // Work unit -> (split, output tile): the splits of one tile are
    // base_tiles apart, so each split sweeps the tiles in the order below.
    const int slot = tile;
    const int ks = tile / p.base_tiles;
    tile -= ks * p.base_tiles;
    tile += p.tile_offset;
    // Tiles are visited in bands of `band` tiles along the fast dimension:
    // inside a band the fast index cycles over the band while the slow index
    // advances, so the band's panels of the fast-dimension operand stay in L2
    // while the other operand streams past them.
    int mi, ni;
    if (p.raster_m_fastest) {
        const int per_band = p.band * p.nt_total;
        const int b = tile / per_band;
        const int in = tile - b * per_band;
        const int width = min(p.band, p.mt_total - b * p.band);
        mi = b * p.band + in % width;
        ni = in / width;
    } else {
        const int per_band = p.band * p.mt_total;
        const int b = tile / per_band;
        const int in = tile - b * per_band;
        const int width = min(p.band, p.nt_total - b * p.band);
        ni = b * p.band + in % width;
        mi = in / width;
    }
    TileCoord c;
    c.s = 0;
    c.ks = ks;
    c.slot = slot;
    if (p.shard_mode == SHARD_N) {
        c.s = ni / p.n_tiles;
        ni -= c.s * p.n_tiles;
    } else if (p.shard_mode == SHARD_M) {
        c.s = mi / p.m_tiles;
        mi -= c.s * p.m_tiles;
    }
    c.m0 = mi * TILE_M;
    c.n0 = ni * TILE_N;
    return c;
}

// Tensor-map coordinates of an operand element given its contiguous and row
// indices inside shard s.
__device__ __forceinline__ void tma_coords(int on, int contig, int row, int s, int& c0, int& c1,
                                           int& c2) {
    if (on == ON_CONTIG) {
        c0 = contig; c1 = s; c2 = row;
    } else if (on == ON_ROWS) {
        c0 = contig; c1 = row; c2 = s;
    } else {
        c0 = contig; c1 = row; c2 = 0;
    }
}

// Loads one operand's [ROWS x BK] slice for the k-block starting at k0 into
// shared address `dst`; completion counts on the mbarrier at `bar` (in a
// pair: the leader's barrier, a shared::cluster address).
//  K-major:  one box of 64 (k) x ROWS (m or n), rows 128 B apart.
//  MN-major: with mn4 (the 4-D map {64, k, mn / 64, shard}), one box of
//            64 x BK x ROWS/64 whose atoms land 8 KiB apart; otherwise
//            (a ragged MN extent) ROWS/64 boxes of 64 (m or n) x BK (k),
//            each 8 KiB.  The producer's issue per box sets the pace of a
//            stage, so fewer boxes is faster.
template <bool MN, int ROWS, bool PAIR>
__device__ __forceinline__ void load_operand(const CUtensorMap* map, uint32_t bar, uint32_t dst,
                                             int on, int mn0, int k0, int s, int mn4) {
    if (MN && mn4) {  // one box: the ROWS / 64 atoms land MN_ATOM_BYTES apart
        const int sh = on == ON_NONE ? 0 : s;
        if constexpr (PAIR)
            tma_load_4d_pair(map, bar, dst, 0, k0, mn0 >> 6, sh);
        else
            tma_load_4d(map, bar, dst, 0, k0, mn0 >> 6, sh);
        return;
    }
    int c0, c1, c2;
#pragma unroll
    for (int j = 0; j < (MN ? ROWS / 64 : 1); ++j) {
        if (!MN)
            tma_coords(on, k0, mn0, s, c0, c1, c2);
        else
            tma_coords(on, mn0 + 64 * j, k0, s, c0, c1, c2);
        if constexpr (PAIR)
            tma_load_3d_pair(map, bar, dst + j * MN_ATOM_BYTES, c0, c1, c2);
        else
            tma_load_3d(map, bar, dst + j * MN_ATOM_BYTES, c0, c1, c2);
    }
}

// Descriptor of an operand stage buffer starting at shared address `base`.
//  K-major:  rows 128 B apart, 8-row groups 1024 B apart (SBO); LBO unused.
//  MN-major: 64-wide MN atoms MN_ATOM_BYTES apart (LBO), 8-deep k groups
//            1024 B apart (SBO).
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base) {
    if (!MN) return smem_desc_sw128(base, 16, 1024);
    return smem_desc_sw128(base, MN_ATOM_BYTES, 1024);
}

// Start-address step (in the descriptor's 16-byte units) from one UMMA_K
// slice to the next: 32 B along a swizzled K-major row, or 16 rows (2 KiB)
// of an MN-major box.
template <bool MN>
constexpr uint64_t desc_k_step() {
    return MN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
}

// ------------------------------------------------------------ epilogue math

// tanh GeLU with u(x) = c x (1 + a x^2), c = sqrt(2/pi), a = 0.044715:
//   GeLU(x)  = 0.5 x (1 + tanh u)
//   GeLU'(x) = 0.5 (1 + th) + 0.5 x (1 - th^2) u'(x),  th = tanh u,
// the latter rearranged as 0.5 + w + th (0.5 - w th) with w = 0.5 x u'(x),
// u'(x) = c (1 + 3 a x^2), to keep the epilogue's instruction count low.
constexpr float kGeluC = 0.7978845608028654f;
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ float gelu_tanh(float x) {
    const float th = tanh_approx(x * fmaf(kGeluC * kGeluA, x * x, kGeluC));
    const float hx = 0.5f * x;
    return fmaf(hx, th, hx);
}

__device__ __forceinline__ float gelu_tanh_grad(float x) {
    const float x2 = x * x;
    const float th = tanh_approx(x * fmaf(kGeluC * kGeluA, x2, kGeluC));
    const float w = x * fmaf(1.5f * kGeluC * kGeluA, x2, 0.5f * kGeluC);
    return fmaf(th, fmaf(-w, th, 0.5f), 0.5f + w);
}

// 32 consecutive bf16 values -> float; entries at or beyond `valid` read 0.
__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* p, int valid, float (&v)[32]) {
    if (valid >= 32) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 u = __ldg(q + i);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = i < valid ? __bfloat162float(p[i]) : 0.0f;
    }
}

// Raw bf16 bits of 32 consecutive values (entries at or beyond `valid` are
// 0), so that the loads can be issued well before the values are needed.
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* p, int valid, uint4 (&r)[4]) {
    if (valid >= 32) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = __ldg(q + i);
    } else {
        const unsigned short* e = reinterpret_cast<const unsigned short*>(p);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint32_t lo = 2 * j < valid ? e[2 * j] : 0u;
            const uint32_t hi = 2 * j + 1 < valid ? e[2 * j + 1] : 0u;
            w[j] = lo | (hi << 16);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

__device__ __forceinline__ void unpack32(const uint4 (&r)[4], float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Writes 32 floats as bf16 into half `half` (bytes 64*half .. 64*half+63)
// of this thread's 128-byte staging row at `row_addr`, in the 128-byte
// swizzle: 16-byte piece c of row r sits at piece position c ^ (r % 8).
__device__ __forceinline__ void stage_row(uint32_t row_addr, int half, uint32_t swz,
                                          const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t piece = static_cast<uint32_t>(half * 4 + j);
        st_shared_v4(row_addr + ((piece ^ swz) << 4), pack_bf16x2(v[8 * j + 0], v[8 * j + 1]),
                     pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    }
}

// Butterfly reduce-scatter over the warp: on return lane l holds the sum of
// v[l] over all 32 lanes (31 shuffles for 32 columns).
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
        }
    }
    return v[0];
}

// --------------------------------------------------------------- the kernel

template <bool A_MN, bool B_MN, int EPI, bool PAIR, int EW, int TN>
__global__ void __launch_bounds__(32 * (EW + 2), 1)
    tcgen05_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO0,  // output (Z for EPI_BIAS_GELU)
                        const __grid_constant__ CUtensorMap tmO1,  // H for EPI_BIAS_GELU
                        const GemmArgs p) {
    using G = Geometry<PAIR, EW, TN>;
    static_assert(!(G::WIDE && EPI == EPI_PARTIAL), "wide tiles store whole sums");
    constexpr int PRODUCER_WARP = EW, MMA_WARP = EW + 1;
    // Every CTA of this persistent grid is resident from the start, so the
    // next kernel on the stream may begin launching at once: its CTAs take
    // SMs as ours leave and run their set-up while our last tiles finish.
    pdl_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzle atoms repeat every 1024 B: align the ring to 1 KiB.
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint8_t* ring_a = smem;
    uint8_t* ring_b = smem + G::STAGES * G::A_STAGE_BYTES;
    uint8_t* staging = smem + G::STAGES * G::STAGE_BYTES;  // 1 KiB aligned
    uint8_t* bar_area = staging + G::STAGING_BYTES;
    const uint32_t tile_resp = smem_u32(bar_area);  // [kTileSlots] 16-byte scheduler responses
    uint64_t* bars = reinterpret_cast<uint64_t*>(bar_area + 16 * kTileSlots);
    uint64_t* full = bars;                      // stage loaded  (STAGES)
    uint64_t* empty = bars + G::STAGES;         // stage drained (STAGES)
    uint64_t* acc_full = bars + 2 * G::STAGES;  // accumulator ready (2)
    uint64_t* acc_empty = acc_full + 2;         // accumulator read  (2)
    uint64_t* drain = acc_empty + 2;            // teardown          (1)
    uint64_t* tile_full = drain + 1;            // scheduler response landed (kTileSlots)
    uint64_t* tile_empty = tile_full + kTileSlots;  // every reader has read it (kTileSlots)
    uint32_t* misc = reinterpret_cast<uint32_t*>(tile_empty + kTileSlots);
    volatile uint32_t* abort_flag = misc + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // In a pair, CTA rank 0 (the leader) issues the MMAs for both; rank r
    // holds accumulator rows 128r..128r+127 and B rows 128r..128r+127.
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], PAIR ? 2 * EW : EW);  // one arrival per epilogue warp
        }
        mbar_init(drain, 1);
        for (int s = 0; s < kTileSlots; ++s) {
            mbar_init(&tile_full[s], 1);  // this CTA's producer expects the 16 bytes
            // readers of a response: each CTA's producer and epilogue warps, the MMA thread
            mbar_init(&tile_empty[s], PAIR ? 2 * (1 + EW) + 1 : (1 + EW) + 1);
        }
        misc[1] = 0u;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&misc[0], TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&misc[0], TMEM_COLS);
            tmem_relinquish();
        }
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmO0);
        if (EPI == EPI_BIAS_GELU) prefetch_tmap(&tmO1);
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();  // the peer's barriers exist before anyone signals them
    else
        __syncthreads();
    tc_fence_after();
    // Set-up (barriers, TMEM, descriptor prefetch) touched no global memory;
    // from here on this kernel reads what the previous kernel wrote and
    // writes what it may still read, so it waits for that kernel to finish.
    pdl_wait();
    const uint32_t tmem_base = misc[0];
    const int total_kb = p.shard_mode == SHARD_K ? p.k_blocks * p.shards : p.k_blocks;

    // The work units of this CTA (pair), in order.  Static: unit, unit +
    // units, ...  Dynamic: unit (its own launch), then for i = 0, 1, ...
    // the unit whose launch the leader's producer cancelled with request i,
    // answered in slot i % kTileSlots of every CTA of the pair; readers
    // release the slot on the leader's tile_empty.  -1: no more units.
    constexpr int kCluster = PAIR ? 2 : 1;
    const bool dyn = p.dynamic_tiles != 0;
    const uint32_t tile_empty_leader =
        PAIR ? map_to_cta(smem_u32(tile_empty), 0) : smem_u32(tile_empty);
    // the unit after the one finished with response i (one thread reads)
    auto next_unit = [&](int tile, int i, bool& ok) -> int {
        if (!dyn) return tile + units < p.num_tiles ? tile + units : -1;
        const int slot = i % kTileSlots;
        if (!wait_bounded<true>(&tile_full[slot], static_cast<uint32_t>(i / kTileSlots) & 1u,
                                abort_flag, p.status)) {
            ok = false;
            return -1;
        }
        const int x = clc_response_ctaid_x(tile_resp + 16u * slot);
        if constexpr (PAIR)
            mbar_arrive_cluster(tile_empty_leader + 8u * slot);
        else
            mbar_arrive(&tile_empty[slot]);
        return x < 0 ? -1 : x / kCluster;
    };

    if (warp == PRODUCER_WARP) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;  // per-stage bits of the last issue
            const uint32_t ring_a_u = smem_u32(ring_a), ring_b_u = smem_u32(ring_b);
            // stage barriers as seen by the TMA: the leader's in a pair
            const uint32_t full_u = PAIR ? map_to_cta(smem_u32(full), 0) : smem_u32(full);
            const bool split_k = p.shard_mode == SHARD_K;
            bool run = true;
            int pending = -1;  // a scheduler request whose answer this thread has not read
            for (int tile = unit, i = 0; tile >= 0 && run; ++i) {
                if (dyn) {
                    // ask for the unit after this one now; the answer is read
                    // once this unit's loads are issued
                    const int slot = i % kTileSlots;
                    if (rank == 0) {
                        if (i >= kTileSlots &&
                            !wait_bounded<true>(&tile_empty[slot],
                                                static_cast<uint32_t>(i / kTileSlots - 1) & 1u,
                                                abort_flag, p.status))
                            break;
                        fence_proxy_async_smem();  // earlier reads of the slot come first
                        mbar_arrive_expect_tx(&tile_full[slot], 16);
                        if constexpr (PAIR)
                            clc_try_cancel_multicast(tile_resp + 16u * slot, smem_u32(&tile_full[slot]));
                        else
                            clc_try_cancel(tile_resp + 16u * slot, smem_u32(&tile_full[slot]));
                    } else {
                        mbar_arrive_expect_tx(&tile_full[slot], 16);  // the leader's answer lands here too
                    }
                    pending = i;
                }
                const TileCoord tc = decode_tile<G::TILE_M, G::TILE_N>(tile, p);
                const int a_row0 = tc.m0 + static_cast<int>(rank) * BM;
                const int b_row0 = tc.n0 + static_cast<int>(rank) * G::B_ROWS;
                // this unit's k-blocks [kb_begin, kb_end) and where they start
                const int kb_begin = tc.ks * total_kb / p.k_splits;
                const int kb_end = (tc.ks + 1) * total_kb / p.k_splits;
                int s = tc.s, kb_in_shard = kb_begin;  // shard of the k range
                if (split_k) {                          // SHARD_K walks the shards
                    s = kb_begin / p.k_blocks;
                    kb_in_shard = kb_begin - s * p.k_blocks;
                }
                int k0 = kb_in_shard * BK;
                bool ok = true;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bounded<true>(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    // in a pair both CTAs' bytes complete the leader's barrier
                    if (!PAIR || rank == 0)
                        mbar_arrive_expect_tx(&full[stage], PAIR ? 2 * G::STAGE_BYTES : G::STAGE_BYTES);
                    const uint32_t bar = full_u + stage * 8;
                    load_operand<A_MN, BM, PAIR>(&tmA, bar, ring_a_u + stage * G::A_STAGE_BYTES,
                                                 p.a_on, a_row0, k0, s, p.a_mn4);
                    load_operand<B_MN, G::B_ROWS, PAIR>(&tmB, bar, ring_b_u + stage * G::B_STAGE_BYTES,
                                                        p.b_on, b_row0, k0, s, p.b_mn4);
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    k0 += BK;
                    if (++kb_in_shard == p.k_blocks) {  // next shard's k range
                        kb_in_shard = 0;
                        k0 = 0;
                        ++s;
                    }
                    if (++stage == G::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tile = next_unit(tile, i, run);
                if (run) pending = -1;
            }
            // A scheduler answer still on its way lands before the CTA may exit.
            if (pending >= 0)
                wait_drain(&tile_full[pending % kTileSlots],
                           static_cast<uint32_t>(pending / kTileSlots) & 1u, p.status);
            // Every copy this thread started lands before the CTA may exit.  A
            // pair's copies complete on the leader's barriers, so there the
            // stage's release by the MMA (which waited for them) is awaited.
            for (int s = 0; s < G::STAGES; ++s) {
                if (!(issued & (1u << s))) continue;
                if constexpr (PAIR)
                    wait_drain(&empty[s], (issued_phase >> s) & 1u, p.status);
                else
                    wait_drain(&full[s], (issued_phase >> s) & 1u, p.status);
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(G::TILE_M, BN, A_MN, B_MN);
            const uint64_t a_desc0 = operand_desc<A_MN>(smem_u32(ring_a));
            const uint64_t b_desc0 = operand_desc<B_MN>(smem_u32(ring_b));
            int stage = 0;
            uint32_t phase = 0;
            int count = 0;
            for (int tile = unit; tile >= 0; ++count) {
                const int acc = G::ACCS == 2 ? (count & 1) : 0;
                const uint32_t acc_phase = G::ACCS == 2 ? (count >> 1) & 1 : count & 1;
                if (!wait_bounded<true>(&acc_empty[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                const int ks = p.k_splits > 1 ? tile / p.base_tiles : 0;
                const int kb_begin = ks * total_kb / p.k_splits;
                const int kb_end = (ks + 1) * total_kb / p.k_splits;
                bool ok = true;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bounded<true>(&full[stage], phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = a_desc0 + ((stage * G::A_STAGE_BYTES) >> 4);
                    const uint64_t bd = b_desc0 + ((stage * G::B_STAGE_BYTES) >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint32_t accum = (kb != kb_begin || kk != 0) ? 1u : 0u;
                        if constexpr (PAIR) {
                            tc_mma_f16_pair(d_tmem, ad + kk * desc_k_step<A_MN>(),
                                            bd + kk * desc_k_step<B_MN>(), idesc, accum);
                            // the second half of each CTA's B rows into
                            // accumulator columns BN..2BN-1 (same A)
                            if constexpr (G::WIDE)
                                tc_mma_f16_pair(d_tmem + BN, ad + kk * desc_k_step<A_MN>(),
                                                bd + (((BN / 2) * BK * 2) >> 4) + kk * desc_k_step<B_MN>(),
                                                idesc, accum);
                        } else
                            tc_mma_f16(d_tmem, ad + kk * desc_k_step<A_MN>(),
                                       bd + kk * desc_k_step<B_MN>(), idesc, accum);
                    }
                    // frees the stage (in both CTAs of a pair) when these MMAs finish
                    if constexpr (PAIR)
                        tc_commit_pair_multicast(&empty[stage], 0x3);
                    else
                        tc_commit(&empty[stage]);
                    if (++stage == G::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    tc_commit_pair_multicast(&acc_full[acc], 0x3);
                else
                    tc_commit(&acc_full[acc]);
                bool run = true;
                tile = next_unit(tile, count, run);
                if (!run) break;
            }
            // No MMA may still be writing TMEM when it is released.
            if constexpr (PAIR)
                tc_commit_pair(drain);
            else
                tc_commit(drain);
            wait_drain(drain, 0, p.status);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------- epilogue
        // Warp w owns accumulator rows 32q..32q+31 (q = w % 4, its TMEM lane
        // quadrant) and the NBLK 64-column blocks from column 64 cb0 on.
        // Per 64-column block: TMEM -> registers -> fused math -> bf16 rows
        // in a swizzled staging buffer -> one TMA store of the 32 x 64 block
        // (full lines; the tensor map clips rows and columns outside the
        // shard).  Two buffers per warp let a block be written while the
        // previous one is still being stored.
        const int q = warp & 3;
        constexpr int NBLK = G::TILE_N / 64 / (EW / 4);
        const int cb0 = (warp >> 2) * NBLK;
        // Output 64-column block of accumulator block c.  Wide tiles: MMA h
        // (columns 256h..256h+255) reads B rows 128h..128h+127 of each CTA,
        // and CTA r holds the tile's B rows 256r..256r+255, so accumulator
        // blocks 2, 3 hold output blocks 4, 5 and 4, 5 hold 2, 3.
        auto out_blk = [](int c) -> int {
            return G::WIDE ? ((c & 1) | (((c >> 1) & 1) << 2) | (((c >> 2) & 1) << 1)) : c;
        };
        const uint32_t release_bar =
            PAIR ? map_to_cta(smem_u32(&acc_empty[0]), 0) : smem_u32(&acc_empty[0]);
        const uint32_t buf_base = smem_u32(staging) + static_cast<uint32_t>(warp) * 2u * EPI_BUF_BYTES;
        const uint32_t my_row = static_cast<uint32_t>(lane) * 128u;
        const uint32_t swz = static_cast<uint32_t>(lane & 7);
        uint32_t seq = 0;  // stores committed so far: selects the buffer
        int count = 0;
        for (int tile = unit; tile >= 0; ++count) {
            const TileCoord tc = decode_tile<G::TILE_M, G::TILE_N>(tile, p);
            const int acc = G::ACCS == 2 ? (count & 1) : 0;
            const uint32_t acc_phase = G::ACCS == 2 ? (count >> 1) & 1 : count & 1;

            const int m_cta = tc.m0 + static_cast<int>(rank) * BM;  // first row of this CTA
            const int row0 = m_cta + q * 32;                           // first row of this warp
            const int m = row0 + lane;                                 // row inside the shard
            const bool row_ok = m < p.M;
            long long grow = m, gcol0 = tc.n0;
            if (p.shard_mode == SHARD_N) gcol0 += static_cast<long long>(tc.s) * p.N;
            if (p.shard_mode == SHARD_M) grow += static_cast<long long>(tc.s) * p.M;
            // The row operand of the fused math (Z for GeLU', the residual) and
            // the bias do not depend on the accumulator: their first 32
            // columns are requested before the wait, and each 32-column
            // block's loads are issued one block ahead of their use, so their
            // latency overlaps TMEM reads and the previous block's math.
            constexpr bool kAux = EPI == EPI_DGELU || EPI == EPI_BIAS_RESIDUAL;
            constexpr bool kBias = EPI == EPI_BIAS_GELU || EPI == EPI_BIAS_RESIDUAL || EPI == EPI_BIAS;
            uint4 aux_cur[4], aux_nxt[4], bias_cur[4], bias_nxt[4];
            if constexpr (kAux) {
                const int v0 = row_ok ? min(32, p.N - (tc.n0 + out_blk(cb0) * 64)) : 0;
                load_raw32(p.aux + grow * p.ld_aux + gcol0 + out_blk(cb0) * 64, v0, aux_cur);
            }
            if constexpr (kBias)  // the same 32 values for every lane (broadcast)
                load_raw32(p.bias + gcol0 + out_blk(cb0) * 64, min(32, p.N - (tc.n0 + out_blk(cb0) * 64)),
                           bias_cur);
            if (!warp_wait_bounded<true>(&acc_full[acc], acc_phase, abort_flag, p.status)) break;
            tc_fence_after();

            if constexpr (EPI == EPI_PARTIAL) {
                // fp32 accumulator blocks of 32 rows x 32 columns (128 B rows)
#pragma unroll 1
                for (int cc = 0; cc < 2 * NBLK; ++cc) {
                    const int c = 2 * cb0 + cc;
                    const int n = tc.n0 + c * 32;
                    const uint32_t buf = buf_base + (seq & 1u) * EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                    uint32_t r[32];
                    tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 32, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(buf + my_row + ((static_cast<uint32_t>(j) ^ swz) << 4), r[4 * j],
                                     r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (row0 < p.M && n < p.N) {  // warp-uniform
                        if (lane == 0) {
                            if (p.partial_compact)
                                tma_store_3d(&tmO0, buf, n - tc.n0, row0 - tc.m0, tc.slot);
                            else
                                tma_store_3d(&tmO0, buf, n, row0, tc.ks);
                            bulk_commit_group();
                        }
                        ++seq;
                    }
                }
            } else {
#pragma unroll 1
            for (int cc = 0; cc < NBLK; ++cc) {
                const int c = cb0 + cc;
                const int n64 = tc.n0 + out_blk(c) * 64;
                uint32_t buf0, buf1;
                if constexpr (EPI == EPI_BIAS_GELU) {
                    // Z in buffer 0, H in buffer 1, each block's two stores
                    // committed as two groups (Z first): here only Z's store
                    // must have read its buffer; H's may still be reading
                    // until the first H row of this block is staged
                    buf0 = buf_base;
                    buf1 = buf_base + EPI_BUF_BYTES;
                    if (lane == 0) bulk_wait_group_read<1>();
                } else {
                    buf0 = buf_base + (seq & 1u) * EPI_BUF_BYTES;
                    buf1 = buf0;
                    if (lane == 0) bulk_wait_group_read<1>();
                }
                __syncwarp();  // the buffer's previous store has read it
                // Both 32-column halves of the block are read from TMEM before
                // one wait, so each block pays the load latency once.
                uint32_t r2[2][32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 64, r2[0]);
                tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c * 64 + 32,
                          r2[1]);
                tmem_wait_ld();
                if (cc == NBLK - 1) {
                    // every column of this warp's part of the accumulator is in
                    // registers: once all epilogue warps are here the MMA may
                    // start the tile after next on it while the last block is
                    // staged and stored
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (PAIR)
                            mbar_arrive_cluster(release_bar + acc * 8);
                        else
                            mbar_arrive(&acc_empty[acc]);
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int n = n64 + half * 32;
                    const bool more = cc * 64 + half * 32 + 32 < NBLK * 64;  // another block follows
                    // tile column of the next 32-column chunk
                    const int nxt = half == 0 ? out_blk(c) * 64 + 32 : (more ? out_blk(c + 1) * 64 : 0);
                    if constexpr (kAux) {
                        if (more) {
                            const int vn = row_ok ? min(32, p.N - (tc.n0 + nxt)) : 0;
                            load_raw32(p.aux + grow * p.ld_aux + gcol0 + nxt, vn, aux_nxt);
                        }
                    }
                    if constexpr (kBias) {
                        if (more)
                            load_raw32(p.bias + gcol0 + nxt, min(32, p.N - (tc.n0 + nxt)), bias_nxt);
                    }
                    const uint32_t(&r)[32] = r2[half];
                    const int cvalid = min(32, p.N - n);  // columns inside the shard
                    const int valid = row_ok ? cvalid : 0;
                    const long long gcol = gcol0 + out_blk(c) * 64 + half * 32;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);

                    if constexpr (EPI == EPI_BIAS_GELU) {
                        {
                            float b[32];
                            unpack32(bias_cur, b);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] += b[i];
                        }
                        if (!p.skip_o0) stage_row(buf0 + my_row, half, swz, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
                        if (half == 0) {
                            if (lane == 0) bulk_wait_group_read<0>();  // the previous H store
                            __syncwarp();
                        }
                        stage_row(buf1 + my_row, half, swz, v);
                    } else if constexpr (EPI == EPI_BIAS_RESIDUAL) {
                        if (valid > 0) {
                            float b[32], res[32];
                            unpack32(bias_cur, b);
                            unpack32(aux_cur, res);
                            if (p.drop.threshold == 0u) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] += b[i] + res[i];
                            } else {
                                // Y = residual + keep * (P + b2) / (1 - p); element
                                // e = row * h + col, counters offset + e (4 per block)
                                const uint64_t g0 = p.drop.offset +
                                                    static_cast<uint64_t>(grow * p.ld_aux + gcol);
#pragma unroll
                                for (int q4 = 0; q4 < 8; ++q4) {
                                    const uint32_t keep =
                                        dropout_keep4(p.drop.seed, g0 + 4 * q4, p.drop.threshold);
#pragma unroll
                                    for (int j = 0; j < 4; ++j) {
                                        const int i = 4 * q4 + j;
                                        v[i] = res[i] + (((keep >> j) & 1u) ? (v[i] + b[i]) * p.drop.scale
                                                                            : 0.0f);
                                    }
                                }
                            }
                        }
                        stage_row(buf0 + my_row, half, swz, v);
                    } else if constexpr (EPI == EPI_BIAS) {
                        {
                            float b[32];
                            unpack32(bias_cur, b);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] += b[i];
                        }
                        stage_row(buf0 + my_row, half, swz, v);
                    } else if constexpr (EPI == EPI_DGELU) {
                        float z[32];
                        unpack32(aux_cur, z);
                        if (valid >= 32) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] *= gelu_tanh_grad(z[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                v[i] = i < valid ? v[i] * gelu_tanh_grad(z[i]) : 0.0f;
                        }
                        stage_row(buf0 + my_row, half, swz, v);
                        // db1 partial: lane l gets column n+l summed over this warp's 32 rows;
                        // one partial row per 32-row block of the shard's rows.
                        const float cs = warp_column_sums(v, lane);
                        if (m_cta < p.M && lane < cvalid)
                            p.colsum[(static_cast<long long>(m_cta / BM) * 4 + q) * p.ld_colsum +
                                     gcol + lane] = cs;
                    } else {
                        stage_row(buf0 + my_row, half, swz, v);
                    }
                    if constexpr (kAux) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) aux_cur[i] = aux_nxt[i];
                    }
                    if constexpr (kBias) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) bias_cur[i] = bias_nxt[i];
                    }
                }
                fence_proxy_async_smem();  // staged rows visible to the TMA store
                __syncwarp();
                // Blocks wholly outside the shard are not stored.  Buffers
                // alternate with the committed stores only, so the wait above
                // (at most one store still reading) always covers the buffer.
                const bool store = row0 < p.M && n64 < p.N;  // warp-uniform
                if (store) {
                    if (lane == 0) {
                        int c0, c1, c2;
                        tma_coords(p.o_on, n64, row0, tc.s, c0, c1, c2);
                        if (EPI != EPI_BIAS_GELU || !p.skip_o0) {
                            tma_store_3d(&tmO0, buf0, c0, c1, c2);
                            bulk_commit_group();
                        }
                        if constexpr (EPI == EPI_BIAS_GELU) {
                            tma_store_3d(&tmO1, buf1, c0, c1, c2);
                            bulk_commit_group();
                        }
                    }
                    ++seq;
                }
            }
            }
            if constexpr (EPI == EPI_PARTIAL) {
                // TMEM of this accumulator may be overwritten from here on (the
                // other epilogues release it after their last TMEM read)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(release_bar + acc * 8);
                    else
                        mbar_arrive(&acc_empty[acc]);
                }
            }
            // the next unit: lane 0 reads it, the warp follows
            bool run = true;
            int nxt = -1;
            if (lane == 0) nxt = next_unit(tile, count, run);
            nxt = __shfl_sync(0xFFFFFFFFu, nxt, 0);
            const uint32_t go = __shfl_sync(0xFFFFFFFFu, run ? 1u : 0u, 0);
            __syncwarp();
            if (!go) break;
            tile = nxt;
        }
        if (lane == 0) bulk_wait_group<0>();  // every output store has completed
        __syncwarp();
    }

    tc_fence_before();
    if constexpr (PAIR) {
        cluster_sync();  // every remote arrive and multicast commit has landed
        if (warp == MMA_WARP) {
            tc_fence_after();
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        }
        cluster_sync();
    } else {
        __syncthreads();
        if (warp == MMA_WARP) {
            tc_fence_after();
            tmem_dealloc(tmem_base, TMEM_COLS);
        }
    }
}

}  // namespace tpmlp
