// capi.cu -- the C ABI of the tensor-parallel MLP block (include/tpmlp.h):
// argument checks, tensor-map construction, tile-space set-up and launches,
// plus the column-sum (bias-gradient) kernels and the bounded-wait self-test.
//
// The block is the Megatron-LM MLP with the column-then-row split ("Megatron-
// LM: Tensor Model Parallel", charles2530.github.io, section "MLP: Column
// Parallel first, then Row Parallel", Figure 3a; "f / g Operators", Figure 4).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/tpmlp.h"
#include "kernels.h"

#define TPMLP_API extern "C" __attribute__((visibility("default")))

namespace tpmlp {

// Device status words: [0] a kernel writes a nonzero code when a bounded
// wait gives up (tpmlp_device_status() reads and clears it); [1] the site of
// the first wait that gave up, where the kernel names one
// (tpmlp_device_wait_site() reads and clears it).
__device__ int g_status_word[2];

namespace {

thread_local int t_last_cuda_error = 0;
thread_local int t_last_launches = 0;

// ------------------------------------------------------------- driver hooks

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

struct DeviceInfo {
    int sms = 0;
    int* status = nullptr;
    bool ok = false;
    // The tail-split cost model's rates, from the device's attributes:
    // a CTA pair's dense bf16 flops per ns and the DRAM bytes per ns.
    double pair_flops_per_ns = 0.0;
    double dram_bytes_per_ns = 0.0;
};

// A CTA pair's tensor cores do 2 x 4096 bf16 multiply-adds a clock.  The
// planner takes 0.58 of that at the peak clock as a pair's sustained rate
// inside a long GEMM step (1.5 PFLOP/s over GB300's 76 pairs at 2.07 GHz:
// the clock settles near 1.5 GHz under the 1.4 kW cap, and a tile's fill
// and epilogue cost the rest), and 0.8 of the DRAM's nominal rate (a copy
// reaches 6.77 of 8.2 TB/s).  The ratios were calibrated on GB300; the
// attributes carry the SM count, clock and memory of whatever device runs.
constexpr double kSustainedRateRatio = 0.58;
constexpr double kDramEfficiency = 0.8;

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};
std::mutex g_dev_mutex;

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return TPMLP_ERR_LAUNCH;
}

// Once per device: SM count, compute capability 10.3, status-word address.
int device_info(DeviceInfo& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TPMLP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo d;
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e);
        d.ok = (major == 10 && minor == 3);
        int clock_khz = 0, mem_khz = 0, bus_bits = 0;
        if ((e = cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&mem_khz, cudaDevAttrMemoryClockRate, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&bus_bits, cudaDevAttrGlobalMemoryBusWidth, dev)) != cudaSuccess)
            return fail_cuda(e);
        // flops per ns = 2 SMs x 8192 flops a clock x GHz; DRAM: double data rate
        d.pair_flops_per_ns = 2.0 * 8192.0 * (clock_khz * 1e-6) * kSustainedRateRatio;
        d.dram_bytes_per_ns = 2.0 * (mem_khz * 1e-6) * (bus_bits / 8.0) * kDramEfficiency;
        if (d.ok) {
            e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
            if (e != cudaSuccess) return fail_cuda(e);
        }
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    out = g_dev[dev];
    return out.ok ? TPMLP_OK : TPMLP_ERR_UNSUPPORTED;
}

// --------------------------------------------------------- argument checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(int T, int h, int F, int t) {
    if (T < 0 || h < 8 || F < 8 || t < 1 || t > TPMLP_MAX_SHARDS) return TPMLP_ERR_SHAPE;
    if (F % t != 0 || h % 8 != 0 || (F / t) % 8 != 0) return TPMLP_ERR_SHAPE;
    return TPMLP_OK;
}

template <typename... P>
bool any_null(P... p) {
    return ((p == nullptr) || ...);
}

template <typename... P>
bool all_aligned(P... p) {
    return (aligned16(p) && ...);
}

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// ------------------------------------------------------------- tensor maps

// 3-D tensor map over a row-major bf16 matrix [rows, cols] (rows `ld`
// elements apart; ld = 0: cols) whose shard index (t shards) sits on the
// contiguous dimension (ON_CONTIG: dims {cols/t, t, rows}), on the row
// dimension (ON_ROWS: dims {cols, rows/t, t}) or nowhere (dims {cols, rows,
// 1}).  Box: 64 contiguous elements (128 bytes, the swizzle width) by
// box_rows rows.
int make_map(CUtensorMap* m, const void* ptr, long long rows, long long cols, int t, int on,
             int box_rows, long long ld = 0) {
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(ld > 0 ? ld : cols) * 2;
    if (on == ON_CONTIG) {
        const long long cs = cols / t;
        dims[0] = cs; dims[1] = t; dims[2] = rows;
        // one shard: the middle dimension has extent 1 and its stride is unused
        strides[0] = t > 1 ? static_cast<cuuint64_t>(cs) * 2 : row_bytes; strides[1] = row_bytes;
        box[0] = 64; box[1] = 1; box[2] = box_rows;
    } else if (on == ON_ROWS) {
        const long long rs = rows / t;
        dims[0] = cols; dims[1] = rs; dims[2] = t;
        strides[0] = row_bytes; strides[1] = static_cast<cuuint64_t>(rs) * row_bytes;
        box[0] = 64; box[1] = box_rows; box[2] = 1;
    } else {
        dims[0] = cols; dims[1] = rows; dims[2] = 1;
        strides[0] = row_bytes; strides[1] = static_cast<cuuint64_t>(rows) * row_bytes;
        box[0] = 64; box[1] = box_rows; box[2] = 1;
    }
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return TPMLP_ERR_LAUNCH;
    }
    return TPMLP_OK;
}

// fp32 map over a [splits, rows, cols] partial-sum workspace: dims {cols, rows,
// splits}, 32 x 32 boxes (128-byte rows, 128-byte swizzle).
int make_partial_map(CUtensorMap* m, void* ptr, long long rows, long long cols, int splits) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(splits)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 4,
                             static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols) * 4};
    cuuint32_t box[3] = {32, 32, 1}, estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return TPMLP_ERR_LAUNCH;
    }
    return TPMLP_OK;
}

// One GEMM operand: a row-major [rows, cols] matrix (rows ld elements apart;
// 0: cols), K-major or MN-major in the product, with its shard placement.
struct Operand {
    const void* ptr;
    long long rows, cols;
    int on;
    bool mn_major;
    long long ld = 0;
};

// 4-D view of an MN-major operand, [rows = k, cols = mn] row-major with the
// shard index on `on` as in make_map: dims {64, k rows, mn / 64, shards},
// so that one box {64, BK, atoms, 1} holds `atoms` 64-wide MN atoms of a
// k-block, each 64 rows of 128 bytes, one after another (the layout the
// MN-major UMMA descriptor reads).  Only for MN extents (per shard) that are
// multiples of 64, so that no atom reaches past its shard or row.
int make_map_mn4(CUtensorMap* m, const void* ptr, long long rows, long long cols, int t, int on,
                 int atoms, long long ld) {
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4] = {64, static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(atoms), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(ld > 0 ? ld : cols) * 2;
    if (on == ON_CONTIG) {  // shards split the MN columns
        const long long cs = cols / t;
        dims[0] = 64; dims[1] = rows; dims[2] = cs / 64; dims[3] = t;
        strides[0] = row_bytes; strides[1] = 128; strides[2] = static_cast<cuuint64_t>(cs) * 2;
    } else if (on == ON_ROWS) {  // shards split the k rows
        const long long rs = rows / t;
        dims[0] = 64; dims[1] = rs; dims[2] = cols / 64; dims[3] = t;
        strides[0] = row_bytes; strides[1] = 128; strides[2] = static_cast<cuuint64_t>(rs) * row_bytes;
    } else {
        dims[0] = 64; dims[1] = rows; dims[2] = cols / 64; dims[3] = 1;
        strides[0] = row_bytes; strides[1] = 128; strides[2] = static_cast<cuuint64_t>(rows) * row_bytes;
    }
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return TPMLP_ERR_LAUNCH;
    }
    return TPMLP_OK;
}

// The operand's tensor map: K-major operands and MN-major ones of ragged
// MN extent as 3-D maps with one box per 64 rows (MN-major: per 64-wide
// atom); other MN-major operands as the 4-D view, one box per stage
// (*mn4 = 1).
int operand_map(CUtensorMap* m, const Operand& o, int t, int tile_rows, int* mn4) {
    *mn4 = 0;
    if (o.mn_major) {
        const long long mn = o.on == ON_CONTIG ? o.cols / t : o.cols;
        if (mn % 64 == 0 && tile_rows % 64 == 0 && (o.on != ON_ROWS || o.rows % t == 0)) {
            *mn4 = 1;
            return make_map_mn4(m, o.ptr, o.rows, o.cols, t, o.on, tile_rows / 64, o.ld);
        }
    }
    return make_map(m, o.ptr, o.rows, o.cols, t, o.on, o.mn_major ? BK : tile_rows, o.ld);
}

// 0: single-CTA kernel only, 1: CTA pairs unless the problem has very few
// tiles, 2: pairs always.
std::atomic<int> g_pair_mode{1};

// A pair loads half of each B tile per SM and keeps six stages in flight
// against a single CTA's four, which pays even when the pairs are fewer than
// the GPU's SM pairs: the row-parallel GEMMs of 64 tiles at T = 1024,
// h = 4096 ran 11-16 % faster on 64 pairs than on 128 single CTAs, and the
// 64-tile weight gradients of the GPT-2-medium block 6-11 %.  Below this
// many 256 x 256 tiles the single CTA's 128-row tiles occupy twice as many
// SMs, which the launch-bound calls of small blocks prefer.
constexpr int kPairMinTiles = 32;
// Epilogue warps of the dZ GEMM (the one GEMM with both forms): 0 = by the
// reduction's length (epi_warps_for), 4 or 8 = always that form.
std::atomic<int> g_epi_mode{0};

// Which of the library's kernels are launched as programmatic dependents of
// the kernel before them on the stream (their set-up overlaps its end): bit 0
// the GEMMs, bit 1 the other kernels; 0: plain stream order.
std::atomic<int> g_dependent_launch{3};

// 0: persistent GEMM grids with a static assignment of units to CTA pairs;
// 1: dynamic units through cluster launch control; 2 (default): dynamic for
// long reductions only (dynamic_units_for).
std::atomic<int> g_tile_scheduler{2};

// 0: 256 x 256 tiles per CTA pair; 1: 256 x 512 tiles for the K-major
// plain-store GEMMs (dX) where no split of the reduction applies.
std::atomic<int> g_wide_tiles{0};

// A pair that has to wait for the answer to its request for the next unit
// loses that time on every tile; over a long reduction (a tile of 192 or
// more k-blocks, 100 us and up) it is nothing, while keeping the tiles in
// flight together saves the DRAM re-reads of the static schedule's drift.
// Over short tiles (16-32 k-blocks, 4-11 us) the wait showed: the K = 1024
// GEMMs of GPT-2-medium were 4-10 % slower dynamic, the MT-NLG weight
// gradients (K = 2048) 2-3 %, while the four K >= 20480 GEMMs were 0.6-2.7 %
// faster and read a third less.
bool dynamic_units_for(long long total_kb) {
    const int mode = g_tile_scheduler.load(std::memory_order_relaxed);
    return mode == 1 || (mode == 2 && total_kb >= 192);
}

// A tile's mainloop lasts its reduction's k-blocks (512 clocks each for a
// CTA pair at the full MMA rate); its epilogue does not shrink with it.  The
// dZ GEMM's epilogue (a read of Z, GeLU', the db1 column sums) is the
// heaviest: with 16 k-blocks or fewer (K <= 1024) four warps bound the tile
// and eight, two per scheduler, hide each other's latencies (dZ of the
// GPT-2-medium block, K = 1024: 81.9 -> 73.7 us).  Elsewhere the stage the
// eight warps' staging buffers take costs more than they gain (measured 2-17 %
// slower on the other GEMMs and at longer K), so only that kernel has the form.
}  // namespace

bool dependent_launch() { return (g_dependent_launch.load(std::memory_order_relaxed) & 2) != 0; }

namespace {

int epi_warps_for(long long total_kb) {
    const int mode = g_epi_mode.load(std::memory_order_relaxed);
    if (mode == 4 || mode == 8) return mode;
    return total_kb <= 16 ? 8 : 4;
}

#ifndef TPMLP_BAND_BUDGET_MB
#define TPMLP_BAND_BUDGET_MB 16
#endif
constexpr long long kBandBudgetBytes = TPMLP_BAND_BUDGET_MB * (1LL << 20);
constexpr long long kBandMaxPanelBytes = 4LL << 20;

// Reduction length of one output tile (all shards' k ranges for SHARD_K).
long long K_total_of(const GemmArgs&, int K, int t, int mode) {
    return mode == SHARD_K ? 1LL * K * t : K;
}

// Fills the tile space of a GEMM with output extent M x N per shard.
void tile_space(GemmArgs& g, int M, int N, int K, int t, int mode, long long a_bytes,
                long long b_bytes, int tile_m, int tile_n = BN) {
    g.M = M;
    g.N = N;
    g.shards = t;
    g.shard_mode = mode;
    g.m_tiles = static_cast<int>(cdiv(M, tile_m));
    g.n_tiles = static_cast<int>(cdiv(N, tile_n));
    g.tile_n = tile_n;
    g.mt_total = g.m_tiles * (mode == SHARD_M ? t : 1);
    g.nt_total = g.n_tiles * (mode == SHARD_N ? t : 1);
    g.k_blocks = static_cast<int>(cdiv(K, BK));
    g.num_tiles = g.mt_total * g.nt_total;
    g.base_tiles = g.num_tiles;
    g.k_splits = 1;
    // Keep the larger operand's panels read once: walk the other operand's
    // tiles fastest so concurrent CTAs share the big panel through L2.
    g.raster_m_fastest = b_bytes >= a_bytes ? 1 : 0;
    // With a short reduction the panels are small and tiles finish quickly,
    // so the fast dimension's panels are re-read across waves: band them to
    // an L2-sized working set.  With a long reduction the concurrent tiles
    // walk K together and share each k-slab, so one band spans everything.
    const int fast_tiles = g.raster_m_fastest ? g.mt_total : g.nt_total;
    const long long panel = 2LL * (g.raster_m_fastest ? tile_m : tile_n) * K_total_of(g, K, t, mode);
    g.band = fast_tiles;
    if (panel <= kBandMaxPanelBytes && panel * fast_tiles > kBandBudgetBytes)
        g.band = static_cast<int>(std::max<long long>(1, kBandBudgetBytes / panel));
}

typedef cudaError_t (*Launcher)(const GemmMaps&, const GemmArgs&, int, bool, cudaStream_t);

// The output of one GEMM: row-major [rows, cols] over all shards; `ptr1` is
// the second output of the bias + GeLU epilogue (H), else null.
struct Output {
    void* ptr0;
    void* ptr1;
    long long rows, cols;
    int k_splits;  // > 1: ptr0 is an fp32 [k_splits, rows, cols] partial-sum workspace
};

// ------------------------------------------------------------ tail split
//
// A persistent GEMM over `tiles` output tiles on `units` CTA pairs runs
// ceil(tiles / units) rounds of tiles; when the last round is only partly
// full the rest of the GPU idles for a whole tile's time (640 tiles on 76
// pairs: 9 rounds for 8.42 rounds of work).  The tail split runs the first
// `main` tiles (whole rounds) as usual, then cuts each of the last X tiles'
// reduction into S contiguous k ranges computed by different pairs as fp32
// partial tiles, and a reduce kernel adds the S partials of each tile in k
// order and applies the fused epilogue (bias, residual, dropout).  Used for
// the row-parallel GEMMs, whose epilogue the reduce kernel can apply.

constexpr long long kTailTileFloats = 2LL * BM * BN;  // one 256 x 256 fp32 partial tile

struct TailPlan {
    long long main;  // tiles computed whole, a multiple of units
    long long X;     // tail tiles
    int S;           // k ranges per tail tile (1: no tail split)
};

// Estimated time of a plan: (main / units + ceil(X S / units) / S) rounds of
// a whole tile, plus the partial tiles' write and read at DRAM speed and two
// more launches.  A tile's time is its 2 x 256 x 256 x K flops at a CTA
// pair's rate under the power cap (pair_flops_per_ns; on GB300 ~19.7
// TFLOP/s a pair, 1.5 PFLOP/s over 76 pairs), the partial tiles' traffic at
// dram_bytes_per_ns (~6.5 TB/s).  Among X = rem, rem + units, rem + 2 units
// and S = 2..8 (at least 8 k-blocks per range; partials within ws_floats)
// the fastest plan is taken when it beats the plain schedule.  Rates of 0
// (no device) fall back to GB300's.
TailPlan plan_tail(long long tiles, long long total_kb, int units, long long ws_floats,
                   double pair_flops_per_ns = 0.0, double dram_bytes_per_ns = 0.0) {
    const double kPairFlopsPerNs =
        pair_flops_per_ns > 0.0 ? pair_flops_per_ns : 2.0 * 8192.0 * 2.07 * kSustainedRateRatio;
    const double kHbmBytesPerNs = dram_bytes_per_ns > 0.0 ? dram_bytes_per_ns : 6500.0;
    constexpr double kLaunchNs = 4000.0;
    TailPlan best{tiles, 0, 1};
    if (units <= 0 || tiles <= units || tiles % units == 0) return best;
    const double tile_ns = 2.0 * 2 * BM * BN * BK * static_cast<double>(total_kb) / kPairFlopsPerNs;
    const double base = static_cast<double>(cdiv(tiles, units)) * tile_ns;
    double best_t = base;
    const long long rem = tiles % units;
    for (long long X = rem; X <= tiles && X <= rem + 2LL * units; X += units) {
        for (int S = 2; S <= 8 && total_kb / S >= 8; ++S) {
            if (X * S * kTailTileFloats > ws_floats) break;
            const double rounds = static_cast<double>((tiles - X) / units) +
                                  static_cast<double>(cdiv(X * S, units)) / S;
            const double t = rounds * tile_ns + 2.0 * kLaunchNs +
                             2.0 * 4.0 * static_cast<double>(X * S * kTailTileFloats) / kHbmBytesPerNs;
            if (t < best_t - 1e-9) {
                best_t = t;
                best = TailPlan{tiles - X, X, S};
            }
        }
    }
    return best;
}

// What a tail split needs besides the GEMM itself: the same GEMM with the
// EPI_PARTIAL epilogue, a workspace for the partial tiles and the fused
// epilogue's operands for the reduce kernel.
struct TailSpec {
    Launcher partial_fn;
    void* ws;
    size_t ws_bytes;
    const tpmlp_bf16* bias;  // may be null (no epilogue: dX)
    const tpmlp_bf16* res;
    Dropout dr;
};

int launch_tail_reduce(const float* P, int S, const GemmArgs& g, long long first, long long X,
                       const TailSpec& ts, tpmlp_bf16* out, cudaStream_t st);

// fp32 map over X S compact partial tiles [X S, 256, 256]: 32 x 32 boxes.
int make_tail_map(CUtensorMap* m, void* ptr, long long slots) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(BN), static_cast<cuuint64_t>(2 * BM),
                          static_cast<cuuint64_t>(slots)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(BN) * 4,
                             static_cast<cuuint64_t>(2 * BM) * BN * 4};
    cuuint32_t box[3] = {32, 32, 1}, estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return TPMLP_ERR_LAUNCH;
    }
    return TPMLP_OK;
}

// One GEMM: M x N output per shard, K reduction (per shard for SHARD_K).
struct GemmShape {
    int M, N, K, t, mode;
    long long a_bytes, b_bytes;
};

int run_gemm(Launcher fn, const Operand& a, const Operand& b, const Output& out, GemmArgs& g,
             const GemmShape& sh, cudaStream_t st, const DeviceInfo& dev,
             const TailSpec* tail = nullptr) {
    const int pair_mode = g_pair_mode.load(std::memory_order_relaxed);
    GemmArgs probe = g;
    tile_space(probe, sh.M, sh.N, sh.K, sh.t, sh.mode, sh.a_bytes, sh.b_bytes, 2 * BM);
    const bool pair = pair_mode == 2 || (pair_mode == 1 && probe.num_tiles >= kPairMinTiles);
    const int tile_m = pair ? 2 * BM : BM;
    const bool wide = pair && fn == launch_dx && out.k_splits <= 1 &&
                      g_wide_tiles.load(std::memory_order_relaxed) == 1;
    const int tile_n = wide ? 2 * BN : BN;
    // When every shard boundary falls on a tile boundary (SHARD_N, SHARD_M)
    // or a k-block boundary (SHARD_K), the shards are runs of whole tiles of
    // the unsharded problem, visited in the same order: run it unsharded.
    GemmShape f = sh;
    Operand fa = a, fb = b;
    if (sh.t > 1 && ((sh.mode == SHARD_K && sh.K % BK == 0) ||
                     (sh.mode == SHARD_N && sh.N % tile_n == 0) ||
                     (sh.mode == SHARD_M && sh.M % tile_m == 0))) {
        if (sh.mode == SHARD_K) f.K = sh.K * sh.t;
        if (sh.mode == SHARD_N) f.N = sh.N * sh.t;
        if (sh.mode == SHARD_M) f.M = sh.M * sh.t;
        f.t = 1;
    }
    if (f.t == 1) {
        // One range: the tile loop needs no shard bookkeeping, and every map
        // takes the form {cols, 1, rows} (rows as the outer dimension, which
        // the tensor memory accelerator streams faster than {cols, rows, 1}).
        f.mode = SHARD_NONE;
        fa.on = fb.on = ON_CONTIG;
    }
    g.a_on = fa.on;
    g.b_on = fb.on;
    // Output maps carry the shard index where the output is split, so that
    // TMA stores clip each shard's ragged edge; 32-row x 64-column boxes.
    int o_t = 1;
    g.o_on = ON_CONTIG;
    if (f.mode == SHARD_N || f.mode == SHARD_M) {
        o_t = f.t;
        g.o_on = f.mode == SHARD_N ? ON_CONTIG : ON_ROWS;
    }
    tile_space(g, f.M, f.N, f.K, f.t, f.mode, f.a_bytes, f.b_bytes, tile_m, tile_n);
    if (g.num_tiles == 0) return TPMLP_OK;
    g.epi_warps = epi_warps_for(1LL * g.k_blocks * (f.mode == SHARD_K ? f.t : 1));
    g.dependent_launch = g_dependent_launch.load(std::memory_order_relaxed) & 1;
    g.dynamic_tiles = dynamic_units_for(1LL * g.k_blocks * (f.mode == SHARD_K ? f.t : 1)) ? 1 : 0;
    if (out.k_splits > 1) {
        g.k_splits = out.k_splits;
        g.num_tiles = g.base_tiles * out.k_splits;
    }
    alignas(64) GemmMaps maps;
    int rc = operand_map(&maps.a, fa, f.t, BM, &g.a_mn4);
    if (rc) return rc;
    rc = operand_map(&maps.b, fb, f.t, pair ? tile_n / 2 : BN, &g.b_mn4);
    if (rc) return rc;
    if (out.k_splits > 1)
        rc = make_partial_map(&maps.o0, out.ptr0, out.rows, out.cols, out.k_splits);
    else
        rc = make_map(&maps.o0, out.ptr0, out.rows, out.cols, o_t, g.o_on, 32);
    if (rc) return rc;
    rc = make_map(&maps.o1, out.ptr1 ? out.ptr1 : out.ptr0, out.rows, out.cols, o_t, g.o_on, 32);
    if (rc) return rc;
    g.status = dev.status;
    const int units = pair ? std::max(1, dev.sms / 2) : dev.sms;
    TailPlan plan{g.num_tiles, 0, 1};
    if (tail != nullptr && pair && !wide && out.k_splits <= 1 && tail->ws != nullptr)
        plan = plan_tail(g.num_tiles, 1LL * g.k_blocks * (f.mode == SHARD_K ? f.t : 1), units,
                         static_cast<long long>(tail->ws_bytes / sizeof(float)), dev.pair_flops_per_ns,
                         dev.dram_bytes_per_ns);
    GemmArgs gm = g;
    if (plan.S > 1) gm.num_tiles = gm.base_tiles = static_cast<int>(plan.main);  // whole rounds
    cudaError_t e = fn(maps, gm, gm.dynamic_tiles ? gm.num_tiles : std::min(gm.num_tiles, units),
                       pair, st);
    if (e != cudaSuccess) return fail_cuda(e);
    ++t_last_launches;
    if (plan.S <= 1) return TPMLP_OK;
    // the tail: X tiles x S k ranges into compact partial tiles, then the reduce
    GemmArgs gt = g;
    gt.tile_offset = static_cast<int>(plan.main);
    gt.base_tiles = static_cast<int>(plan.X);
    gt.k_splits = plan.S;
    gt.num_tiles = static_cast<int>(plan.X * plan.S);
    gt.partial_compact = 1;
    if ((rc = make_tail_map(&maps.o0, tail->ws, plan.X * plan.S))) return rc;
    maps.o1 = maps.o0;
    e = tail->partial_fn(maps, gt, gt.dynamic_tiles ? gt.num_tiles : std::min(gt.num_tiles, units),
                         pair, st);
    if (e != cudaSuccess) return fail_cuda(e);
    ++t_last_launches;
    return launch_tail_reduce(static_cast<const float*>(tail->ws), plan.S, g, plan.main, plan.X,
                              *tail, static_cast<tpmlp_bf16*>(out.ptr0), st);
}

GemmArgs blank_args() {
    GemmArgs g;
    std::memset(&g, 0, sizeof g);
    return g;
}

const __nv_bfloat16* cb(const tpmlp_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); }

// ------------------------------------------------------------ the six GEMMs

int column_gelu(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1, int T, int h,
                int F, int t, tpmlp_bf16* Z, tpmlp_bf16* H, cudaStream_t st, const DeviceInfo& d) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{T, f, h, t, SHARD_N, 1LL * T * h, 1LL * h * F};
    g.a_on = ON_NONE;
    g.b_on = ON_CONTIG;
    g.bias = cb(b1);
    Operand a{X, T, h, ON_NONE, false};
    Operand b{A, h, F, ON_CONTIG, true};
    g.skip_o0 = Z == nullptr;  // H only: Z is recomputed by the backward pass
    Output o{Z ? Z : H, H, T, F};
    return run_gemm(launch_column_gelu, a, b, o, g, sh, st, d);
}

// ----------------------------------------------------- split reductions

// The row-parallel GEMMs (a3, a7) have only ceil(T/256) x ceil(h/256) output
// tiles.  When that leaves SM pairs idle, each tile's k range (the shards, in
// order) is cut into `splits` contiguous runs computed by different CTA pairs
// as fp32 partial sums -- the pages' per-rank partials -- and a second kernel
// adds them in run order, then b2 and the residual.  `units` is the number of
// CTA pairs.  Returns 1 (no split) unless splitting saves >= 20 % of the waves.
int choose_splits(long long M, long long N, long long total_kb, int units) {
    const long long tiles = cdiv(M, 2 * BM) * cdiv(N, BN);
    if (units <= 0 || tiles <= 0) return 1;
    const double base = static_cast<double>(cdiv(tiles, units));
    double best = base;
    int best_s = 1;
    for (int sp = 2; sp <= 8 && total_kb / sp >= 8; ++sp) {
        const double c = static_cast<double>(cdiv(tiles * sp, units)) / sp;
        if (c < best - 1e-9) {
            best = c;
            best_s = sp;
        }
    }
    return best <= 0.8 * base ? best_s : 1;
}

// The row-parallel GEMMs' split, with the partial outputs counted: among 1..8
// splits, the one with the least estimated time -- rounds of a 1/sp tile at
// a pair's rate plus, for sp > 1, the fp32 partials' write and read (2 x 4
// sp M N bytes at DRAM speed) and the reduce launch -- when it beats the
// unsplit time by 5 % or more.  The rates are plan_tail's.
int choose_row_splits(long long M, long long N, long long total_kb, int units,
                      double pair_flops_per_ns = 0.0, double dram_bytes_per_ns = 0.0) {
    const long long tiles = cdiv(M, 2 * BM) * cdiv(N, BN);
    if (units <= 0 || tiles <= 0) return 1;
    const double flops_ns =
        pair_flops_per_ns > 0.0 ? pair_flops_per_ns : 2.0 * 8192.0 * 2.07 * kSustainedRateRatio;
    const double dram_ns = dram_bytes_per_ns > 0.0 ? dram_bytes_per_ns : 6500.0;
    constexpr double kLaunchNs = 4000.0;
    const double tile_ns = 2.0 * 2 * BM * BN * BK * static_cast<double>(total_kb) / flops_ns;
    const double base = static_cast<double>(cdiv(tiles, units)) * tile_ns;
    double best = base;
    int best_s = 1;
    for (int sp = 2; sp <= 8 && total_kb / sp >= 8; ++sp) {
        const double c = static_cast<double>(cdiv(tiles * sp, units)) * tile_ns / sp + kLaunchNs +
                         8.0 * sp * static_cast<double>(M) * static_cast<double>(N) / dram_ns;
        if (c < best - 1e-9) {
            best = c;
            best_s = sp;
        }
    }
    return best <= 0.95 * base ? best_s : 1;
}

// CTA pairs the split heuristic assumes when sizing workspaces (GB300: 152 SMs).
constexpr int kSizingPairs = 76;

long long row_total_kb(int F, int t) { return cdiv(F / t, BK) * t; }

// Floats of split-reduction workspace the row-parallel GEMMs of this shape
// use: a whole split, or else the partial tiles of a tail split.
size_t split_partial_floats(int T, int h, int F, int t) {
    const long long total_kb = row_total_kb(F, t);
    const int sp = choose_row_splits(T, h, total_kb, kSizingPairs);
    if (sp > 1) return static_cast<size_t>(sp) * T * h;
    const long long tiles = cdiv(T, 2 * BM) * cdiv(h, BN);
    const TailPlan p = plan_tail(tiles, total_kb, kSizingPairs, 1LL << 60);
    return p.S > 1 ? static_cast<size_t>(p.X * p.S * kTailTileFloats) : 0;
}

// The fused epilogue of the row-parallel GEMMs on 8 fp32 sums of elements
// i..i+7 of a row-major [., n] output: + bias[i % n] + res[i]; with dropout,
// res[i] + keep(i) * (sum + bias[i % n]) * scale; bias null: the sums alone.
// Returns them as bf16.
__device__ __forceinline__ uint4 finish8(float (&a)[8], long long i, int n,
                                         const __nv_bfloat16* __restrict__ bias,
                                         const __nv_bfloat16* __restrict__ res, const Dropout& dr) {
    if (bias != nullptr) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias + i % n));
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(res + i));
        const uint32_t bw[4] = {b.x, b.y, b.z, b.w}, rw[4] = {r.x, r.y, r.z, r.w};
        if (dr.threshold == 0u) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                a[2 * j] += __uint_as_float(bw[j] << 16) + __uint_as_float(rw[j] << 16);
                a[2 * j + 1] += __uint_as_float(bw[j] & 0xFFFF0000u) + __uint_as_float(rw[j] & 0xFFFF0000u);
            }
        } else {
            const uint32_t keep = dropout_keep4(dr.seed, dr.offset + i, dr.threshold) |
                                  (dropout_keep4(dr.seed, dr.offset + i + 4, dr.threshold) << 4);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t bb = (j & 1) ? (bw[j >> 1] & 0xFFFF0000u) : (bw[j >> 1] << 16);
                const uint32_t rr = (j & 1) ? (rw[j >> 1] & 0xFFFF0000u) : (rw[j >> 1] << 16);
                a[j] = __uint_as_float(rr) +
                       (((keep >> j) & 1u) ? (a[j] + __uint_as_float(bb)) * dr.scale : 0.0f);
            }
        }
    }
    uint4 o;
    o.x = pack_bf16x2(a[0], a[1]);
    o.y = pack_bf16x2(a[2], a[3]);
    o.z = pack_bf16x2(a[4], a[5]);
    o.w = pack_bf16x2(a[6], a[7]);
    return o;
}

// out[i] = finish8(sum_s P[s][i]), 8 elements a thread, P: [splits, count].
__global__ void __launch_bounds__(256)
    split_reduce_kernel(const float* __restrict__ P, int splits, long long count, int n,
                        const __nv_bfloat16* __restrict__ bias, const __nv_bfloat16* __restrict__ res,
                        Dropout dr, __nv_bfloat16* __restrict__ out) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // its inputs come from the kernel before it
    const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
    if (i >= count) return;
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = 0.0f;
    for (int sp = 0; sp < splits; ++sp) {
        const float4* q = reinterpret_cast<const float4*>(P + sp * count + i);
        const float4 x = __ldg(q), y = __ldg(q + 1);
        a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
        a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
    *reinterpret_cast<uint4*>(out + i) = finish8(a, i, n, bias, res, dr);
}

// The tail tiles of a tail split (plan_tail): tile `local` of X is output
// tile first + local of the GEMM's raster order; its S partial tiles sit in
// slots s X + local (s = 0..S-1, k order) of P, 256 x 256 fp32 each.  A
// thread adds 8 consecutive columns of one row over s in order and applies
// finish8; 32 CTAs cover a tile.
__global__ void __launch_bounds__(256)
    tail_reduce_kernel(const float* __restrict__ P, int S, GemmArgs g, int X,
                       const __nv_bfloat16* __restrict__ bias, const __nv_bfloat16* __restrict__ res,
                       Dropout dr, __nv_bfloat16* __restrict__ out) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // its inputs come from the kernel before it
    const int local = static_cast<int>(blockIdx.x >> 5);
    const int e = static_cast<int>(((blockIdx.x & 31u) * blockDim.x + threadIdx.x) * 8u);
    const int r = e / BN, c = e % BN;
    const TileCoord tc = decode_tile<2 * BM>(local, g);
    const int row = tc.m0 + r, col = tc.n0 + c;
    if (row >= g.M || col >= g.N) return;
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) a[j] = 0.0f;
    for (int sp = 0; sp < S; ++sp) {
        const float4* q = reinterpret_cast<const float4*>(
            P + (static_cast<long long>(sp) * X + local) * kTailTileFloats + e);
        const float4 x = __ldg(q), y = __ldg(q + 1);
        a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
        a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    }
    const long long i = static_cast<long long>(row) * g.N + col;
    *reinterpret_cast<uint4*>(out + i) = finish8(a, i, g.N, bias, res, dr);
}

int launch_tail_reduce(const float* P, int S, const GemmArgs& g, long long first, long long X,
                       const TailSpec& ts, tpmlp_bf16* out, cudaStream_t st) {
    GemmArgs r = g;
    r.tile_offset = static_cast<int>(first);
    r.base_tiles = static_cast<int>(X);
    cudaError_t e = launch_dependent(tail_reduce_kernel, dim3(static_cast<unsigned>(X * 32)),
                                     dim3(256), 0, st, P, S, r, static_cast<int>(X), cb(ts.bias),
                                     cb(ts.res), ts.dr, reinterpret_cast<__nv_bfloat16*>(out));
    if (e != cudaSuccess) return fail_cuda(e);
    ++t_last_launches;
    return TPMLP_OK;
}

int launch_split_reduce(const float* P, int splits, int T, int h, const tpmlp_bf16* bias,
                        const tpmlp_bf16* res, const Dropout& dr, tpmlp_bf16* out,
                        cudaStream_t st) {
    const long long count = 1LL * T * h;
    cudaError_t e = launch_dependent(split_reduce_kernel,
                                     dim3(static_cast<unsigned>(cdiv(count / 8, 256))), dim3(256), 0,
                                     st, P, splits, count, h, cb(bias), cb(res), dr,
                                     reinterpret_cast<__nv_bfloat16*>(out));
    if (e != cudaSuccess) return fail_cuda(e);
    ++t_last_launches;
    return TPMLP_OK;
}

// Splits to use for a row-parallel GEMM given the caller's workspace.
int row_splits(int T, int h, int F, int t, size_t ws_bytes, const DeviceInfo& d) {
    int sp = choose_row_splits(T, h, row_total_kb(F, t), d.sms / 2, d.pair_flops_per_ns,
                               d.dram_bytes_per_ns);
    const size_t per = sizeof(float) * static_cast<size_t>(T) * h;
    while (sp > 1 && static_cast<size_t>(sp) * per > ws_bytes) --sp;
    return sp;
}

// Splits of a weight gradient's token reduction (cdiv(T, BK) k-blocks) when
// its M x N output tiles leave CTA pairs idle (a small hidden size: dWo of
// h x h at h = 1024 has 16 tiles of 256 x 256), limited by the caller's
// workspace, which holds the splits' fp32 partial outputs.
int weight_splits(int T, long long M, long long N, size_t ws_bytes, const DeviceInfo& d) {
    int sp = choose_splits(M, N, cdiv(T, BK), d.sms / 2);
    const size_t per = sizeof(float) * static_cast<size_t>(M) * static_cast<size_t>(N);
    while (sp > 1 && static_cast<size_t>(sp) * per > ws_bytes) --sp;
    return sp;
}

// Floats of partial outputs a split weight gradient of this shape uses.
size_t weight_split_floats(int T, long long M, long long N) {
    const int sp = choose_splits(M, N, cdiv(T, BK), kSizingPairs);
    return sp > 1 ? static_cast<size_t>(sp) * static_cast<size_t>(M) * static_cast<size_t>(N) : 0;
}

int row_sum(const tpmlp_bf16* H, const tpmlp_bf16* B, const tpmlp_bf16* b2,
            const tpmlp_bf16* R, int T, int h, int F, int t, tpmlp_bf16* Y, void* ws,
            size_t ws_bytes, cudaStream_t st, const DeviceInfo& d, const Dropout& dr = Dropout{}) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{T, h, f, t, SHARD_K, 1LL * T * F, 1LL * F * h};
    g.a_on = ON_CONTIG;
    g.b_on = ON_ROWS;
    g.bias = cb(b2);
    g.aux = cb(R);
    g.ld_aux = h;
    g.drop = dr;
    Operand a{H, T, F, ON_CONTIG, false};
    Operand b{B, F, h, ON_ROWS, true};
    const int sp = ws ? row_splits(T, h, F, t, ws_bytes, d) : 1;
    if (sp == 1) {
        Output o{Y, nullptr, T, h, 1};
        const TailSpec ts{launch_row_partial, ws, ws_bytes, b2, R, dr};
        return run_gemm(launch_row_sum, a, b, o, g, sh, st, d, &ts);
    }
    Output o{ws, nullptr, T, h, sp};
    if (int rc = run_gemm(launch_row_partial, a, b, o, g, sh, st, d)) return rc;
    return launch_split_reduce(static_cast<const float*>(ws), sp, T, h, b2, R, dr, Y, st);
}

// dP = keep * dY * scale (bf16): the gradient that reaches the MLP's output
// through the dropout.  HBM-bound (4 bytes of traffic per element) with a
// Philox block per four elements of integer work beside it.  A thread owns
// kDropVec 16-byte pieces (8 elements each) spaced a CTA-width apart (so a
// warp's loads and stores stay coalesced), issues all their loads before
// any Philox block, and stores after: the loads' latency overlaps the
// arithmetic.  The tail (count not a multiple of the CTA's span) is masked.
constexpr int kDropThreads = 256;
constexpr int kDropVec = 4;

__global__ void __launch_bounds__(kDropThreads)
    dropout_grad_kernel(const __nv_bfloat16* __restrict__ dY, long long count, Dropout dr,
                        __nv_bfloat16* __restrict__ dP) {
    pdl_launch_dependents();  // the next kernel may begin its launch
    pdl_wait();               // its inputs come from the kernel before it
    const long long base = static_cast<long long>(blockIdx.x) * kDropThreads * kDropVec * 8;
    uint4 g[kDropVec];
#pragma unroll
    for (int v = 0; v < kDropVec; ++v) {
        const long long i = base + (static_cast<long long>(v) * kDropThreads + threadIdx.x) * 8;
        g[v] = i < count ? __ldg(reinterpret_cast<const uint4*>(dY + i)) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int v = 0; v < kDropVec; ++v) {
        const long long i = base + (static_cast<long long>(v) * kDropThreads + threadIdx.x) * 8;
        if (i >= count) continue;
        const uint32_t gw[4] = {g[v].x, g[v].y, g[v].z, g[v].w};
        const uint32_t keep = dropout_keep4(dr.seed, dr.offset + i, dr.threshold) |
                              (dropout_keep4(dr.seed, dr.offset + i + 4, dr.threshold) << 4);
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t gg = (j & 1) ? (gw[j >> 1] & 0xFFFF0000u) : (gw[j >> 1] << 16);
            a[j] = ((keep >> j) & 1u) ? __uint_as_float(gg) * dr.scale : 0.0f;
        }
        uint4 o;
        o.x = pack_bf16x2(a[0], a[1]);
        o.y = pack_bf16x2(a[2], a[3]);
        o.z = pack_bf16x2(a[4], a[5]);
        o.w = pack_bf16x2(a[6], a[7]);
        *reinterpret_cast<uint4*>(dP + i) = o;
    }
}

int dropout_grad(const tpmlp_bf16* dY, int T, int h, const Dropout& dr, tpmlp_bf16* dP,
                 cudaStream_t st) {
    const long long count = 1LL * T * h;
    if (count == 0) return TPMLP_OK;
    cudaError_t e = launch_dependent(
        dropout_grad_kernel, dim3(static_cast<unsigned>(cdiv(count, 8LL * kDropThreads * kDropVec))),
        dim3(kDropThreads), 0, st, cb(dY), count, dr, reinterpret_cast<__nv_bfloat16*>(dP));
    if (e != cudaSuccess) return fail_cuda(e);
    ++t_last_launches;
    return TPMLP_OK;
}

// Dropout parameters from the caller's rate p in [0, 1): keep iff the
// element's Philox word >= floor(p * 2^32), survivors scaled by 1 / (1 - p).
// The element counters advance four to a Philox block, so `offset` must be a
// multiple of 4.
int make_dropout(double p, uint64_t seed, uint64_t offset, Dropout& dr) {
    if (!(p >= 0.0 && p < 1.0) || offset % 4 != 0) return TPMLP_ERR_SHAPE;
    dr.threshold = static_cast<uint32_t>(p * 4294967296.0);
    dr.scale = static_cast<float>(1.0 / (1.0 - p));
    dr.seed = seed;
    dr.offset = offset;
    return TPMLP_OK;
}

int dgelu_gemm(const tpmlp_bf16* dY, const tpmlp_bf16* B, const tpmlp_bf16* Z, int T, int h,
               int F, int t, tpmlp_bf16* dZ, float* colsum, cudaStream_t st, const DeviceInfo& d) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{T, f, h, t, SHARD_N, 1LL * T * h, 1LL * F * h};
    g.a_on = ON_NONE;
    g.b_on = ON_ROWS;
    g.aux = cb(Z);
    g.ld_aux = F;
    g.colsum = colsum;
    g.ld_colsum = F;
    Operand a{dY, T, h, ON_NONE, false};
    Operand b{B, F, h, ON_ROWS, false};
    Output o{dZ, nullptr, T, F};
    return run_gemm(launch_dgelu, a, b, o, g, sh, st, d);
}

int dx_gemm(const tpmlp_bf16* dZ, const tpmlp_bf16* A, int T, int h, int F, int t,
            tpmlp_bf16* dX, void* ws, size_t ws_bytes, cudaStream_t st, const DeviceInfo& d) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{T, h, f, t, SHARD_K, 1LL * T * F, 1LL * h * F};
    g.a_on = ON_CONTIG;
    g.b_on = ON_CONTIG;
    Operand a{dZ, T, F, ON_CONTIG, false};
    Operand b{A, h, F, ON_CONTIG, false};
    const int sp = ws ? row_splits(T, h, F, t, ws_bytes, d) : 1;
    if (sp == 1) {
        Output o{dX, nullptr, T, h, 1};
        const TailSpec ts{launch_dx_partial, ws, ws_bytes, nullptr, nullptr, Dropout{}};
        return run_gemm(launch_dx, a, b, o, g, sh, st, d, &ts);
    }
    Output o{ws, nullptr, T, h, sp};
    if (int rc = run_gemm(launch_dx_partial, a, b, o, g, sh, st, d)) return rc;
    return launch_split_reduce(static_cast<const float*>(ws), sp, T, h, nullptr, nullptr, Dropout{}, dX, st);
}

// A weight gradient whole, or -- one shard (t = 1) and a workspace given --
// as k-range splits of fp32 partial outputs (weight_splits) added in split
// order by split_reduce_kernel.
int weight_grad(const Operand& a, const Operand& b, long long M, long long N, int T,
                GemmArgs& g, const GemmShape& sh, tpmlp_bf16* out, void* ws, size_t ws_bytes,
                cudaStream_t st, const DeviceInfo& d) {
    const int sp = (ws != nullptr && sh.t == 1) ? weight_splits(T, M, N, ws_bytes, d) : 1;
    if (sp == 1) {
        Output o{out, nullptr, M, N, 1};
        return run_gemm(launch_weight_grad, a, b, o, g, sh, st, d);
    }
    Output o{ws, nullptr, M, N, sp};
    if (int rc = run_gemm(launch_weight_grad_partial, a, b, o, g, sh, st, d)) return rc;
    return launch_split_reduce(static_cast<const float*>(ws), sp, static_cast<int>(M),
                               static_cast<int>(N), nullptr, nullptr, Dropout{}, out, st);
}

int dA_gemm(const tpmlp_bf16* X, const tpmlp_bf16* dZ, int T, int h, int F, int t,
            tpmlp_bf16* dA, cudaStream_t st, const DeviceInfo& d, void* ws = nullptr,
            size_t ws_bytes = 0) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{h, f, T, t, SHARD_N, 1LL * T * h, 1LL * T * F};
    g.a_on = ON_NONE;
    g.b_on = ON_CONTIG;
    Operand a{X, T, h, ON_NONE, true};
    Operand b{dZ, T, F, ON_CONTIG, true};
    return weight_grad(a, b, h, F, T, g, sh, dA, ws, ws_bytes, st, d);
}

int dB_gemm(const tpmlp_bf16* H, const tpmlp_bf16* dY, int T, int h, int F, int t,
            tpmlp_bf16* dB, cudaStream_t st, const DeviceInfo& d, void* ws = nullptr,
            size_t ws_bytes = 0) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{f, h, T, t, SHARD_M, 1LL * T * F, 1LL * T * h};
    g.a_on = ON_CONTIG;
    g.b_on = ON_NONE;
    Operand a{H, T, F, ON_CONTIG, true};
    Operand b{dY, T, h, ON_NONE, true};
    return weight_grad(a, b, F, h, T, g, sh, dB, ws, ws_bytes, st, d);
}

// a8 and a9 from the transposed operands, both K-major: Xt = X^T [h, ldT],
// dZt = dZ^T [F, ldT] (shard i: rows i F/t ..), Ht = H^T [F, ldT], dYt =
// dY^T [h, ldT]; the maps stop at column T, so a row's tail is never read.
// The sums are the MN-major kernels' (same k blocks, same order).
int dA_kmajor_gemm(const tpmlp_bf16* Xt, const tpmlp_bf16* dZt, int T, int ldT, int h, int F,
                   int t, tpmlp_bf16* dA, cudaStream_t st, const DeviceInfo& d) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{h, f, T, t, SHARD_N, 1LL * T * h, 1LL * T * F};
    Operand a{Xt, h, T, ON_NONE, false, ldT};
    Operand b{dZt, F, T, ON_ROWS, false, ldT};
    Output o{dA, nullptr, h, F};
    return run_gemm(launch_dx, a, b, o, g, sh, st, d);
}

int dB_kmajor_gemm(const tpmlp_bf16* Ht, const tpmlp_bf16* dYt, int T, int ldT, int h, int F,
                   int t, tpmlp_bf16* dB, cudaStream_t st, const DeviceInfo& d) {
    const int f = F / t;
    GemmArgs g = blank_args();
    const GemmShape sh{f, h, T, t, SHARD_M, 1LL * T * F, 1LL * T * h};
    Operand a{Ht, F, T, ON_ROWS, false, ldT};
    Operand b{dYt, h, T, ON_NONE, false, ldT};
    Output o{dB, nullptr, F, h};
    return run_gemm(launch_dx, a, b, o, g, sh, st, d);
}

int transpose(const tpmlp_bf16* in, int rows, int cols, tpmlp_bf16* out, int ld_out,
              cudaStream_t st) {
    cudaError_t e = launch_transpose(cb(in), rows, cols, reinterpret_cast<__nv_bfloat16*>(out),
                                     ld_out, st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

// Row pitch of a transposed [., T] operand: T rounded up to 8 elements (16 B).
int pitch_of(int T) { return (T + 7) & ~7; }

// Whether an M x N weight gradient (reduction over the T tokens; N the
// extent of one shard) is computed from transposed, K-major operands.  With
// both extents multiples of 64 the MN-major GEMM reads each operand's part
// of a stage as one box (the 4-D view of make_map_mn4) and runs within 1.3 %
// of the K-major one, which is less than the two transposes cost (4 T (M +
// N) bytes of HBM traffic; MT-NLG dA: 3.62 ms MN-major against 3.57 + 0.15
// ms).  With a ragged extent the MN-major operand takes two boxes per stage
// and runs 8-20 % slower; there the transposes pay when the GEMM's work per
// transposed element, M N / (M + N), is large (measured with F = 4h: gained
// with h >= 8192, lost with h <= 4096, at every T from 1024 to 16384).
bool kmajor_weight_grad(long long M, long long N) {
    if (M % 64 == 0 && N % 64 == 0) return false;
    return M * N >= 6144LL * (M + N);
}

// -------------------------------------------------- column sums (bias grads)

int launch_rowsum(const float* P, int rows, int n, float* out, cudaStream_t st) {
    cudaError_t e = launch_rowsum_f32(P, rows, n, out, st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

int bias_grad(const tpmlp_bf16* G, int T, int n, float* db, float* partial, cudaStream_t st) {
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(db, 0, sizeof(float) * static_cast<size_t>(n), st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    cudaError_t e = launch_colsum(cb(G), T, n, db, partial, st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

// ------------------------------------------------------ bounded-wait check

__global__ void wait_selftest_kernel(int* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must give up by itself.
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&bar, 0)) {
            if (global_ns() - t0 > limit_ns) {
                atomicExch(status, kStatusTimeout);
                break;
            }
        }
    }
}

size_t dgelu_partial_floats(int T, int F) {
    return static_cast<size_t>(4 * cdiv(T, BM)) * static_cast<size_t>(F);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Backward workspace: dZ, the db1 and db2 partial sums, the transposed
// operands of the weight gradients when they take the K-major form (X^T,
// dY^T: [h, ldT]; dZ^T, H^T: [F, ldT]) and the split-reduction scratch of dX.
struct BackwardLayout {
    size_t dz, colsum, db2, xt, dyt, dzt, ht, split, total;
};

BackwardLayout backward_layout(int T, int h, int F, int t) {
    BackwardLayout L;
    L.dz = 0;
    L.colsum = align256(L.dz + sizeof(uint16_t) * static_cast<size_t>(T) * F);
    L.db2 = align256(L.colsum + sizeof(float) * dgelu_partial_floats(T, F));
    const size_t db2_floats = colsum_workspace_floats(T, h);
    // the transposes only where a8 and a9 take the K-major form
    const size_t ldT = kmajor_weight_grad(h, F / t) ? static_cast<size_t>(pitch_of(T)) : 0;
    L.xt = align256(L.db2 + sizeof(float) * db2_floats);
    L.dyt = align256(L.xt + sizeof(uint16_t) * ldT * h);
    L.dzt = align256(L.dyt + sizeof(uint16_t) * ldT * h);
    L.ht = align256(L.dzt + sizeof(uint16_t) * ldT * F);
    L.split = align256(L.ht + sizeof(uint16_t) * ldT * F);
    L.total = align256(L.split + sizeof(float) * split_partial_floats(T, h, F, t));
    return L;
}

}  // namespace
}  // namespace tpmlp

using namespace tpmlp;

// ======================================================================
//                                 C ABI
// ======================================================================

#define TPMLP_PROLOGUE(dims_check)                 \
    t_last_launches = 0;                           \
    {                                              \
        int rc_ = (dims_check);                    \
        if (rc_) return rc_;                       \
    }

static int enter(DeviceInfo& d) {
    if (!get_encoder()) return TPMLP_ERR_UNSUPPORTED;
    return device_info(d);
}

TPMLP_API int tp_mlp_column_gelu(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                                 int T, int h, int F, int t, tpmlp_bf16* Z, tpmlp_bf16* H,
                                 void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (T == 0) return TPMLP_OK;
    if (any_null(X, A, b1, H)) return TPMLP_ERR_NULL;  // Z NULL: H only
    if (!all_aligned(X, A, b1, Z, H)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return column_gelu(X, A, b1, T, h, F, t, Z, H, static_cast<cudaStream_t>(stream), d);
}

TPMLP_API int tp_mlp_row_sum(const tpmlp_bf16* H, const tpmlp_bf16* B, const tpmlp_bf16* b2,
                             const tpmlp_bf16* residual, int T, int h, int F, int t, tpmlp_bf16* Y,
                             void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (T == 0) return TPMLP_OK;
    if (any_null(H, B, b2, residual, Y)) return TPMLP_ERR_NULL;
    if (!all_aligned(H, B, b2, residual, Y, workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return row_sum(H, B, b2, residual, T, h, F, t, Y, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), d);
}

TPMLP_API int tp_mlp_forward(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                             const tpmlp_bf16* B, const tpmlp_bf16* b2,
                             const tpmlp_bf16* residual, int T, int h, int F, int t,
                             tpmlp_bf16* Y, tpmlp_bf16* Z, tpmlp_bf16* H, void* workspace,
                             size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (T == 0) return TPMLP_OK;
    if (any_null(X, A, b1, B, b2, residual, Y, Z, H)) return TPMLP_ERR_NULL;
    if (!all_aligned(X, A, b1, B, b2, residual, Y, Z, H)) return TPMLP_ERR_ALIGN;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (int rc = column_gelu(X, A, b1, T, h, F, t, Z, H, st, d)) return rc;
    return row_sum(H, B, b2, residual, T, h, F, t, Y, workspace, workspace_bytes, st, d);
}

TPMLP_API size_t tp_mlp_bias_grad_workspace_floats(int T, int n) {
    if (T < 0 || n < 1) return 0;
    return colsum_workspace_floats(T, n);
}

TPMLP_API int tp_mlp_bias_grad(const tpmlp_bf16* G, int T, int n, float* db, float* partial,
                               void* stream) {
    t_last_launches = 0;
    if (T < 0 || n < 8 || n % 8 != 0) return TPMLP_ERR_SHAPE;
    if (any_null(db) || (T > 0 && any_null(G, partial))) return TPMLP_ERR_NULL;
    if (!all_aligned(G, db, partial)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return bias_grad(G, T, n, db, partial, static_cast<cudaStream_t>(stream));
}

// ----------------------------------------------------------------------
// Column sums without any allocation.
//
// Some callers cannot allocate device memory at the point where they need
// the bias gradient: a host framework that hands this library only the
// tensors it already owns and keeps every other byte of device memory to
// itself, or a plug-in that is forbidden to call cudaMalloc (or any
// allocator) once its set-up is over.  For them the partial sums of
// tp_mlp_bias_grad live in this fixed array instead of a caller buffer.  It
// is part of the loaded module, so every GPU that loads the library holds
// its 256 KiB until the process exits.
constexpr int kNoAllocScratchFloats = 1 << 16;
static __device__ __align__(256) float g_noalloc_colsum_scratch[kNoAllocScratchFloats];

namespace {
float* g_noalloc_scratch_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mutex;

// Device address of the array on the current device.  In host code the
// array's name stands for a host-side shadow, not for device memory, so the
// address is looked up once per device (with that device current) and kept.
int noalloc_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TPMLP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_colsum_scratch);
        if (e != cudaSuccess) return fail_cuda(e);
        g_noalloc_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_scratch_ptr[dev];
    return TPMLP_OK;
}
}  // namespace

TPMLP_API size_t tp_mlp_bias_grad_noalloc_max_floats(void) {
    return static_cast<size_t>(kNoAllocScratchFloats);
}

TPMLP_API int tp_mlp_bias_grad_noalloc(const tpmlp_bf16* G, int T, int n, float* db,
                                       void* stream) {
    t_last_launches = 0;
    if (T < 0 || n < 8 || n % 8 != 0) return TPMLP_ERR_SHAPE;
    if (any_null(db) || (T > 0 && any_null(G))) return TPMLP_ERR_NULL;
    if (!all_aligned(G, db)) return TPMLP_ERR_ALIGN;
    // Same row chunks as tp_mlp_bias_grad; one chunk needs no partials.
    // Every partial row is written before it is read, so nothing carries
    // over from an earlier call.
    if (T > 0 && colsum_chunks(T, n) > 1 &&
        colsum_workspace_floats(T, n) > static_cast<size_t>(kNoAllocScratchFloats))
        return TPMLP_ERR_WORKSPACE;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    float* scratch = nullptr;
    if (int rc = noalloc_scratch(&scratch)) return rc;
    return bias_grad(G, T, n, db, scratch, static_cast<cudaStream_t>(stream));
}

TPMLP_API size_t tp_mlp_dgelu_partial_floats(int T, int F) {
    if (T < 0 || F < 1) return 0;
    return dgelu_partial_floats(T, F);
}

TPMLP_API int tp_mlp_dgelu(const tpmlp_bf16* dY, const tpmlp_bf16* B, const tpmlp_bf16* Z, int T,
                           int h, int F, int t, tpmlp_bf16* dZ, float* db1,
                           float* colsum_partial, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (any_null(db1) || (T > 0 && any_null(dY, B, Z, dZ, colsum_partial))) return TPMLP_ERR_NULL;
    if (!all_aligned(dY, B, Z, dZ, db1, colsum_partial)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(db1, 0, sizeof(float) * static_cast<size_t>(F), st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    if (int rc = dgelu_gemm(dY, B, Z, T, h, F, t, dZ, colsum_partial, st, d)) return rc;
    return launch_rowsum(colsum_partial, static_cast<int>(4 * cdiv(T, BM)), F, db1, st);
}

TPMLP_API int tp_mlp_dx(const tpmlp_bf16* dZ, const tpmlp_bf16* A, int T, int h, int F, int t,
                        tpmlp_bf16* dX, void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (T == 0) return TPMLP_OK;
    if (any_null(dZ, A, dX)) return TPMLP_ERR_NULL;
    if (!all_aligned(dZ, A, dX, workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return dx_gemm(dZ, A, T, h, F, t, dX, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), d);
}

TPMLP_API int tp_mlp_dA_ws(const tpmlp_bf16* X, const tpmlp_bf16* dZ, int T, int h, int F, int t,
                           tpmlp_bf16* dA, void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (any_null(dA) || (T > 0 && any_null(X, dZ))) return TPMLP_ERR_NULL;
    if (!all_aligned(X, dZ, dA) || !aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(uint16_t) * static_cast<size_t>(h) * F, st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    return dA_gemm(X, dZ, T, h, F, t, dA, st, d, workspace, workspace ? workspace_bytes : 0);
}

TPMLP_API int tp_mlp_dA(const tpmlp_bf16* X, const tpmlp_bf16* dZ, int T, int h, int F, int t,
                        tpmlp_bf16* dA, void* stream) {
    return tp_mlp_dA_ws(X, dZ, T, h, F, t, dA, nullptr, 0, stream);
}

TPMLP_API int tp_mlp_dB_ws(const tpmlp_bf16* H, const tpmlp_bf16* dY, int T, int h, int F, int t,
                           tpmlp_bf16* dB, void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (any_null(dB) || (T > 0 && any_null(H, dY))) return TPMLP_ERR_NULL;
    if (!all_aligned(H, dY, dB) || !aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dB, 0, sizeof(uint16_t) * static_cast<size_t>(F) * h, st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    return dB_gemm(H, dY, T, h, F, t, dB, st, d, workspace, workspace ? workspace_bytes : 0);
}

TPMLP_API int tp_mlp_dB(const tpmlp_bf16* H, const tpmlp_bf16* dY, int T, int h, int F, int t,
                        tpmlp_bf16* dB, void* stream) {
    return tp_mlp_dB_ws(H, dY, T, h, F, t, dB, nullptr, 0, stream);
}

TPMLP_API size_t tp_weight_grad_workspace_bytes(int T, int M, int N) {
    if (T <= 0 || M <= 0 || N <= 0) return 0;
    return sizeof(float) * weight_split_floats(T, M, N);
}

TPMLP_API int tp_weight_grad_kmajor(int M, int N) {
    return M > 0 && N > 0 && kmajor_weight_grad(M, N) ? 1 : 0;
}

TPMLP_API int tp_transpose(const tpmlp_bf16* in, int rows, int cols, tpmlp_bf16* out,
                           int ld_out, void* stream) {
    t_last_launches = 0;
    if (rows < 0 || rows > 0x7FFFFFF0 || cols < 0 || cols % 8 != 0 || ld_out % 8 != 0 ||
        ld_out < pitch_of(rows))
        return TPMLP_ERR_SHAPE;
    if (rows == 0 || cols == 0) return TPMLP_OK;
    if (any_null(in, out)) return TPMLP_ERR_NULL;
    if (!all_aligned(in, out)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return transpose(in, rows, cols, out, ld_out, static_cast<cudaStream_t>(stream));
}

// check_dims plus the row pitch of the transposed operands
static int check_dims_ldT(int T, int ldT, int h, int F, int t) {
    if (int rc = check_dims(T, h, F, t)) return rc;
    return T > 0x7FFFFFF0 || ldT % 8 != 0 || ldT < pitch_of(T) ? TPMLP_ERR_SHAPE : TPMLP_OK;
}

TPMLP_API int tp_mlp_dA_kmajor(const tpmlp_bf16* Xt, const tpmlp_bf16* dZt, int T, int ldT,
                               int h, int F, int t, tpmlp_bf16* dA, void* stream) {
    TPMLP_PROLOGUE(check_dims_ldT(T, ldT, h, F, t));
    if (any_null(dA) || (T > 0 && any_null(Xt, dZt))) return TPMLP_ERR_NULL;
    if (!all_aligned(Xt, dZt, dA)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dA, 0, sizeof(uint16_t) * static_cast<size_t>(h) * F, st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    return dA_kmajor_gemm(Xt, dZt, T, ldT, h, F, t, dA, st, d);
}

TPMLP_API int tp_mlp_dB_kmajor(const tpmlp_bf16* Ht, const tpmlp_bf16* dYt, int T, int ldT,
                               int h, int F, int t, tpmlp_bf16* dB, void* stream) {
    TPMLP_PROLOGUE(check_dims_ldT(T, ldT, h, F, t));
    if (any_null(dB) || (T > 0 && any_null(Ht, dYt))) return TPMLP_ERR_NULL;
    if (!all_aligned(Ht, dYt, dB)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dB, 0, sizeof(uint16_t) * static_cast<size_t>(F) * h, st);
        return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
    }
    return dB_kmajor_gemm(Ht, dYt, T, ldT, h, F, t, dB, st, d);
}

TPMLP_API size_t tp_mlp_split_workspace_bytes(int T, int h, int F, int t) {
    if (check_dims(T, h, F, t) || T == 0) return 0;
    return sizeof(float) * split_partial_floats(T, h, F, t);
}

TPMLP_API size_t tp_mlp_forward_workspace_bytes(int T, int h, int F, int t) {
    return tp_mlp_split_workspace_bytes(T, h, F, t);
}

TPMLP_API size_t tp_mlp_backward_workspace_bytes(int T, int h, int F, int t) {
    if (check_dims(T, h, F, t)) return 0;
    return backward_layout(T, h, F, t).total;
}

// Steps a4..a9 given the gradient dY at the MLP's output and a workspace laid
// out by backward_layout (arguments already checked).
static int backward_steps(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* A,
                          const tpmlp_bf16* B, const tpmlp_bf16* Z, const tpmlp_bf16* H, int T,
                          int h, int F, int t, tpmlp_bf16* dX, tpmlp_bf16* dA, tpmlp_bf16* dB,
                          float* db1, float* db2, uint8_t* ws, const BackwardLayout& L,
                          cudaStream_t st, const DeviceInfo& d) {
    tpmlp_bf16* dZ = reinterpret_cast<tpmlp_bf16*>(ws + L.dz);
    float* colsum = reinterpret_cast<float*>(ws + L.colsum);
    float* db2_part = reinterpret_cast<float*>(ws + L.db2);
    // a4: db2 = sum_rows dY (the g operator passes dY to every shard unchanged)
    if (int rc = bias_grad(dY, T, h, db2, db2_part, st)) return rc;
    if (T == 0) {
        cudaError_t e;
        if ((e = cudaMemsetAsync(db1, 0, sizeof(float) * static_cast<size_t>(F), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dA, 0, sizeof(uint16_t) * static_cast<size_t>(h) * F, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dB, 0, sizeof(uint16_t) * static_cast<size_t>(F) * h, st)) != cudaSuccess)
            return fail_cuda(e);
        return TPMLP_OK;
    }
    // a5 + a6: dZ = (dY B_i^T) * GeLU'(Z_i), db1 partials fused, then reduced
    if (int rc = dgelu_gemm(dY, B, Z, T, h, F, t, dZ, colsum, st, d)) return rc;
    if (int rc = launch_rowsum(colsum, static_cast<int>(4 * cdiv(T, BM)), F, db1, st)) return rc;
    // a7: dX = sum_i dZ_i A_i^T (the f-operator sum inside the accumulator)
    if (int rc = dx_gemm(dZ, A, T, h, F, t, dX, ws + L.split, L.total - L.split, st, d)) return rc;
    // a8, a9: weight gradients of every shard; on large blocks of ragged
    // shard width both operands K-major after transposing X, dZ, H and dY
    if (!kmajor_weight_grad(h, F / t)) {
        if (int rc = dA_gemm(X, dZ, T, h, F, t, dA, st, d)) return rc;
        return dB_gemm(H, dY, T, h, F, t, dB, st, d);
    }
    const int ldT = pitch_of(T);
    tpmlp_bf16* Xt = reinterpret_cast<tpmlp_bf16*>(ws + L.xt);
    tpmlp_bf16* dYt = reinterpret_cast<tpmlp_bf16*>(ws + L.dyt);
    tpmlp_bf16* dZt = reinterpret_cast<tpmlp_bf16*>(ws + L.dzt);
    tpmlp_bf16* Ht = reinterpret_cast<tpmlp_bf16*>(ws + L.ht);
    if (int rc = transpose(X, T, h, Xt, ldT, st)) return rc;
    if (int rc = transpose(dZ, T, F, dZt, ldT, st)) return rc;
    if (int rc = dA_kmajor_gemm(Xt, dZt, T, ldT, h, F, t, dA, st, d)) return rc;
    if (int rc = transpose(H, T, F, Ht, ldT, st)) return rc;
    if (int rc = transpose(dY, T, h, dYt, ldT, st)) return rc;
    return dB_kmajor_gemm(Ht, dYt, T, ldT, h, F, t, dB, st, d);
}

TPMLP_API int tp_mlp_backward(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* A,
                              const tpmlp_bf16* B, const tpmlp_bf16* Z, const tpmlp_bf16* H,
                              int T, int h, int F, int t, tpmlp_bf16* dX, tpmlp_bf16* dA,
                              tpmlp_bf16* dB, float* db1, float* db2, void* workspace,
                              size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (any_null(A, B, dA, dB, db1, db2) || (T > 0 && any_null(dY, X, Z, H, dX)))
        return TPMLP_ERR_NULL;
    if (!all_aligned(dY, X, A, B, Z, H, dX, dA, dB, db1, db2)) return TPMLP_ERR_ALIGN;
    const BackwardLayout L = backward_layout(T, h, F, t);
    if (T > 0 && (workspace == nullptr || workspace_bytes < L.total)) return TPMLP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return backward_steps(dY, X, A, B, Z, H, T, h, F, t, dX, dA, dB, db1, db2,
                          static_cast<uint8_t*>(workspace), L, static_cast<cudaStream_t>(stream), d);
}

// ------------------------------------------------ activation recompute

// Forward with recompute: H lives in the workspace only until a3 has read it;
// the split-reduction scratch follows it.
static size_t recompute_h_bytes(int T, int F) {
    return align256(sizeof(uint16_t) * static_cast<size_t>(T) * F);
}

TPMLP_API size_t tp_mlp_forward_recompute_workspace_bytes(int T, int h, int F, int t) {
    if (check_dims(T, h, F, t) || T == 0) return 0;
    return recompute_h_bytes(T, F) + sizeof(float) * split_partial_floats(T, h, F, t);
}

TPMLP_API int tp_mlp_forward_recompute(const tpmlp_bf16* X, const tpmlp_bf16* A,
                                       const tpmlp_bf16* b1, const tpmlp_bf16* B,
                                       const tpmlp_bf16* b2, const tpmlp_bf16* residual, int T,
                                       int h, int F, int t, tpmlp_bf16* Y, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (T == 0) return TPMLP_OK;
    if (any_null(X, A, b1, B, b2, residual, Y)) return TPMLP_ERR_NULL;
    if (!all_aligned(X, A, b1, B, b2, residual, Y)) return TPMLP_ERR_ALIGN;
    const size_t hb = recompute_h_bytes(T, F);
    if (workspace == nullptr || workspace_bytes < hb) return TPMLP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    tpmlp_bf16* H = reinterpret_cast<tpmlp_bf16*>(ws);
    if (int rc = column_gelu(X, A, b1, T, h, F, t, nullptr, H, st, d)) return rc;
    return row_sum(H, B, b2, residual, T, h, F, t, Y, ws + hb, workspace_bytes - hb, st, d);
}

// Backward with recompute: Z and H are rebuilt in the workspace, followed by
// the block's own backward workspace.
TPMLP_API size_t tp_mlp_backward_recompute_workspace_bytes(int T, int h, int F, int t) {
    if (check_dims(T, h, F, t)) return 0;
    return 2 * recompute_h_bytes(T, F) + backward_layout(T, h, F, t).total;
}

TPMLP_API int tp_mlp_backward_recompute(const tpmlp_bf16* dY, const tpmlp_bf16* X,
                                        const tpmlp_bf16* A, const tpmlp_bf16* b1,
                                        const tpmlp_bf16* B, int T, int h, int F, int t,
                                        tpmlp_bf16* dX, tpmlp_bf16* dA, tpmlp_bf16* dB,
                                        float* db1, float* db2, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    if (any_null(A, B, dA, dB, db1, db2) || (T > 0 && any_null(dY, X, b1, dX)))
        return TPMLP_ERR_NULL;
    if (!all_aligned(dY, X, A, b1, B, dX, dA, dB, db1, db2)) return TPMLP_ERR_ALIGN;
    const BackwardLayout L = backward_layout(T, h, F, t);
    if (T > 0 && (workspace == nullptr ||
                  workspace_bytes < tp_mlp_backward_recompute_workspace_bytes(T, h, F, t)))
        return TPMLP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t hb = recompute_h_bytes(T, F);
    tpmlp_bf16* Z = T > 0 ? reinterpret_cast<tpmlp_bf16*>(ws) : nullptr;
    tpmlp_bf16* H = T > 0 ? reinterpret_cast<tpmlp_bf16*>(ws + hb) : nullptr;
    // the recompute: a2 again, from the saved input X
    if (T > 0)
        if (int rc = column_gelu(X, A, b1, T, h, F, t, Z, H, st, d)) return rc;
    return backward_steps(dY, X, A, B, Z, H, T, h, F, t, dX, dA, dB, db1, db2,
                          ws == nullptr ? nullptr : ws + 2 * hb, L, st, d);
}

// ------------------------------------------------ dropout before the residual

TPMLP_API int tp_mlp_row_sum_dropout(const tpmlp_bf16* H, const tpmlp_bf16* B,
                                     const tpmlp_bf16* b2, const tpmlp_bf16* residual, int T,
                                     int h, int F, int t, double p, uint64_t seed, uint64_t offset,
                                     tpmlp_bf16* Y, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    Dropout dr;
    if (int rc = make_dropout(p, seed, offset, dr)) return rc;
    if (T == 0) return TPMLP_OK;
    if (any_null(H, B, b2, residual, Y)) return TPMLP_ERR_NULL;
    if (!all_aligned(H, B, b2, residual, Y, workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return row_sum(H, B, b2, residual, T, h, F, t, Y, workspace, workspace_bytes,
                   static_cast<cudaStream_t>(stream), d, dr);
}

TPMLP_API int tp_mlp_forward_dropout(const tpmlp_bf16* X, const tpmlp_bf16* A,
                                     const tpmlp_bf16* b1, const tpmlp_bf16* B,
                                     const tpmlp_bf16* b2, const tpmlp_bf16* residual, int T,
                                     int h, int F, int t, double p, uint64_t seed, uint64_t offset,
                                     tpmlp_bf16* Y, tpmlp_bf16* Z, tpmlp_bf16* H, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    Dropout dr;
    if (int rc = make_dropout(p, seed, offset, dr)) return rc;
    if (T == 0) return TPMLP_OK;
    if (any_null(X, A, b1, B, b2, residual, Y, Z, H)) return TPMLP_ERR_NULL;
    if (!all_aligned(X, A, b1, B, b2, residual, Y, Z, H)) return TPMLP_ERR_ALIGN;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (int rc = column_gelu(X, A, b1, T, h, F, t, Z, H, st, d)) return rc;
    return row_sum(H, B, b2, residual, T, h, F, t, Y, workspace, workspace_bytes, st, d, dr);
}

TPMLP_API int tp_mlp_dropout_grad(const tpmlp_bf16* dY, int T, int h, double p, uint64_t seed,
                                  uint64_t offset, tpmlp_bf16* dP, void* stream) {
    t_last_launches = 0;
    if (T < 0 || h < 8 || h % 8 != 0) return TPMLP_ERR_SHAPE;
    Dropout dr;
    if (int rc = make_dropout(p, seed, offset, dr)) return rc;
    if (T == 0) return TPMLP_OK;
    if (any_null(dY, dP)) return TPMLP_ERR_NULL;
    if (!all_aligned(dY, dP)) return TPMLP_ERR_ALIGN;
    return dropout_grad(dY, T, h, dr, dP, static_cast<cudaStream_t>(stream));
}

// The dropout backward keeps dP = keep * dY / (1 - p) after the block's own
// backward workspace.
static size_t dropout_dp_offset(const BackwardLayout& L) { return align256(L.total); }

TPMLP_API size_t tp_mlp_backward_dropout_workspace_bytes(int T, int h, int F, int t) {
    if (check_dims(T, h, F, t)) return 0;
    const BackwardLayout L = backward_layout(T, h, F, t);
    return align256(dropout_dp_offset(L) + sizeof(uint16_t) * static_cast<size_t>(T) * h);
}

TPMLP_API int tp_mlp_backward_dropout(const tpmlp_bf16* dY, const tpmlp_bf16* X,
                                      const tpmlp_bf16* A, const tpmlp_bf16* B,
                                      const tpmlp_bf16* Z, const tpmlp_bf16* H, int T, int h,
                                      int F, int t, double p, uint64_t seed, uint64_t offset,
                                      tpmlp_bf16* dX, tpmlp_bf16* dA, tpmlp_bf16* dB, float* db1,
                                      float* db2, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    TPMLP_PROLOGUE(check_dims(T, h, F, t));
    Dropout dr;
    if (int rc = make_dropout(p, seed, offset, dr)) return rc;
    if (any_null(A, B, dA, dB, db1, db2) || (T > 0 && any_null(dY, X, Z, H, dX)))
        return TPMLP_ERR_NULL;
    if (!all_aligned(dY, X, A, B, Z, H, dX, dA, dB, db1, db2)) return TPMLP_ERR_ALIGN;
    const BackwardLayout L = backward_layout(T, h, F, t);
    if (T > 0 && (workspace == nullptr ||
                  workspace_bytes < tp_mlp_backward_dropout_workspace_bytes(T, h, F, t)))
        return TPMLP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    tpmlp_bf16* dP = T > 0 ? reinterpret_cast<tpmlp_bf16*>(ws + dropout_dp_offset(L)) : nullptr;
    if (int rc = dropout_grad(dY, T, h, dr, dP, st)) return rc;
    return backward_steps(dP, X, A, B, Z, H, T, h, F, t, dX, dA, dB, db1, db2, ws, L, st, d);
}

// ----------------------------------------------- residual add + LayerNorm

// LayerNorm rows are staged in shared memory as fp32.
constexpr int kLnMaxHidden = 49152;

static int check_ln(int T, int h, float eps) {
    if (T < 0 || h < 8 || h % 8 != 0 || h > kLnMaxHidden || !(eps > 0.0f)) return TPMLP_ERR_SHAPE;
    return TPMLP_OK;
}

TPMLP_API int tp_ln_residual_forward(const tpmlp_bf16* a, const tpmlp_bf16* r,
                                     const tpmlp_bf16* gamma, const tpmlp_bf16* beta, int T, int h,
                                     float eps, tpmlp_bf16* X, tpmlp_bf16* s, float* mean,
                                     float* rstd, void* stream) {
    TPMLP_PROLOGUE(check_ln(T, h, eps));
    if (any_null(gamma, beta) || (T > 0 && any_null(a, r, X, mean, rstd))) return TPMLP_ERR_NULL;
    if (!all_aligned(a, r, gamma, beta, X, s)) return TPMLP_ERR_ALIGN;
    if (T == 0) return TPMLP_OK;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaError_t e = launch_ln_forward(cb(a), cb(r), cb(gamma), cb(beta), T, h, eps,
                                      reinterpret_cast<__nv_bfloat16*>(X),
                                      reinterpret_cast<__nv_bfloat16*>(s), mean, rstd,
                                      static_cast<cudaStream_t>(stream), &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

TPMLP_API size_t tp_ln_residual_backward_workspace_floats(int T, int h) {
    if (check_ln(T, h, 1.0f)) return 0;
    return 2 * static_cast<size_t>(ln_param_chunks(T, h)) * static_cast<size_t>(h);
}

TPMLP_API int tp_ln_residual_backward(const tpmlp_bf16* dX, const tpmlp_bf16* dres,
                                      const tpmlp_bf16* a, const tpmlp_bf16* r,
                                      const tpmlp_bf16* gamma, const float* mean, const float* rstd,
                                      int T, int h, tpmlp_bf16* ds, float* dgamma, float* dbeta,
                                      float* partial, void* stream) {
    TPMLP_PROLOGUE(check_ln(T, h, 1.0f));
    if (any_null(gamma, dgamma, dbeta) ||
        (T > 0 && any_null(dX, a, r, mean, rstd, ds, partial)))
        return TPMLP_ERR_NULL;
    if (!all_aligned(dX, dres, a, r, gamma, ds, dgamma, dbeta, partial)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e;
        if ((e = cudaMemsetAsync(dgamma, 0, sizeof(float) * static_cast<size_t>(h), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dbeta, 0, sizeof(float) * static_cast<size_t>(h), st)) != cudaSuccess)
            return fail_cuda(e);
        return TPMLP_OK;
    }
    cudaError_t e = launch_ln_backward(cb(dX), cb(dres), cb(a), cb(r), cb(gamma), mean, rstd, T, h,
                                       reinterpret_cast<__nv_bfloat16*>(ds), dgamma, dbeta, partial,
                                       st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

// ---------------------------------------------- head-parallel attention

namespace tpmlp {
namespace {

// Head dims with a compiled attention kernel.
bool attn_head_dim_ok(int d) { return d == 64 || d == 96 || d == 128 || d == 160; }

int check_attn(int nb, int s, int h, int nh, int t) {
    if (nb < 0 || s < 1 || h < 8 || h % 8 != 0 || nh < 1 || h % nh != 0 || t < 1 ||
        t > TPMLP_MAX_SHARDS || nh % t != 0)
        return TPMLP_ERR_SHAPE;
    if (!attn_head_dim_ok(h / nh)) return TPMLP_ERR_SHAPE;
    if (static_cast<long long>(nb) * s >= (1LL << 31) || 3LL * h >= (1LL << 31))
        return TPMLP_ERR_SHAPE;
    return TPMLP_OK;
}

// 3-D tensor map {cols, s, nb} over a row-major bf16 [nb * s, cols] matrix
// (token n * s + pos), boxes of 64 columns x box_rows positions, so that a
// tile never crosses into the next sequence and ragged tails read zeros.
int make_seq_map(CUtensorMap* m, const void* ptr, int nb, int s, long long cols, int box_rows) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(s),
                          static_cast<cuuint64_t>(nb)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                             static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(s)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1}, estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        t_last_cuda_error = static_cast<int>(r);
        return TPMLP_ERR_LAUNCH;
    }
    return TPMLP_OK;
}

// QKV = X Wqkv + bqkv over all 3h columns: the column-parallel projection.
// Shard i's columns are its heads' blocks of Q, K and V; with no reduction
// across columns the t shards are one GEMM on one GPU.
int qkv_gemm(const tpmlp_bf16* X, const tpmlp_bf16* W, const tpmlp_bf16* b, int T, int h,
             tpmlp_bf16* QKV, cudaStream_t st, const DeviceInfo& d) {
    GemmArgs g = blank_args();
    const GemmShape sh{T, 3 * h, h, 1, SHARD_N, 1LL * T * h, 3LL * h * h};
    g.a_on = ON_NONE;
    g.b_on = ON_CONTIG;
    g.bias = cb(b);
    Operand a{X, T, h, ON_NONE, false};
    Operand bb{W, h, 3LL * h, ON_CONTIG, true};
    Output o{QKV, nullptr, T, 3LL * h, 1};
    return run_gemm(launch_column_bias, a, bb, o, g, sh, st, d);
}

// Bytes of caller memory that hold the persistent attention kernels' item
// counters (cleared on the stream by each call, so calls share nothing).
constexpr size_t kAttnCoreWorkBytes = 256;

int attn_core_forward(const tpmlp_bf16* QKV, int nb, int s, int h, int nh, tpmlp_bf16* O,
                      float* lse, void* work, cudaStream_t st, const DeviceInfo& d) {
    CUtensorMap tm, tm64;
    if (int rc = make_seq_map(&tm, QKV, nb, s, 3LL * h, 128)) return rc;
    if (int rc = make_seq_map(&tm64, QKV, nb, s, 3LL * h, 64)) return rc;
    AttnParams p{};
    p.nb = nb; p.s = s; p.h = h; p.nh = nh;
    p.O = reinterpret_cast<__nv_bfloat16*>(O);
    p.lse = lse;
    p.work = static_cast<unsigned int*>(work);
    p.status = d.status;
    cudaError_t e = launch_attn_forward(tm, tm64, h / nh, p, st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

int attn_core_backward(const tpmlp_bf16* QKV, const tpmlp_bf16* O, const float* lse,
                       const tpmlp_bf16* dO, int nb, int s, int h, int nh, tpmlp_bf16* dQKV,
                       float* delta, void* work, cudaStream_t st, const DeviceInfo& d) {
    CUtensorMap q128, q64, do128, do64;
    if (int rc = make_seq_map(&q128, QKV, nb, s, 3LL * h, 128)) return rc;
    if (int rc = make_seq_map(&q64, QKV, nb, s, 3LL * h, 64)) return rc;
    if (int rc = make_seq_map(&do128, dO, nb, s, h, 128)) return rc;
    if (int rc = make_seq_map(&do64, dO, nb, s, h, 64)) return rc;
    AttnParams p{};
    p.nb = nb; p.s = s; p.h = h; p.nh = nh;
    p.O_in = cb(O);
    p.dO = cb(dO);
    p.lse_in = lse;
    p.delta_out = delta;
    p.dqkv = reinterpret_cast<__nv_bfloat16*>(dQKV);
    p.work = static_cast<unsigned int*>(work);
    p.status = d.status;
    cudaError_t e = launch_attn_backward(q128, q64, do128, do64, h / nh, p, st, &t_last_launches);
    return e == cudaSuccess ? TPMLP_OK : fail_cuda(e);
}

size_t attn_colsum_floats(int T, int h) {
    return std::max(colsum_workspace_floats(T, h), colsum_workspace_floats(T, 3 * h));
}

// Attention backward workspace: dO, delta, dQKV, the column-sum partials,
// the transposed operands of dWo (O^T, dY^T) and dWqkv (X^T, dQKV^T) where
// those take the K-major form, and the split-reduction scratch (the
// row-parallel GEMMs' and, where dWo or dWqkv is split, its partials).
struct AttnBackwardLayout {
    size_t work, dO, delta, dqkv, colsum, ot, dyt, xt, dqkvt, split, total;
};

AttnBackwardLayout attn_backward_layout(int nb, int s, int h, int nh) {
    const long long T = 1LL * nb * s;
    AttnBackwardLayout L;
    L.work = 0;
    L.dO = kAttnCoreWorkBytes;
    L.delta = align256(L.dO + sizeof(uint16_t) * static_cast<size_t>(T) * h);
    L.dqkv = align256(L.delta + sizeof(float) * static_cast<size_t>(T) * nh);
    L.colsum = align256(L.dqkv + sizeof(uint16_t) * static_cast<size_t>(T) * 3 * h);
    const size_t ldT = static_cast<size_t>(pitch_of(static_cast<int>(T)));
    const size_t lo = kmajor_weight_grad(h, h) ? ldT : 0;       // dWo
    const size_t lq = kmajor_weight_grad(h, 3LL * h) ? ldT : 0;  // dWqkv
    L.ot = align256(L.colsum + sizeof(float) * attn_colsum_floats(static_cast<int>(T), h));
    L.dyt = align256(L.ot + sizeof(uint16_t) * lo * h);
    L.xt = align256(L.dyt + sizeof(uint16_t) * lo * h);
    L.dqkvt = align256(L.xt + sizeof(uint16_t) * lq * h);
    L.split = align256(L.dqkvt + sizeof(uint16_t) * lq * 3 * h);
    size_t sp = std::max(split_partial_floats(static_cast<int>(T), h, h, 1),
                         split_partial_floats(static_cast<int>(T), h, 3 * h, 1));
    if (!lo) sp = std::max(sp, weight_split_floats(static_cast<int>(T), h, h));
    if (!lq) sp = std::max(sp, weight_split_floats(static_cast<int>(T), h, 3LL * h));
    L.total = align256(L.split + sizeof(float) * sp);
    return L;
}

}  // namespace
}  // namespace tpmlp

TPMLP_API int tp_attn_qkv(const tpmlp_bf16* X, const tpmlp_bf16* Wqkv, const tpmlp_bf16* bqkv,
                          int T, int h, tpmlp_bf16* QKV, void* stream) {
    TPMLP_PROLOGUE((T < 0 || h < 8 || h % 8 != 0) ? TPMLP_ERR_SHAPE : TPMLP_OK);
    if (T == 0) return TPMLP_OK;
    if (any_null(X, Wqkv, bqkv, QKV)) return TPMLP_ERR_NULL;
    if (!all_aligned(X, Wqkv, bqkv, QKV)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return qkv_gemm(X, Wqkv, bqkv, T, h, QKV, static_cast<cudaStream_t>(stream), d);
}

TPMLP_API size_t tp_attn_core_workspace_bytes(int nb, int s, int h, int nh) {
    if (check_attn(nb, s, h, nh, 1) || nb == 0) return 0;
    return kAttnCoreWorkBytes;
}

TPMLP_API int tp_attn_core_forward(const tpmlp_bf16* QKV, int nb, int s, int h, int nh,
                                   tpmlp_bf16* O, float* lse, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_attn(nb, s, h, nh, 1));
    if (nb == 0) return TPMLP_OK;
    if (any_null(QKV, O, lse)) return TPMLP_ERR_NULL;
    if (workspace == nullptr || workspace_bytes < kAttnCoreWorkBytes) return TPMLP_ERR_WORKSPACE;
    if (!all_aligned(QKV, O, lse, workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return attn_core_forward(QKV, nb, s, h, nh, O, lse, workspace,
                             static_cast<cudaStream_t>(stream), d);
}

TPMLP_API int tp_attn_core_backward(const tpmlp_bf16* QKV, const tpmlp_bf16* O, const float* lse,
                                    const tpmlp_bf16* dO, int nb, int s, int h, int nh,
                                    tpmlp_bf16* dQKV, float* delta, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_attn(nb, s, h, nh, 1));
    if (nb == 0) return TPMLP_OK;
    if (any_null(QKV, O, lse, dO, dQKV, delta)) return TPMLP_ERR_NULL;
    if (workspace == nullptr || workspace_bytes < kAttnCoreWorkBytes) return TPMLP_ERR_WORKSPACE;
    if (!all_aligned(QKV, O, lse, dO, dQKV, delta, workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    return attn_core_backward(QKV, O, lse, dO, nb, s, h, nh, dQKV, delta, workspace,
                              static_cast<cudaStream_t>(stream), d);
}

// tp_attn_forward's workspace: the core kernel's item counter, then the
// output projection's split-reduction scratch.
TPMLP_API size_t tp_attn_forward_workspace_bytes(int nb, int s, int h, int nh, int t) {
    if (check_attn(nb, s, h, nh, t) || nb == 0) return 0;
    return kAttnCoreWorkBytes + sizeof(float) * split_partial_floats(nb * s, h, h, t);
}

TPMLP_API int tp_attn_forward(const tpmlp_bf16* X, const tpmlp_bf16* Wqkv, const tpmlp_bf16* bqkv,
                              const tpmlp_bf16* Wo, const tpmlp_bf16* bo,
                              const tpmlp_bf16* residual, int nb, int s, int h, int nh, int t,
                              tpmlp_bf16* Y, tpmlp_bf16* QKV, tpmlp_bf16* O, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_attn(nb, s, h, nh, t));
    if (nb == 0) return TPMLP_OK;
    if (any_null(X, Wqkv, bqkv, Wo, bo, residual, Y, QKV, O, lse)) return TPMLP_ERR_NULL;
    if (workspace == nullptr || workspace_bytes < kAttnCoreWorkBytes) return TPMLP_ERR_WORKSPACE;
    if (!all_aligned(X, Wqkv, bqkv, Wo, bo, residual, Y, QKV, O, lse, workspace))
        return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int T = nb * s;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (int rc = qkv_gemm(X, Wqkv, bqkv, T, h, QKV, st, d)) return rc;
    if (int rc = attn_core_forward(QKV, nb, s, h, nh, O, lse, ws, st, d)) return rc;
    // row-parallel output projection: Y = sum_i O_i Wo_i + bo + residual, the
    // g-operator sum folded into one accumulator (the MLP's a3 GEMM with F = h)
    return row_sum(O, Wo, bo, residual, T, h, h, t, Y, ws + kAttnCoreWorkBytes,
                   workspace_bytes - kAttnCoreWorkBytes, st, d);
}

TPMLP_API size_t tp_attn_backward_workspace_bytes(int nb, int s, int h, int nh, int t) {
    if (check_attn(nb, s, h, nh, t)) return 0;
    return attn_backward_layout(nb, s, h, nh).total;
}

TPMLP_API int tp_attn_backward(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* Wqkv,
                               const tpmlp_bf16* Wo, const tpmlp_bf16* QKV, const tpmlp_bf16* O,
                               const float* lse, int nb, int s, int h, int nh, int t,
                               tpmlp_bf16* dX, tpmlp_bf16* dWqkv, float* dbqkv, tpmlp_bf16* dWo,
                               float* dbo, void* workspace, size_t workspace_bytes, void* stream) {
    TPMLP_PROLOGUE(check_attn(nb, s, h, nh, t));
    if (any_null(Wqkv, Wo, dWqkv, dbqkv, dWo, dbo) ||
        (nb > 0 && any_null(dY, X, QKV, O, lse, dX)))
        return TPMLP_ERR_NULL;
    if (!all_aligned(dY, X, Wqkv, Wo, QKV, O, lse, dX, dWqkv, dbqkv, dWo, dbo))
        return TPMLP_ERR_ALIGN;
    const AttnBackwardLayout L = attn_backward_layout(nb, s, h, nh);
    if (nb > 0 && (workspace == nullptr || workspace_bytes < L.total)) return TPMLP_ERR_WORKSPACE;
    if (!aligned16(workspace)) return TPMLP_ERR_ALIGN;
    DeviceInfo d;
    if (int rc = enter(d)) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int T = nb * s;
    if (T == 0) {
        cudaError_t e;
        if ((e = cudaMemsetAsync(dbo, 0, sizeof(float) * static_cast<size_t>(h), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dbqkv, 0, sizeof(float) * 3 * static_cast<size_t>(h), st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dWo, 0, sizeof(uint16_t) * static_cast<size_t>(h) * h, st)) != cudaSuccess ||
            (e = cudaMemsetAsync(dWqkv, 0, sizeof(uint16_t) * 3 * static_cast<size_t>(h) * h, st)) != cudaSuccess)
            return fail_cuda(e);
        return TPMLP_OK;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    tpmlp_bf16* dO = reinterpret_cast<tpmlp_bf16*>(ws + L.dO);
    float* delta = reinterpret_cast<float*>(ws + L.delta);
    tpmlp_bf16* dQKV = reinterpret_cast<tpmlp_bf16*>(ws + L.dqkv);
    float* colsum = reinterpret_cast<float*>(ws + L.colsum);
    // dbo = sum_rows dY (g backward: the identity on every shard)
    if (int rc = bias_grad(dY, T, h, dbo, colsum, st)) return rc;
    // dWo_i = O_i^T dY: shard i's rows of dWo.  No sum crosses the shards,
    // so all rows are one GEMM (t only labels them), free of the ragged
    // per-shard row tiles that h / t rows would leave
    const int ldT = pitch_of(T);
    if (kmajor_weight_grad(h, h)) {
        tpmlp_bf16* Ot = reinterpret_cast<tpmlp_bf16*>(ws + L.ot);
        tpmlp_bf16* dYt = reinterpret_cast<tpmlp_bf16*>(ws + L.dyt);
        if (int rc = transpose(O, T, h, Ot, ldT, st)) return rc;
        if (int rc = transpose(dY, T, h, dYt, ldT, st)) return rc;
        if (int rc = dB_kmajor_gemm(Ot, dYt, T, ldT, h, h, 1, dWo, st, d)) return rc;
    } else if (int rc = dB_gemm(O, dY, T, h, h, 1, dWo, st, d, ws + L.split,
                                L.total - L.split)) {
        return rc;
    }
    // dO = dY Wo^T: shard i's columns of dO from its rows of Wo, no sum
    if (int rc = dx_gemm(dY, Wo, T, h, h, 1, dO, ws + L.split, L.total - L.split, st, d)) return rc;
    // local attention backward of every head
    if (int rc = attn_core_backward(QKV, O, lse, dO, nb, s, h, nh, dQKV, delta, ws + L.work, st, d))
        return rc;
    // dbqkv = sum_rows dQKV ; dWqkv = X^T dQKV (column blocks per shard)
    if (int rc = bias_grad(dQKV, T, 3 * h, dbqkv, colsum, st)) return rc;
    if (kmajor_weight_grad(h, 3LL * h)) {
        tpmlp_bf16* Xt = reinterpret_cast<tpmlp_bf16*>(ws + L.xt);
        tpmlp_bf16* dQKVt = reinterpret_cast<tpmlp_bf16*>(ws + L.dqkvt);
        if (int rc = transpose(X, T, h, Xt, ldT, st)) return rc;
        if (int rc = transpose(dQKV, T, 3 * h, dQKVt, ldT, st)) return rc;
        if (int rc = dA_kmajor_gemm(Xt, dQKVt, T, ldT, h, 3 * h, 1, dWqkv, st, d)) return rc;
    } else if (int rc = dA_gemm(X, dQKV, T, h, 3 * h, 1, dWqkv, st, d, ws + L.split,
                                L.total - L.split)) {
        return rc;
    }
    // dX = sum_i dQKV_i Wqkv_i^T: the f-operator sum as one accumulation over
    // all 3h columns
    return dx_gemm(dQKV, Wqkv, T, h, 3 * h, 1, dX, ws + L.split, L.total - L.split, st, d);
}

TPMLP_API const char* tp_mlp_status_string(int status) {
    switch (status) {
        case TPMLP_OK: return "ok";
        case TPMLP_ERR_NULL: return "a required pointer is NULL";
        case TPMLP_ERR_SHAPE: return "invalid shape (need h%8==0, (F/t)%8==0, F%t==0, h,F>=8, T>=0)";
        case TPMLP_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case TPMLP_ERR_WORKSPACE: return "workspace missing or too small";
        case TPMLP_ERR_LAUNCH: return "a CUDA call failed (see tpmlp_last_cuda_error)";
        case TPMLP_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
        case TPMLP_ERR_UNSUPPORTED: return "the current device is not sm_103 or the driver lacks TMA";
        default: return "unknown status";
    }
}

TPMLP_API const char* tpmlp_status_string(int status) { return tp_mlp_status_string(status); }

TPMLP_API int tpmlp_set_cta_pair_mode(int mode) {
    if (mode < 0 || mode > 2) return -1;
    return g_pair_mode.exchange(mode);
}

TPMLP_API int tpmlp_set_dependent_launch(int mode) {
    if (mode < 0 || mode > 3) return -1;
    return g_dependent_launch.exchange(mode);
}

TPMLP_API int tpmlp_set_tile_scheduler(int mode) {
    if (mode < 0 || mode > 2) return -1;
    return g_tile_scheduler.exchange(mode);
}

TPMLP_API int tpmlp_set_wide_tiles(int mode) {
    if (mode < 0 || mode > 1) return -1;
    return g_wide_tiles.exchange(mode);
}

TPMLP_API int tpmlp_set_epilogue_warps(int mode) {
    if (mode != 0 && mode != 4 && mode != 8) return -1;
    return g_epi_mode.exchange(mode);
}

TPMLP_API int tpmlp_last_cuda_error(void) { return t_last_cuda_error; }

TPMLP_API int tpmlp_last_launch_count(void) { return t_last_launches; }

static int read_clear_status(int index, int* out) {
    DeviceInfo d;
    if (int rc = device_info(d)) return rc;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e);
    int v = 0;
    if ((e = cudaMemcpy(&v, d.status + index, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda(e);
    const int zero = 0;
    if ((e = cudaMemcpy(d.status + index, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
        return fail_cuda(e);
    *out = v;
    return TPMLP_OK;
}

TPMLP_API int tpmlp_device_status(void) {
    int v = 0;
    if (int rc = read_clear_status(0, &v)) return rc;
    return v;
}

TPMLP_API int tpmlp_device_wait_site(void) {
    int v = 0;
    if (int rc = read_clear_status(1, &v)) return -rc;
    return v;
}

TPMLP_API int tpmlp_selftest_bounded_wait(int timeout_us, void* stream) {
    t_last_launches = 0;
    if (timeout_us < 1 || timeout_us > 1000000) return TPMLP_ERR_SHAPE;
    DeviceInfo d;
    if (int rc = device_info(d)) return rc;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d.status, 1000ull * static_cast<unsigned long long>(timeout_us));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e);
    t_last_launches = 1;
    return TPMLP_OK;
}
