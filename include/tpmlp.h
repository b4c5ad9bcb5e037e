/*
 * tpmlp.h -- C ABI of the GB300 (sm_103a) tensor-parallel Transformer MLP block.
 *
 * The block is the Megatron-LM MLP with the column-then-row split:
 *
 *     Y = GeLU(X A + b1) B + b2 + residual
 *
 * A [h, F] is split by columns into A_1..A_t, B [F, h] by rows into
 * B_1..B_t, b1 [F] with A's columns ("Megatron-LM: Tensor Model Parallel",
 * charles2530.github.io, section "MLP: Column Parallel first, then Row
 * Parallel", Figure 3a).  Shard i computes GeLU(X A_i + b1_i) locally and
 * contributes the partial product H_i B_i to the g-operator sum; the backward
 * pass gathers dX through the f-operator sum (same page, section "f / g
 * Operators", Figure 4).  All t shards run on the calling GPU: the g and f
 * sums are fp32 accumulations inside the row-parallel GEMMs, not collectives.
 * GeLU is the tanh approximation 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))
 * (the pages name GeLU without defining it).
 *
 * Conventions shared by every entry point:
 *  - T tokens, hidden size h, FFN width F, shard count t, shard width
 *    f = F / t.  Matrices are dense row-major with no padding.
 *  - Tensors are bfloat16 (raw 16-bit patterns, type tpmlp_bf16) except the
 *    bias gradients db1/db2 and the workspace, which are float32.
 *    Products accumulate in float32; bf16 outputs are rounded to nearest even.
 *  - Every pointer is a DEVICE pointer into memory the caller allocated and
 *    owns, aligned to 16 bytes.  The library allocates nothing and keeps no
 *    reference to any buffer after the call returns.  A pointer to an array
 *    with no elements (every [T, .] array when T == 0) may be NULL.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Outputs must not alias inputs.
 *  - Shape rules: T >= 0, h >= 8, F >= 8, 1 <= t <= TPMLP_MAX_SHARDS,
 *    F % t == 0, h % 8 == 0 and f % 8 == 0 (16-byte row strides, the tensor
 *    memory accelerator's rule), T, h, F < 2^31.  T == 0 is a valid empty
 *    batch.
 *  - Return value: TPMLP_OK, or an error code below; arguments are checked
 *    before anything is launched, so a rejected call has no effect.  A launch
 *    failure returns TPMLP_ERR_LAUNCH and tpmlp_last_cuda_error() holds the
 *    CUDA error.  Device-side waits are bounded: a kernel whose wait gives up
 *    records TPMLP_ERR_DEVICE_TIMEOUT in a device status word, which
 *    tpmlp_device_status() reads (synchronously) and clears.
 *  - Thread safety and shared state.  Every scratch word a kernel counts
 *    or accumulates in is caller memory passed with the call (a workspace,
 *    cleared on the stream where it must start at zero), so calls on
 *    different streams or threads, and calls captured into CUDA graphs and
 *    replayed beside eager calls, share no device state -- except the
 *    array of tp_mlp_bias_grad_noalloc, which its calls share (see there).
 *    Process-wide host state: the GEMM launch modes of
 *    tpmlp_set_cta_pair_mode, tpmlp_set_epilogue_warps, tpmlp_set_wide_tiles,
 *    tpmlp_set_dependent_launch and tpmlp_set_tile_scheduler (atomics, read at
 *    each launch: change them only
 *    while no other thread launches, or results stay equal but the launch
 *    shape may differ between two calls), a once-per-process lookup of the
 *    driver's tensor-map encoder, once-per-device kernel attributes and
 *    device addresses (the status word, the no-allocation array), all
 *    guarded.  The device status word is per device: a timeout recorded by
 *    one call is read by whichever thread calls tpmlp_device_status next.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t tpmlp_bf16; /* raw bfloat16 bits */

#define TPMLP_MAX_SHARDS 64

enum tpmlp_status {
    TPMLP_OK = 0,
    TPMLP_ERR_NULL = 1,           /* a required pointer is NULL */
    TPMLP_ERR_SHAPE = 2,          /* a shape rule above is violated */
    TPMLP_ERR_ALIGN = 3,          /* a pointer is not 16-byte aligned */
    TPMLP_ERR_WORKSPACE = 4,      /* workspace missing or too small */
    TPMLP_ERR_LAUNCH = 5,         /* a CUDA call failed; see tpmlp_last_cuda_error */
    TPMLP_ERR_DEVICE_TIMEOUT = 6, /* a bounded device wait gave up */
    TPMLP_ERR_UNSUPPORTED = 7     /* the current device is not sm_103 */
};

/* ---------------------------------------------------------------------- */
/* Whole block                                                             */
/* ---------------------------------------------------------------------- */

/* Bytes of optional float32 scratch that lets the row-parallel GEMMs (a3,
 * a7) split their reduction when their ceil(T/256) x ceil(h/256) output tiles
 * cannot occupy the GPU (small T).  0 when these sizes never split. */
size_t tp_mlp_split_workspace_bytes(int T, int h, int F, int t);

/* Same value, named for tp_mlp_forward's `workspace`. */
size_t tp_mlp_forward_workspace_bytes(int T, int h, int F, int t);

/* Forward pass (steps a2 + a3 below):
 *   Z = X A + b1, H = GeLU(Z)         (all t column shards)
 *   Y = sum_i H_i B_i + b2 + residual (g-operator sum of the row shards)
 * In:  X [T,h], A [h,F], b1 [F], B [F,h], b2 [h], residual [T,h].
 * Out: Y [T,h]; Z, H [T,F] are saved for the backward pass.
 * `workspace` (16-byte aligned, may be NULL) of tp_mlp_forward_workspace_bytes
 * bytes lets a3 split its reduction (see tp_mlp_row_sum); with NULL or fewer
 * bytes it splits less or not at all -- the result is the same sum up to
 * float32 rounding order. */
int tp_mlp_forward(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                   const tpmlp_bf16* B, const tpmlp_bf16* b2, const tpmlp_bf16* residual,
                   int T, int h, int F, int t, tpmlp_bf16* Y, tpmlp_bf16* Z, tpmlp_bf16* H,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of float32/bf16 scratch tp_mlp_backward needs for these sizes. */
size_t tp_mlp_backward_workspace_bytes(int T, int h, int F, int t);

/* Backward pass given dY = dL/dY (steps a4..a9 below):
 *   db2 = sum_rows dY                      (g backward is the identity)
 *   dZ_i = (dY B_i^T) * GeLU'(Z_i)         db1_i = sum_rows dZ_i
 *   dX = sum_i dZ_i A_i^T                  (f-operator sum)
 *   dA_i = X^T dZ_i ; dB_i = H_i^T dY
 * In:  dY, X [T,h]; A [h,F]; B [F,h]; Z, H [T,F] from tp_mlp_forward.
 * Out: dX [T,h], dA [h,F], dB [F,h] (bf16); db1 [F], db2 [h] (float32).
 * d(residual) equals dY and is not written.  `workspace` must hold
 * tp_mlp_backward_workspace_bytes(T,h,F,t) bytes (16-byte aligned); its
 * contents on entry do not matter and on return are unspecified. */
int tp_mlp_backward(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* A,
                    const tpmlp_bf16* B, const tpmlp_bf16* Z, const tpmlp_bf16* H,
                    int T, int h, int F, int t, tpmlp_bf16* dX, tpmlp_bf16* dA,
                    tpmlp_bf16* dB, float* db1, float* db2, void* workspace,
                    size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- */
/* The steps of the hot path, one call each.  tp_mlp_forward and          */
/* tp_mlp_backward are exactly these calls in this order (the backward     */
/* takes a8 and a9 in their transposed-operand form, below tp_mlp_dB,      */
/* where tp_weight_grad_kmajor says so).                                   */
/* ---------------------------------------------------------------------- */

/* a2: column-parallel GEMM with fused bias and GeLU, all t shards in one
 * launch: Z[:, i f:(i+1) f] = X A_i + b1_i, H = GeLU(Z).
 * (Figure 3a of the page above: each shard applies GeLU to its own columns
 * with no synchronisation before the nonlinearity.)  Z may be NULL: only H
 * is written (the forward pass of activation recompute, which rebuilds Z in
 * the backward pass). */
int tp_mlp_column_gelu(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                       int T, int h, int F, int t, tpmlp_bf16* Z, tpmlp_bf16* H, void* stream);

/* a3: row-parallel GEMM whose fp32 accumulator walks the shards in order,
 * so the partials H_i B_i meet in the accumulator (the g-operator sum),
 * with b2 and the residual fused into the epilogue:
 * Y = sum_i H_i B_i + b2 + residual.  H [T,F], B [F,h] -> Y [T,h].
 * When the output tiles are too few for the GPU and `workspace` (16-byte
 * aligned, tp_mlp_split_workspace_bytes bytes; may be NULL) allows, each
 * tile's k range -- the shards in order -- is cut into contiguous runs whose
 * fp32 partial sums go to the workspace, and a second kernel adds them in
 * run order with b2 and the residual (two launches instead of one).  When
 * the tiles fill more than one round of the CTA pairs but the last round
 * only partly (CTA pairs only; the tail split), the whole rounds run as
 * usual and only the last round's tiles are cut that way (three launches). */
int tp_mlp_row_sum(const tpmlp_bf16* H, const tpmlp_bf16* B, const tpmlp_bf16* b2,
                   const tpmlp_bf16* residual, int T, int h, int F, int t, tpmlp_bf16* Y,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Float32 elements of scratch tp_mlp_bias_grad needs: the row chunks'
 * partial sums. */
size_t tp_mlp_bias_grad_workspace_floats(int T, int n);

/* a4 (and the reduction of a6): column sums of a [T, n] bf16 matrix,
 * db[j] = sum_r G[r, j], in float32, deterministic.  Used for db2 = sum_rows
 * dY (the g operator is the identity backward, so dY reaches b2 whole).
 * `partial` must hold tp_mlp_bias_grad_workspace_floats(T, n) floats, any
 * contents.  One kernel writes the row chunks' partial sums, a second adds
 * them in chunk order (one kernel when T is small enough for one chunk). */
int tp_mlp_bias_grad(const tpmlp_bf16* G, int T, int n, float* db, float* partial,
                     void* stream);

/* Column sums like tp_mlp_bias_grad, for callers that cannot allocate
 * device memory (a framework that passes only the tensors it owns and
 * reserves all other memory, or code that may not call an allocator after
 * its set-up).  The source pages have no counterpart: this is a service of
 * the library.  The partial sums go to a fixed 256 KiB array inside the
 * library (tp_mlp_bias_grad_noalloc_max_floats() floats), so this call
 * allocates nothing; every GPU that loads the library holds that array
 * until the process exits.  Arguments as tp_mlp_bias_grad minus `partial`.
 * Limit: what tp_mlp_bias_grad_workspace_floats(T, n) asks for must fit
 * the array; every n <= 24576 fits at any T, larger shapes may return
 * TPMLP_ERR_WORKSPACE (nothing launched).  The first call on each device
 * looks up the array's device address: make it before any stream capture.
 * All calls on a device share the array, which keeps what the last call
 * left there: each call overwrites the partial rows it uses before reading
 * them, so no result depends on an earlier call and nothing needs clearing;
 * calls whose kernels overlap on the GPU (different streams, no ordering)
 * race on it. */
int tp_mlp_bias_grad_noalloc(const tpmlp_bf16* G, int T, int n, float* db, void* stream);

/* Capacity, in floats, of the array tp_mlp_bias_grad_noalloc uses. */
size_t tp_mlp_bias_grad_noalloc_max_floats(void);

/* Float32 elements of the per-tile column partials tp_mlp_dgelu writes. */
size_t tp_mlp_dgelu_partial_floats(int T, int F);

/* a5 + a6: dZ_i = (dY B_i^T) * GeLU'(Z_i) for all shards in one launch, with
 * the db1 column partial sums of each 128-row tile fused into the epilogue
 * (written to `colsum_partial`, tp_mlp_dgelu_partial_floats(T,F) floats),
 * then reduced into db1 [F] (float32).
 * dY [T,h], B [F,h], Z [T,F] -> dZ [T,F] (bf16), db1 [F]. */
int tp_mlp_dgelu(const tpmlp_bf16* dY, const tpmlp_bf16* B, const tpmlp_bf16* Z, int T, int h,
                 int F, int t, tpmlp_bf16* dZ, float* db1, float* colsum_partial,
                 void* stream);

/* a7: dX = sum_i dZ_i A_i^T; the accumulator walks the shards in order, so
 * the f-operator sum happens in fp32 inside the GEMM.
 * dZ [T,F], A [h,F] -> dX [T,h].  `workspace` as for tp_mlp_row_sum. */
int tp_mlp_dx(const tpmlp_bf16* dZ, const tpmlp_bf16* A, int T, int h, int F, int t,
              tpmlp_bf16* dX, void* workspace, size_t workspace_bytes, void* stream);

/* a8: dA_i = X^T dZ_i for every shard.  X [T,h], dZ [T,F] -> dA [h,F]. */
int tp_mlp_dA(const tpmlp_bf16* X, const tpmlp_bf16* dZ, int T, int h, int F, int t,
              tpmlp_bf16* dA, void* stream);

/* a9: dB_i = H_i^T dY for every shard.  H [T,F], dY [T,h] -> dB [F,h]. */
int tp_mlp_dB(const tpmlp_bf16* H, const tpmlp_bf16* dY, int T, int h, int F, int t,
              tpmlp_bf16* dB, void* stream);

/* a8 and a9 as above, with a caller workspace (device memory, 16-byte
 * aligned, owned by the caller, not read before it is written).  With t == 1
 * and an output of few 256 x 256 tiles -- the attention block's dWo (h x h)
 * and dWqkv (h x 3h) at small h -- the token reduction is cut into k ranges
 * that run on otherwise idle SM pairs as fp32 partial outputs in the
 * workspace, added in range order by a second kernel (deterministic; the
 * sum order differs from tp_mlp_dA / tp_mlp_dB by that split).  Otherwise,
 * or with a NULL or smaller workspace (fewer ranges), the result is that of
 * tp_mlp_dA / tp_mlp_dB.  tp_weight_grad_workspace_bytes(T, M, N) is the
 * workspace that allows every split for an M x N gradient (0: none is
 * taken).  Errors: those of tp_mlp_dA / tp_mlp_dB, ERR_ALIGN for a
 * misaligned workspace.  tp_attn_backward computes dWo and dWqkv this way. */
size_t tp_weight_grad_workspace_bytes(int T, int M, int N);
int tp_mlp_dA_ws(const tpmlp_bf16* X, const tpmlp_bf16* dZ, int T, int h, int F, int t,
                 tpmlp_bf16* dA, void* workspace, size_t workspace_bytes, void* stream);
int tp_mlp_dB_ws(const tpmlp_bf16* H, const tpmlp_bf16* dY, int T, int h, int F, int t,
                 tpmlp_bf16* dB, void* workspace, size_t workspace_bytes, void* stream);

/* Transpose of a bf16 matrix, the layout the two calls below read:
 * out[c * ld_out + r] = in[r * cols + c] for r < rows, c < cols, and
 * out[c * ld_out + r] = 0 for rows <= r < (rows rounded up to 8); the rest of
 * each output row is not touched.  in [rows, cols] row-major, out [cols,
 * ld_out], both device memory, 16-byte aligned, not overlapping.
 * Rules: rows >= 0, cols >= 0, cols % 8 == 0, ld_out % 8 == 0, ld_out >=
 * rows rounded up to 8.  rows or cols 0: nothing is launched. */
int tp_transpose(const tpmlp_bf16* in, int rows, int cols, tpmlp_bf16* out, int ld_out,
                 void* stream);

/* 1 when the composite calls (tp_mlp_backward and its variants,
 * tp_attn_backward) compute an M x N weight gradient (per shard: dA_i,
 * dB_i: h x F/t or F/t x h; dWqkv: h x 3h; dWo: h x h) from transposed
 * operands with tp_transpose and the two calls below, else 0 (they call
 * tp_mlp_dA / tp_mlp_dB).  The rule: 0 when M and N are both multiples of
 * 64 (the row-major operands are then read in one box per stage, as fast
 * as the transposed ones); otherwise 1 when M N / (M + N) >= 6144, where
 * the K-major GEMM repays the two transposes.  No device work. */
int tp_weight_grad_kmajor(int M, int N);

/* a8 and a9 from transposed operands, so that both GEMM operands are read
 * along their contiguous dimension (K-major).  Faster than the row-major X,
 * dZ, H, dY of tp_mlp_dA / tp_mlp_dB where a shard's width is not a
 * multiple of 64 (those operands then take two boxes a pipeline stage);
 * level with them otherwise.  Same sums, same outputs:
 *   dA_i = X^T dZ_i   from Xt = X^T [h, ldT] and dZt = dZ^T [F, ldT]
 *   dB_i = H_i^T dY   from Ht = H^T [F, ldT] and dYt = dY^T [h, ldT]
 * (shard i of dZt / Ht is rows i F/t .. (i+1) F/t - 1), as tp_transpose
 * writes them with ld_out = ldT.  Only the first T entries of each row are
 * read.  Rules: those of tp_mlp_dA plus ldT % 8 == 0, ldT >= T rounded up
 * to 8.  T == 0: the output is zeroed. */
int tp_mlp_dA_kmajor(const tpmlp_bf16* Xt, const tpmlp_bf16* dZt, int T, int ldT, int h, int F,
                     int t, tpmlp_bf16* dA, void* stream);
int tp_mlp_dB_kmajor(const tpmlp_bf16* Ht, const tpmlp_bf16* dYt, int T, int ldT, int h, int F,
                     int t, tpmlp_bf16* dB, void* stream);

/* ---------------------------------------------------------------------- */
/* Residual add + LayerNorm feeding the block's input X                    */
/* ---------------------------------------------------------------------- */

/* The step in front of the MLP: "Megatron-DeepSpeed to ZeRO-3"
 * (seekfood.cn), section 4.3, names a fused LayerNorm + residual kernel
 * (output, input, residual, gamma, beta, n); "Megatron-LM: Tensor Model
 * Parallel", Figure 2, places layer normalization and the residual
 * connection around the MLP.  Per row of h values:
 *   s = a + r ; mu = mean(s) ; var = mean((s - mu)^2) (biased)
 *   X = (s - mu) / sqrt(var + eps) * gamma + beta
 * X feeds tp_mlp_forward and s is its `residual`.
 * In:  a, r [T,h] (sublayer output and incoming residual stream), gamma,
 *      beta [h] (bf16), eps > 0.
 * Out: X [T,h]; s [T,h] (may be NULL: not written); mean, rstd [T] float32
 *      (rstd = 1/sqrt(var+eps)), saved for the backward pass.
 * Rules: T >= 0, h % 8 == 0, 8 <= h <= 49152 (a row is staged in shared
 * memory). */
int tp_ln_residual_forward(const tpmlp_bf16* a, const tpmlp_bf16* r, const tpmlp_bf16* gamma,
                           const tpmlp_bf16* beta, int T, int h, float eps, tpmlp_bf16* X,
                           tpmlp_bf16* s, float* mean, float* rstd, void* stream);

/* Float32 elements of partial-sum scratch tp_ln_residual_backward needs. */
size_t tp_ln_residual_backward_workspace_floats(int T, int h);

/* Backward pass of tp_ln_residual_forward.  dres (may be NULL) is the
 * gradient reaching s directly -- for the MLP block, its dY:
 *   xhat = (s - mu) rstd ; g = dX * gamma
 *   ds = rstd (g - mean(g) - xhat mean(g xhat)) + dres    (= da = dr)
 *   dgamma = sum_rows dX xhat ; dbeta = sum_rows dX      (float32, deterministic)
 * In:  dX, dres, a, r [T,h]; gamma [h]; mean, rstd [T] from the forward pass.
 * Out: ds [T,h] (bf16), dgamma, dbeta [h] (float32).  `partial` holds
 * tp_ln_residual_backward_workspace_floats(T,h) floats. */
int tp_ln_residual_backward(const tpmlp_bf16* dX, const tpmlp_bf16* dres, const tpmlp_bf16* a,
                            const tpmlp_bf16* r, const tpmlp_bf16* gamma, const float* mean,
                            const float* rstd, int T, int h, tpmlp_bf16* ds, float* dgamma,
                            float* dbeta, float* partial, void* stream);

/* ---------------------------------------------------------------------- */
/* Activation recompute                                                    */
/* ---------------------------------------------------------------------- */

/* "MT-NLG 530B deep dive" (zzszmyf.github.io), section 2.2 (activation
 * checkpointing): keep only each layer's input, and rerun the layer's
 * forward computation when the backward pass needs its intermediate
 * activations -- about a third more compute for much less activation
 * memory; "Megatron-LM: Tensor Model Parallel", training-recipe table (row
 * "Memory"), checkpoints after every Transformer layer.  For this block the
 * saved activations shrink from Z and H (2 T F values) to X (T h, which the
 * caller holds anyway); Z and H are rebuilt by a2 at the start of the
 * backward pass. */

/* Bytes of scratch tp_mlp_forward_recompute needs: H [T,F] bf16, live only
 * during the call, plus a3's split-reduction scratch. */
size_t tp_mlp_forward_recompute_workspace_bytes(int T, int h, int F, int t);

/* Forward pass that saves nothing for the backward pass: a2 writes only H,
 * into the workspace, and a3 reads it; Y as tp_mlp_forward.  The workspace
 * (16-byte aligned, at least the H part; the split part is optional as for
 * tp_mlp_forward) may be reused by other calls once this one completes. */
int tp_mlp_forward_recompute(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                             const tpmlp_bf16* B, const tpmlp_bf16* b2,
                             const tpmlp_bf16* residual, int T, int h, int F, int t,
                             tpmlp_bf16* Y, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Bytes of scratch tp_mlp_backward_recompute needs: the recomputed Z and H
 * ([T,F] bf16 each) plus tp_mlp_backward's workspace. */
size_t tp_mlp_backward_recompute_workspace_bytes(int T, int h, int F, int t);

/* Backward pass from the layer input alone: a2 recomputes Z = X A + b1 and
 * H = GeLU(Z) into the workspace (bitwise the values tp_mlp_forward saves),
 * then steps a4..a9 run as in tp_mlp_backward.  In: dY, X [T,h]; A [h,F];
 * b1 [F]; B [F,h].  Out as tp_mlp_backward. */
int tp_mlp_backward_recompute(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* A,
                              const tpmlp_bf16* b1, const tpmlp_bf16* B, int T, int h, int F,
                              int t, tpmlp_bf16* dX, tpmlp_bf16* dA, tpmlp_bf16* dB, float* db1,
                              float* db2, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- */
/* Dropout before the residual add                                         */
/* ---------------------------------------------------------------------- */

/* "Megatron-LM: Tensor Model Parallel", Figure 2 places dropout between the
 * MLP's output and the residual add, and its training-recipe table (row
 * "Stabilization") gives the rate 0.1.  The same page (section "Hybrid
 * MP + DP", the paragraph on random numbers) puts this dropout outside the
 * model-parallel region: every shard of a model instance must draw the same
 * pattern.  Here the pattern is a pure function of (seed, element), so it
 * cannot depend on the shard count or the GPU's schedule:
 *   g    = offset + row * h + col            (element counter)
 *   w    = Philox4x32-10(counter = (g/4 mod 2^32, g/4 >> 32, 0, 0),
 *                        key = (seed mod 2^32, seed >> 32))[g mod 4]
 *   keep = w >= floor(p * 2^32)              (exact integer comparison)
 *   Y    = residual + keep * (sum_i H_i B_i + b2) / (1 - p)
 * (Philox4x32 with 10 rounds: Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11.)  Rules beyond the block's: p is a
 * double in [0, 1) -- p = 0 gives tp_mlp_forward's result exactly -- and
 * offset is a multiple of 4 (a Philox block holds four element counters);
 * otherwise TPMLP_ERR_SHAPE.  A caller advances offset by T*h (rounded up to
 * a multiple of 4) per call to draw a fresh pattern with the same seed. */

/* a3 with bias-dropout-add in its epilogue (and in the split reduction when
 * the GEMM splits).  Arguments as tp_mlp_row_sum plus p, seed, offset. */
int tp_mlp_row_sum_dropout(const tpmlp_bf16* H, const tpmlp_bf16* B, const tpmlp_bf16* b2,
                           const tpmlp_bf16* residual, int T, int h, int F, int t, double p,
                           uint64_t seed, uint64_t offset, tpmlp_bf16* Y, void* workspace,
                           size_t workspace_bytes, void* stream);

/* tp_mlp_forward with the dropout above: a2, then tp_mlp_row_sum_dropout.
 * Workspace as tp_mlp_forward's. */
int tp_mlp_forward_dropout(const tpmlp_bf16* X, const tpmlp_bf16* A, const tpmlp_bf16* b1,
                           const tpmlp_bf16* B, const tpmlp_bf16* b2, const tpmlp_bf16* residual,
                           int T, int h, int F, int t, double p, uint64_t seed, uint64_t offset,
                           tpmlp_bf16* Y, tpmlp_bf16* Z, tpmlp_bf16* H, void* workspace,
                           size_t workspace_bytes, void* stream);

/* The gradient the dropout passes to the MLP's output:
 * dP = keep * dY / (1 - p), bf16, keep drawn as above from (seed, offset).
 * dY, dP [T,h]; rules T >= 0, h % 8 == 0, h >= 8. */
int tp_mlp_dropout_grad(const tpmlp_bf16* dY, int T, int h, double p, uint64_t seed,
                        uint64_t offset, tpmlp_bf16* dP, void* stream);

/* Bytes of scratch tp_mlp_backward_dropout needs: tp_mlp_backward's plus
 * the bf16 dP [T,h]. */
size_t tp_mlp_backward_dropout_workspace_bytes(int T, int h, int F, int t);

/* Backward pass of tp_mlp_forward_dropout: tp_mlp_dropout_grad into the
 * workspace, then tp_mlp_backward's steps a4..a9 on dP (so db2 = sum_rows dP
 * and dB_i = H_i^T dP).  The residual's gradient is dY itself, not written.
 * Arguments as tp_mlp_backward plus p, seed, offset (the forward pass's). */
int tp_mlp_backward_dropout(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* A,
                            const tpmlp_bf16* B, const tpmlp_bf16* Z, const tpmlp_bf16* H, int T,
                            int h, int F, int t, double p, uint64_t seed, uint64_t offset,
                            tpmlp_bf16* dX, tpmlp_bf16* dA, tpmlp_bf16* dB, float* db1,
                            float* db2, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- */
/* Head-parallel self-attention block                                      */
/* ---------------------------------------------------------------------- */

/* "Megatron-LM: Tensor Model Parallel" (charles2530.github.io), section
 * "Attention: split Q/K/V by head" (Figure 3b): the Q, K and V projections
 * are split by columns so that each rank owns nh / t of the nh heads; each
 * head's scores, softmax and value sum are local; the output projection is
 * split by rows, and its per-rank partials meet in the g-operator sum before
 * the residual add:
 *
 *   QKV = X Wqkv + bqkv                            (column-parallel)
 *   per sequence and head j:  S = Q_j K_j^T / sqrt(d), causal mask,
 *                             P = softmax over each row, O_j = P V_j
 *   Y   = sum_i O_i Wo_i + bo + residual           (row-parallel, g sum)
 *
 * Layout: nb sequences of s tokens, T = nb * s, token n * s + pos;
 * X, residual, Y, O [T, h]; QKV [T, 3h] with columns [Q | K | V] and head j
 * at columns j*d .. j*d + d - 1 of each part (d = h / nh); Wqkv [h, 3h],
 * bqkv [3h], Wo [h, h] (head j's rows at j*d), bo [h]; lse float32 [nh, T].
 * Shard i owns heads i*nh/t .. (i+1)*nh/t - 1: their Wqkv columns, bqkv
 * entries and Wo rows.  The mask is causal within a sequence (a token sees
 * itself and the earlier tokens of its sequence), as in the pages' GPT
 * models; the page fixes only the split, the rest is the plain reading.
 *
 * Rules (else TPMLP_ERR_SHAPE): nb >= 0, s >= 1, h % 8 == 0, nh >= 1,
 * h % nh == 0, d = h / nh in {64, 96, 128, 160} (the head dims with a
 * compiled kernel: GPT-2 355M, 2.5B and 8.3B of the Megatron-LM page's
 * Table 2, and MT-NLG 530B's 20480 / 128), 1 <= t <= 64,
 * nh % t == 0, T < 2^31.  nb == 0 is an empty batch.  Pointers, ownership,
 * streams and status codes as for the MLP block above. */

/* QKV = X Wqkv + bqkv (bf16 out, fp32 accumulation): the column-parallel
 * projection of every shard as one GEMM (no sum crosses its columns).
 * Rules T >= 0, h % 8 == 0, h >= 8. */
int tp_attn_qkv(const tpmlp_bf16* X, const tpmlp_bf16* Wqkv, const tpmlp_bf16* bqkv, int T, int h,
                tpmlp_bf16* QKV, void* stream);

/* Bytes of scratch the two core calls below need (0 when nb == 0): the
 * item counters of their persistent kernels, which each call clears on its
 * stream before its kernels run (contents on entry do not matter). */
size_t tp_attn_core_workspace_bytes(int nb, int s, int h, int nh);

/* Causal attention of every (sequence, head) from QKV: O [T, h] (bf16) and
 * lse [nh, T] (float32), lse = log2 sum_k 2^(c q.k) over the visible keys
 * with c = log2(e) / sqrt(d), saved for the backward pass.  `workspace`:
 * device memory of tp_attn_core_workspace_bytes bytes, 16-byte aligned
 * (TPMLP_ERR_WORKSPACE if NULL or smaller when nb > 0). */
int tp_attn_core_forward(const tpmlp_bf16* QKV, int nb, int s, int h, int nh, tpmlp_bf16* O,
                         float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* Backward of tp_attn_core_forward given dO [T, h]: dQKV [T, 3h] (bf16;
 * dQ, dK, dV in the layout of QKV).  delta [nh, T] float32 is scratch
 * (rowsum(dO * O) per head); `workspace` as for tp_attn_core_forward.  Every
 * gradient is written once, in a fixed summation order, with no atomics, so
 * results are reproducible. */
int tp_attn_core_backward(const tpmlp_bf16* QKV, const tpmlp_bf16* O, const float* lse,
                          const tpmlp_bf16* dO, int nb, int s, int h, int nh, tpmlp_bf16* dQKV,
                          float* delta, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch of tp_attn_forward: the core call's counters (required), then
 * room that lets the output projection split its reduction when its output
 * tiles cannot occupy the GPU (optional: with fewer bytes it splits less or
 * not at all).  0 when nb == 0. */
size_t tp_attn_forward_workspace_bytes(int nb, int s, int h, int nh, int t);

/* The block's forward pass: tp_attn_qkv, tp_attn_core_forward, then the
 * row-parallel output projection (tp_mlp_row_sum with F = h: Y = sum_i O_i
 * Wo_i + bo + residual, the g sum folded into one fp32 accumulator).  QKV, O
 * and lse are outputs saved for the backward pass.  workspace: at least
 * tp_attn_core_workspace_bytes bytes when nb > 0 (16-byte aligned), up to
 * tp_attn_forward_workspace_bytes. */
int tp_attn_forward(const tpmlp_bf16* X, const tpmlp_bf16* Wqkv, const tpmlp_bf16* bqkv,
                    const tpmlp_bf16* Wo, const tpmlp_bf16* bo, const tpmlp_bf16* residual,
                    int nb, int s, int h, int nh, int t, tpmlp_bf16* Y, tpmlp_bf16* QKV,
                    tpmlp_bf16* O, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream);

/* Bytes of scratch tp_attn_backward needs: dO [T,h] bf16, delta [nh,T] f32,
 * dQKV [T,3h] bf16, column-sum partials, split-reduction partials. */
size_t tp_attn_backward_workspace_bytes(int nb, int s, int h, int nh, int t);

/* The block's backward pass (chain rule of the forward formula):
 *   dbo = sum_rows dY ; dWo_i = O_i^T dY ; dO_i = dY Wo_i^T ;
 *   attention backward -> dQKV ; dbqkv = sum_rows dQKV ;
 *   dWqkv = X^T dQKV ; dX = sum_i dQKV_i Wqkv_i^T (the f-operator sum, one
 *   fp32 accumulation over all 3h columns).
 * dX is the gradient through the block; the residual's gradient is dY
 * itself and is not written.  dX, dWqkv, dWo bf16; dbqkv, dbo float32.
 * workspace must hold tp_attn_backward_workspace_bytes (it may be NULL when
 * nb == 0, in which case the parameter gradients are zeroed). */
int tp_attn_backward(const tpmlp_bf16* dY, const tpmlp_bf16* X, const tpmlp_bf16* Wqkv,
                     const tpmlp_bf16* Wo, const tpmlp_bf16* QKV, const tpmlp_bf16* O,
                     const float* lse, int nb, int s, int h, int nh, int t, tpmlp_bf16* dX,
                     tpmlp_bf16* dWqkv, float* dbqkv, tpmlp_bf16* dWo, float* dbo,
                     void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------- */
/* Status                                                                  */
/* ---------------------------------------------------------------------- */

/* Which GEMM kernel the library launches (process-wide; returns the
 * previous mode, or -1 for an invalid mode):
 *   0  single-CTA kernel (128 x 256 output tiles, one SM each);
 *   1  default: CTA pairs (cluster of 2, 256 x 256 tiles shared by two SMs
 *      through tcgen05 cta_group::2) when the problem has at least 32
 *      256 x 256 tiles, else single CTAs;
 *   2  CTA pairs always.
 * Both kernels compute the same sums in the same order (the split of a
 * reduction does not depend on the mode), so results are bitwise identical
 * across modes -- except where a row-parallel GEMM takes the tail split,
 * which only CTA pairs do: the tiles of its last partly full round are
 * summed in k ranges (see tp_mlp_row_sum). */
int tpmlp_set_cta_pair_mode(int mode);

/* How many epilogue warps the dZ GEMM (step a5, the one GEMM kernel with
 * both forms) launches with (process-wide; returns the previous mode, or -1
 * for an invalid mode):
 *   0  default: eight for reductions of at most 16 k-blocks of 64 (K <=
 *      1024), where a tile's mainloop is too short to hide four warps'
 *      epilogue, else four;
 *   4  four warps always;  8  eight warps always.
 * Each output element gets the same arithmetic in either form, so results
 * are bitwise identical across modes. */
int tpmlp_set_epilogue_warps(int mode);

/* Which of the library's kernels are launched as programmatic dependents of
 * the kernel before them on the stream (process-wide; returns the previous
 * mode, or -1 for a mode outside 0..3): bit 0 the GEMMs, bit 1 the
 * column-sum, reduction, transpose and dropout kernels.  A dependent's CTAs
 * may start, and set up their barriers and tensor memory, while the kernel
 * before it finishes; they read and write global memory only after it has
 * completed, so results are identical in every mode.  0: plain stream
 * order; 3 (both) is the default. */
int tpmlp_set_dependent_launch(int mode);

/* How the GEMM kernels assign output tiles (work units) to CTA pairs
 * (process-wide; returns the previous mode, or -1 for a mode outside 0..2):
 *   0  a persistent grid of as many pairs as fit, pair u taking units u,
 *      u + pairs, ... in the tile raster order;
 *   1  one pair per unit in the grid; a running pair takes the next unit by
 *      cancelling the launch of a pair that has not started (cluster launch
 *      control), so the units in flight are always a contiguous run of the
 *      raster order however unevenly the pairs progress;
 *   2  default: 1 for GEMMs whose tiles reduce over 192 or more k-blocks
 *      of 64 (K >= 12288), where pairs sharing an operand panel otherwise
 *      drift apart, 0 for the rest, whose short tiles would wait on the next
 *      unit (MT-NLG 530B step 3.8 % faster than with 0).
 * Every mode computes every unit with the same sums: results are bitwise
 * identical across modes. */
int tpmlp_set_tile_scheduler(int mode);

/* Output tile of the GEMMs with K-major operands and a plain store (dX, and
 * the weight gradients from transposed operands), process-wide; returns the
 * previous mode, or -1 for a mode outside 0..1:
 *   0  default: 256 x 256 per CTA pair;
 *   1  256 x 512 per CTA pair where the reduction is not split: two N = 256
 *      MMAs share each A stage, a quarter fewer operand bytes from L2 per
 *      flop; TMEM holds one accumulator, so a tile's epilogue does not
 *      overlap the next tile's MMAs.
 * Each output element gets the same sums in the same order: results are
 * bitwise identical across modes. */
int tpmlp_set_wide_tiles(int mode);

/* Static text for a status code. */
const char* tp_mlp_status_string(int status);

/* The same function under its earlier name. */
const char* tpmlp_status_string(int status);

/* The CUDA error code (cudaError_t) behind the last TPMLP_ERR_LAUNCH on the
 * calling thread, 0 if none. */
int tpmlp_last_cuda_error(void);

/* Reads and clears the device status word of the current device: TPMLP_OK,
 * or TPMLP_ERR_DEVICE_TIMEOUT if a bounded wait in a kernel gave up since the
 * last read.  Synchronises the device. Returns TPMLP_ERR_LAUNCH if the read
 * itself fails. */
int tpmlp_device_status(void);

/* Reads and clears the site code of the first bounded wait that gave up on
 * the current device since the last read: 0 if none; otherwise a code that
 * names the kernel and the wait (0x1nn attention forward, 0x2nn attention dQ,
 * 0x3nn attention dK/dV; the GEMM kernels record none).  Synchronises the
 * device.  A failed read returns minus the status code. */
int tpmlp_device_wait_site(void);

/* Number of kernels the last successful call on the calling thread
 * launched (for launch accounting). */
int tpmlp_last_launch_count(void);

/* Self-test of the bounded device wait: launches one small kernel whose
 * thread waits on a barrier that nothing ever completes, with a limit of
 * `timeout_us` microseconds (1..1000000).  Returns TPMLP_OK after the launch;
 * tpmlp_device_status() then reports TPMLP_ERR_DEVICE_TIMEOUT. */
int tpmlp_selftest_bounded_wait(int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
