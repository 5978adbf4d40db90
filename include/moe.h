/*
 * moe.h -- C ABI of libmoe: the single-GPU forward pass of an expert-parallel
 * Mixture-of-Experts layer on GB300 (sm_103a).
 *
 * The problem statement follows "Kernel fusion for expert parallelism"
 * (brunomaga.github.io), section "Expert parallelism: dispatch and combine":
 * N tokens of width H, E experts of which every token selects its top k, and
 * W ranks holding E/W experts each.  Here the W ranks are partitions of one
 * GPU's memory: rank r owns the rows of the experts in placement slots
 * [r*E/W, (r+1)*E/W).  The placement permutation follows "Expert Coupling"
 * (arXiv 2610.09372), Sec. V-A: slot p holds global expert placement[p].
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates and frees nothing and keeps no global state besides cached
 *    device attributes.  bf16 tensors are passed as uint16_t (bit patterns).
 *    Every tensor is dense, row-major, and 16-byte aligned; a bf16 tensor (or
 *    the fp32 accumulator of moe_ffn_down_combine) whose base is not 16-byte
 *    aligned is refused with MOE_ERR_INVALID_ARG.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *    asynchronous on it, except moe_get_error.
 *  - Argument checks run on the host before any launch and return
 *    MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE with nothing
 *    launched.  A failed launch returns MOE_ERR_CUDA.  Problems that only the
 *    device can see (an expert id out of range, a placement that is not a
 *    permutation, a wait that ran out of time) write a status code into the
 *    workspace's error word; kernels then keep every access in bounds and never
 *    trap.  moe_get_error reads and clears that word.
 *  - Sizes: 1 <= k <= min(E, 32), 1 <= E <= 1024, 1 <= W, E % W == 0,
 *    H % 8 == 0, I % 8 == 0, N >= 0 and N * k < 2^31.  N == 0 is a no-op.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad pointer, size or shape (host), bad ids/placement (device) */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported limits listed above */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_bytes() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_TIMEOUT = 5,       /* a device-side wait gave up (the kernel returned early) */
    MOE_ERR_DEVICE_ASSERT = 6  /* a device-side consistency check failed */
} moe_status;

/* Which tensor-core kernel runs the grouped GEMMs (moe_shape.gemm).  All give
 * the same results to fp32 accumulation order; they differ in speed only.
 *  MOE_GEMM_AUTO        the CTA-pair kernel when the problem has at least 512
 *                       rows per expert on average (N*k >= 512*E), else the
 *                       single-CTA kernel; moe_layer_forward, when H <= 128
 *                       (H <= 256 without dedup) and N*k >= 4096 or
 *                       I <= 256, runs the expert FFN as the fused kernel
 *                       instead (as with MOE_GEMM_FUSED; moe_layer_fuses_ffn)
 *  MOE_GEMM_SINGLE_CTA  128-row tiles, one CTA each (cta_group::1); the only
 *                       kernel with a gather mode
 *  MOE_GEMM_CTA_PAIR    256-row tiles shared by a 2-CTA cluster (cta_group::2)
 *  MOE_GEMM_FUSED       moe_expert_ffn and moe_layer_forward run the expert FFN
 *                       as one kernel that keeps h on chip (moe_ffn_fused; h
 *                       is not written and may be NULL there); the other GEMM
 *                       calls run the single-CTA kernel.  Only for H <= 256:
 *                       a shape with a larger H and this value is refused
 *                       with MOE_ERR_UNSUPPORTED.
 * Calls that gather rows inside the GEMM (moe_ffn_gate_up_gather, the dedup
 * form of moe_expert_ffn) and moe_ffn_down_combine always run the single-CTA
 * kernel for their gathered / fused launch. */
typedef enum {
    MOE_GEMM_AUTO = 0,
    MOE_GEMM_SINGLE_CTA = 1,
    MOE_GEMM_CTA_PAIR = 2,
    MOE_GEMM_FUSED = 3
} moe_gemm_kernel;

/* Layout of the routed experts' weights in every call that takes them
 * (moe_shape.weights).
 *  MOE_WEIGHTS_ROW_MAJOR  nn.Linear layout: w_gate, w_up bf16 [E, I, H];
 *                         w_down bf16 [E, H, I].
 *  MOE_WEIGHTS_PACKED     the tile-contiguous copies that moe_pack_weights
 *                         writes: w_gate points to the packed gate/up weights
 *                         (both matrices), w_up is not read (may be NULL), and
 *                         w_down points to the packed down weights.  A GEMM
 *                         then reads each 64-deep slice of a 256-row weight
 *                         tile as one contiguous 32 KB block instead of 256
 *                         strided 128-byte pieces, which lets the weight
 *                         stream of an HBM-bound layer run closer to the DRAM's
 *                         sequential read rate.  Results are bit-identical to
 *                         the row-major form.
 * The shared expert's weights (moe_shared_expert_ffn) are always row-major. */
typedef enum {
    MOE_WEIGHTS_ROW_MAJOR = 0,
    MOE_WEIGHTS_PACKED = 1
} moe_weight_layout;

/* N tokens of width H; E experts, top-k; W ranks; SwiGLU intermediate width I;
 * dedup != 0 selects the deduplicating dispatcher ("Expert Coupling" Sec. V-A):
 * one row per distinct (token, rank) instead of one per (token, expert).
 * gemm: a moe_gemm_kernel value (0 = automatic choice); weights: a
 * moe_weight_layout value (0 = row-major); any other value of either is
 * refused with MOE_ERR_INVALID_ARG, and packed weights of more than 2^31 rows
 * of 64 bf16 (256 GB) with MOE_ERR_UNSUPPORTED.  Every behaviour of the
 * library is set by these fields and the call's arguments: nothing is read
 * from the environment. */
typedef struct {
    int32_t N, H, E, k, W, I;
    int32_t dedup;
    int32_t gemm;
    int32_t weights;
} moe_shape;

/* Dispatch layout: caller-owned device arrays of int32, written by
 * moe_dispatch_layout.  R = N*k plain rows; R_d dedup rows.
 *  expert_counts[E]       rows of expert e
 *  expert_offsets[E+1]    first row of expert e's segment; [E] = R.  Segments
 *                         are stored in placement-slot order.
 *  rank_offsets[W+1]      first plain row of rank r; [W] = R
 *  row_token[N*k]         token of every plain row (ascending inside a segment)
 *  pair_row[N*k]          plain row of pair (t, j), at t*k + j
 *  dedup_counts[W]        dedup rows received by rank r
 *  dedup_offsets[W+1]     first dedup row of rank r; [W] = R_d
 *  dedup_row_token[N*min(k,W)]  token of every dedup row (rank-major,
 *                         ascending tokens inside a rank)
 *  pair_dedup_row[N*k]    dedup row that carries pair (t, j)
 *  expand_src[N*k]        dedup row that plain row i is expanded from
 *  n_dedup_rows[1]        R_d
 * The dedup arrays are written only when shape->dedup != 0 and may then be
 * NULL otherwise. */
typedef struct {
    int32_t* expert_counts;
    int32_t* expert_offsets;
    int32_t* rank_offsets;
    int32_t* row_token;
    int32_t* pair_row;
    int32_t* dedup_counts;
    int32_t* dedup_offsets;
    int32_t* dedup_row_token;
    int32_t* pair_dedup_row;
    int32_t* expand_src;
    int32_t* n_dedup_rows;
} moe_layout;

/* Bytes of device workspace that the calls taking `ws` need for this shape
 * (error word, per-block counts, the CTA-pair GEMM's tile counters).  0 if the
 * shape is invalid.
 * The caller zero-fills the workspace once after allocating it (the first
 * int32 is the error word); the calls keep it valid afterwards.  One workspace
 * must not be shared by calls running concurrently. */
size_t moe_workspace_bytes(const moe_shape* shape);

/* Bytes of the packed gate/up weights and of the packed down weights that
 * moe_pack_weights writes for this shape (0 if the shape is invalid):
 *   gate/up  E * ceil(I/128) * ceil(H/64) blocks of 256 x 64 bf16 (32 KB)
 *   down     E * ceil(H/256) * ceil(I/64) blocks of 256 x 64 bf16 */
size_t moe_packed_gate_up_bytes(const moe_shape* shape);
size_t moe_packed_down_bytes(const moe_shape* shape);

/* Copies row-major expert weights (w_gate, w_up bf16 [E, I, H]; w_down bf16
 * [E, H, I]) into the layout of MOE_WEIGHTS_PACKED, on the device (a storage
 * layout of this library: the gated MLP of FarSkip-Collective Sec. 2.1 is the
 * same computation on either).  Block
 * (e, b, q) sits at block index (e * NB + b) * KB + q and holds 256 rows of
 * 64 bf16, row-major (128 bytes a row):
 *   gate/up (NB = ceil(I/128), KB = ceil(H/64)): row r < 128 is
 *     w_gate[e, 128b + r, 64q .. 64q + 63] and row 128 + r the same slice of
 *     w_up[e, 128b + r, :], so one block is the 256-column operand slice of a
 *     gate/up tile (128 gate and the matching 128 up columns);
 *   down (NB = ceil(H/256), KB = ceil(I/64)): row r is
 *     w_down[e, 256b + r, 64q .. 64q + 63];
 * entries past the matrix (rows >= I or H, columns >= H or I) are zero.
 * Pure copies, done once per set of weights (a reformat at load time, not a
 * per-step cost).  gate_up_packed (moe_packed_gate_up_bytes) and down_packed
 * (moe_packed_down_bytes) are device buffers that must not overlap the
 * inputs; either may be NULL, and its inputs are then not read.
 * shape->weights is not read.  Asynchronous on stream. */
moe_status moe_pack_weights(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                            const moe_shape* shape, uint16_t* gate_up_packed,
                            uint16_t* down_packed, void* stream);

/* Top-k routing ("Expert Coupling" Appendix A-A1, Table II: fp32 gate, top-k
 * of E; FarSkip-Collective Sec. 2.1: G is a sparse top-k selection).
 * logits   fp32 [N, E]
 * topk_ids int32 [N, k]: the k largest logits of token t, descending, ties to
 *          the lower expert index
 * topk_w   fp32 [N, k]: softmax over the k selected logits (sums to one).
 * Non-finite logits are outside the contract. */
moe_status moe_route(const float* logits, const moe_shape* shape, int32_t* topk_ids,
                     float* topk_w, void* stream);

/* Router variant with the literal reading of "Expert Coupling" Appendix A-A1,
 * Table II ("softmax over all E, then top-k; gate weights = selected softmax
 * probabilities"): the same topk_ids as moe_route, and
 * topk_w[t, j] = exp(L_j - L_max) / sum over all E of exp(L_e - L_max),
 * which do not sum to one. */
moe_status moe_route_full_softmax(const float* logits, const moe_shape* shape, int32_t* topk_ids,
                                  float* topk_w, void* stream);

/* Router variant: the auxiliary-loss-free sigmoid router with a per-expert
 * bias ("Expert Coupling" Appendix A-B, the DeepSeek-V3 router).  Scores
 * s_e = sigmoid(L_e) are evaluated in double and rounded once to fp32; the
 * k largest s_e + bias[e] (an fp32 add; descending, ties to the lower expert
 * index) are selected; topk_w[t, j] = s_j / sum of the selected s (the bias
 * steers the selection only).  bias: device fp32 [E]. */
moe_status moe_route_sigmoid_bias(const float* logits, const float* bias, const moe_shape* shape,
                                  int32_t* topk_ids, float* topk_w, void* stream);

/* Dispatch layout (kernel-fusion page, "Expert parallelism: dispatch and
 * combine" and "Fusing the layer into one kernel" stage 3 "group"; "Expert
 * Coupling" Sec. V-A and Appendix A-A2).  Stable counting sort of the (t, j)
 * pairs by placement slot of topk_ids[t, j]; with dedup, also the distinct
 * (token, rank) rows and the expansion map.  Bit-exact and deterministic.
 * placement int32 [E] or NULL (identity = contiguous placement). */
moe_status moe_dispatch_layout(const int32_t* topk_ids, const int32_t* placement,
                               const moe_shape* shape, const moe_layout* layout, void* ws,
                               size_t ws_bytes, void* stream);

/* Dispatch (the all-to-all of the pages, here a copy between HBM partitions).
 * Plain:  xd[i, :] = x[row_token[i], :], xd bf16 [N*k, H].
 * Dedup:  xd[d, :] = x[dedup_row_token[d], :], xd bf16 [N*min(k,W), H]; only
 *         the first R_d rows are written.
 * x bf16 [N, H].  Every row is a bit-exact copy. */
moe_status moe_dispatch(const uint16_t* x, const moe_layout* layout, const moe_shape* shape,
                        uint16_t* xd, void* stream);

/* Grouped SwiGLU expert FFN (FarSkip-Collective Sec. 2.1; kernel-fusion page
 * stages 4-6).  For every plain row i of expert e:
 *   h[i, :] = bf16( SiLU(x_i Wg[e]^T) * (x_i Wu[e]^T) )      bf16 [N*k, I]
 *   y[i, :] = bf16( h[i, :] Wd[e]^T )                          bf16 [N*k, H]
 * with fp32 accumulation on the tensor cores.  Weights in the layout that
 * shape->weights names (moe_weight_layout): nn.Linear layout w_gate, w_up
 * bf16 [E, I, H], w_down bf16 [E, H, I]; or packed, with w_up unused.  The
 * same holds for every call below that takes expert weights.
 * Plain: xd holds the expert-major rows [N*k, H].
 * Dedup: xd holds the dedup rows; the gate/up GEMM reads them in expert-major
 *        order through layout->expand_src (the receiver's "group" step, done
 *        by the GEMM's gather warps instead of a copy into xe).
 * xe is not used and may be NULL (kept so that callers of the materialised
 * form, moe_expand + moe_ffn_gate_up, can share one buffer set).
 * shape->gemm == MOE_GEMM_FUSED: one moe_ffn_fused call (xd, through
 * expand_src when dedup); h is not written and may be NULL.
 * ws: workspace of moe_workspace_bytes(shape) bytes. */
moe_status moe_expert_ffn(const uint16_t* xd, const moe_layout* layout, const moe_shape* shape,
                          const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          uint16_t* xe, uint16_t* h, uint16_t* y, void* ws, size_t ws_bytes,
                          void* stream);

/* The steps of moe_expert_ffn as separate calls (kernel-fusion page,
 * "Fusing the layer into one kernel": stage 3 "group", stages 4-5 "MatMul" +
 * "SwiGLU", stage 6 "MatMul").  moe_expert_ffn is exactly
 *   plain: moe_ffn_gate_up(xd -> h); moe_ffn_down(h -> y)
 *   dedup: moe_ffn_gate_up_gather(xd, expand_src -> h); moe_ffn_down(h -> y)
 * on one stream, and its h equals, bit for bit, that of the materialised form
 *   moe_expand(xd -> xe); moe_ffn_gate_up(xe -> h).
 * moe_expand:      xe[i, :] = xd[expand_src[i], :] for the N*k expert-major rows
 *                  (dedup only; bit-exact copies).  Returns MOE_ERR_INVALID_ARG
 *                  when shape->dedup == 0.
 * moe_ffn_gate_up: h = bf16(SiLU(rows Wg[e]^T) * (rows Wu[e]^T)) for the
 *                  expert-major rows [N*k, H] (xd when plain, xe when dedup).
 * moe_ffn_down:    y = bf16(h Wd[e]^T).
 * Both GEMM calls take the workspace (the CTA-pair kernel keeps its tile
 * counters there; they return to zero after every launch). */
moe_status moe_expand(const uint16_t* xd, const moe_layout* layout, const moe_shape* shape,
                      uint16_t* xe, void* stream);
moe_status moe_ffn_gate_up(const uint16_t* rows, const moe_layout* layout, const moe_shape* shape,
                           const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h, void* ws,
                           size_t ws_bytes, void* stream);
moe_status moe_ffn_down(const uint16_t* h, const moe_layout* layout, const moe_shape* shape,
                        const uint16_t* w_down, uint16_t* y, void* ws, size_t ws_bytes,
                        void* stream);

/* moe_ffn_gate_up with the rows gathered inside the GEMM (the kernel-fusion
 * page's MegaKernel idea of feeding the MatMul without a separate "group" or
 * "pack" copy): problem row i (expert-major, i < N*k) is row row_index[i] of
 * src bf16 [src_rows, H].  With src = the dedup rows and row_index =
 * layout->expand_src this is the dedup expansion; with src = x and row_index
 * = layout->row_token it is the plain dispatch.  Out-of-range indices read
 * row 0.  Results are bit-identical to materialising the rows first.  Four
 * extra warps of the (single-CTA) GEMM copy the rows' 128-byte k-blocks with
 * 16-byte cp.async into the swizzled operand tiles; src_rows < 2^31. */
moe_status moe_ffn_gate_up_gather(const uint16_t* src, const int32_t* row_index, int64_t src_rows,
                                  const moe_layout* layout, const moe_shape* shape,
                                  const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h,
                                  void* ws, size_t ws_bytes, void* stream);

/* moe_ffn_down followed by moe_combine, fused: the down GEMM's epilogue scales
 * each output row by its routing weight and adds it into an fp32 accumulator
 * instead of storing y (the kernel-fusion page's MegaKernel direction, with the
 * stage-7 "reduce" moved into the MatMul), then
 *   out[t, :] = bf16( residual[t, :] + acc[t, :] ),
 *   acc[t, :] = sum_j topk_w[t, j] * (h[pair_row[t, j], :] Wd[e_j]^T)    fp32
 * acc: caller-owned fp32 [N, H] scratch, zeroed by this call.  residual is
 * nullable; out may equal residual.  The k terms of a token are added by
 * fp32 atomics in whatever order the tiles finish, so the result equals
 * moe_ffn_down + moe_combine up to fp32 reassociation and y's bf16 rounding
 * (y is never rounded here) and is not bit-reproducible from run to run.
 * The dedup form gives the same sums (its two-level order is not kept).
 * Always runs the single-CTA GEMM. */
moe_status moe_ffn_down_combine(const uint16_t* h, const float* topk_w, const moe_layout* layout,
                                const moe_shape* shape, const uint16_t* w_down,
                                const uint16_t* residual, float* acc, uint16_t* out, void* ws,
                                size_t ws_bytes, void* stream);

/* The expert FFN with h kept on chip (kernel-fusion page, "Fusing the layer
 * into one kernel": the expert's intermediate activations stay in the SM's
 * local memory between the two MatMuls).  One kernel computes, for every
 * plain row i of expert e,
 *   y[i, :] = bf16( bf16(SiLU(x_i Wg[e]^T) * (x_i Wu[e]^T)) Wd[e]^T )   bf16 [N*k, H]
 * with x_i = src[row_index[i], :] (row_index NULL: src[i, :], i < N*k, and
 * then src_rows >= N*k), src bf16 [src_rows, H], 0 < src_rows < 2^31; indices
 * out of range read row 0.  h never leaves the SM: a 128-row tile's h is made
 * 64 columns at a time (128 from I = 1024 on) into shared memory and consumed
 * there by the down MMA, whose 128 x H fp32 accumulator stays in TMEM, which is
 * why H <= 256 is required (MOE_ERR_UNSUPPORTED otherwise); I is not limited.
 * Same roundings and fp32 accumulation orders as moe_ffn_gate_up +
 * moe_ffn_down: y is bit-identical to theirs.  With
 * src = x and row_index = layout->row_token it includes the plain dispatch;
 * with src = the dedup rows and row_index = layout->expand_src the dedup
 * expansion.  Weights as shape->weights says. */
moe_status moe_ffn_fused(const uint16_t* src, const int32_t* row_index, int64_t src_rows,
                         const moe_layout* layout, const moe_shape* shape, const uint16_t* w_gate,
                         const uint16_t* w_up, const uint16_t* w_down, uint16_t* y, void* ws,
                         size_t ws_bytes, void* stream);

/* 1 when moe_ffn_fused accepts this shape (a valid shape with H <= 256), else 0. */
int32_t moe_ffn_fused_supported(const moe_shape* shape);

/* Combine (kernel-fusion page, "Expert parallelism: dispatch and combine" and
 * stage 7 "reduce"; residual add of FarSkip-Collective Sec. 3).
 * Plain: out[t, :] = bf16( residual[t, :] + sum_j topk_w[t, j] * y[pair_row[t, j], :] ),
 *        fp32 sum in j order.
 * Dedup: the rank holding the experts first forms one partial row per
 *        (token, rank), partial[d, :] = bf16( sum over the token's j carried by
 *        row d of topk_w[t, j] * y[pair_row[t, j], :] ) (j order), bf16
 *        [N*min(k,W), H]; the owner then sums the token's partials in ascending
 *        rank order and adds the residual.  With partial == NULL one kernel
 *        forms each token's partials in registers (same bf16 rounding, same
 *        orders: bit-identical out) and nothing is written but out; with a
 *        partial buffer the rank side writes the partial rows there (the
 *        message a multi-GPU layer would send) and the owner side reads them.
 * residual may be NULL (out is then the MoE output alone) and out may equal
 * residual (in-place add into the residual stream).  partial is ignored when
 * dedup == 0. */
moe_status moe_combine(const uint16_t* y, const float* topk_w, const moe_layout* layout,
                       const moe_shape* shape, uint16_t* partial, const uint16_t* residual,
                       uint16_t* out, void* stream);

/* Shared expert (FarSkip-Collective Sec. 2.1: "shared-experts" MLP layers run
 * on all tokens in addition to the routed experts): one dense SwiGLU MLP over
 * every token row of x, on the same tensor-core kernels as the routed
 * experts, reading x directly (no dispatch):
 *   h_s = bf16(SiLU(x Wg_s^T) * (x Wu_s^T))   bf16 [N, I_shared]
 *   y_s = bf16(h_s Wd_s^T)                    bf16 [N, H]
 * w_gate_s, w_up_s bf16 [I_shared, H]; w_down_s bf16 [H, I_shared], row-major
 * whatever shape->weights says; I_shared % 8 == 0.  ws: the layer's workspace (a reserved corner holds this
 * call's tile counters). */
moe_status moe_shared_expert_ffn(const uint16_t* x, const moe_shape* shape, int32_t I_shared,
                                 const uint16_t* w_gate_s, const uint16_t* w_up_s,
                                 const uint16_t* w_down_s, uint16_t* h_s, uint16_t* y_s, void* ws,
                                 size_t ws_bytes, void* stream);

/* moe_combine plus the shared expert's output:
 *   out[t, :] = bf16( sum_j topk_w[t, j] * y[pair_row[t, j], :]   (j order; dedup:
 *                     the owner's sum of partials, ascending rank)
 *                     + y_shared[t, :] + residual[t, :] )          fp32 sums
 * y_shared bf16 [N, H] (required); residual nullable; out may equal residual. */
moe_status moe_combine_shared(const uint16_t* y, const float* topk_w, const moe_layout* layout,
                              const moe_shape* shape, uint16_t* partial, const uint16_t* y_shared,
                              const uint16_t* residual, uint16_t* out, void* stream);

/* The whole layer in order on one stream: moe_route, moe_dispatch_layout,
 * moe_dispatch, moe_expert_ffn, moe_combine, with the buffers documented for
 * each of them -- except that, in the plain form, when
 * moe_layer_skips_dispatch(shape) is 1 the dispatch copy is fused into the
 * gate/up GEMM (moe_ffn_gate_up_gather(x, row_token)) and xd is not written.
 * When moe_layer_fuses_ffn(shape) is 1 the expert FFN is moe_ffn_fused
 * (plain: moe_ffn_fused(x, row_token), no dispatch copy; dedup:
 * moe_ffn_fused(xd, expand_src) after moe_dispatch) and h is not written (may
 * be NULL).  xe is not used (may be NULL). */
moe_status moe_layer_forward(const float* logits, const uint16_t* x, const int32_t* placement,
                             const uint16_t* w_gate, const uint16_t* w_up,
                             const uint16_t* w_down, const uint16_t* residual,
                             const moe_shape* shape, int32_t* topk_ids, float* topk_w,
                             const moe_layout* layout, uint16_t* xd, uint16_t* xe, uint16_t* h,
                             uint16_t* y, uint16_t* partial, uint16_t* out, void* ws,
                             size_t ws_bytes, void* stream);

/* 1 when moe_layer_forward, for this shape, gathers the plain rows inside the
 * gate/up GEMM (or inside the fused FFN) instead of running moe_dispatch
 * first; 0 otherwise (dedup form, or a shape whose GEMMs run on the CTA-pair
 * kernel, which has no gather mode).  A function of the shape alone (its gemm
 * field included).  Lets a caller that runs the stages itself do the same. */
int32_t moe_layer_skips_dispatch(const moe_shape* shape);

/* 1 when moe_layer_forward, for this shape, runs the expert FFN as the one
 * fused kernel (moe_ffn_fused: gemm MOE_GEMM_FUSED, or MOE_GEMM_AUTO with
 * H <= 128, or H <= 256 and dedup == 0, and N*k >= 4096 or I <= 256), 0 when
 * it runs the two GEMMs (or the shape is invalid).  A function of the shape
 * alone. */
int32_t moe_layer_fuses_ffn(const moe_shape* shape);

/* Co-selection counts of "Expert Coupling" Sec. V-A / Appendix A-D Algorithm 1:
 * coselect[e*E + e'] = number of tokens whose topk_ids contain both e and e'
 * (symmetric; the diagonal counts the tokens that select e).  coselect is a
 * device int32 [E, E], overwritten.  Integer counts: bit-exact and
 * deterministic.  Ids out of range are reported in the workspace error word
 * and counted as expert 0. */
moe_status moe_coselection(const int32_t* topk_ids, const moe_shape* shape, int32_t* coselect,
                           void* ws, size_t ws_bytes, void* stream);

/* Correlated placement search ("Expert Coupling" Sec. V-A, Appendix A-D
 * Algorithm 1), on the HOST: coselect is a host int32 [E, E] (as written by
 * moe_coselection and copied back), placement a host int32 [E] output.  The
 * experts are partitioned into `ranks` equal groups that keep frequently
 * co-selected experts together: from contiguous groups, the swap of two
 * experts of different groups with the largest gain in within-group
 * co-selection is applied (ties: the pair (a, b), a < b, first in
 * lexicographic order) until no swap gains or max_swaps swaps were made.
 * With nodes > 1 the experts are first split across nodes, then each node's
 * experts (ascending ids) across its ranks/nodes ranks.  Output: slot p holds
 * expert placement[p]; rank r owns slots [r*E/ranks, (r+1)*E/ranks), its
 * experts in ascending id order.  swaps_made (nullable) receives the number of
 * swaps.  Requires nodes | ranks and ranks | E.  Synchronous. */
moe_status moe_placement_search(const int32_t* coselect, int32_t E, int32_t ranks, int32_t nodes,
                                int64_t max_swaps, int32_t* placement, int64_t* swaps_made);

/* moe_dispatch_layout without a workspace argument, for callers that cannot
 * allocate device memory when they call the library (an inference runtime's
 * enqueue path that forbids allocation while it executes, a host whose device
 * memory is entirely owned by its own pool).  The pages have no counterpart:
 * it exists only for such callers.  Same inputs, outputs and results as
 * moe_dispatch_layout; its scratch is a static 1 MiB device array per GPU
 * (held until the process exits), so shapes with moe_workspace_bytes() > 1 MiB
 * return MOE_ERR_WORKSPACE.  It allocates nothing.  Every call on a GPU shares
 * that array: calls that overlap on the GPU race.  The first call on a device
 * looks up the array's address; make it before any stream capture.  That
 * address is kept for the life of the process, so after cudaDeviceReset on a
 * device this entry point must not be called on it again.  Shapes up to
 * N = 253,440 tokens fit at E = 256, W = 8 (697,856 at E = 64, W = 32).
 * Device-detected input problems are not reported by this variant. */
moe_status moe_dispatch_layout_noalloc(const int32_t* topk_ids, const int32_t* placement,
                                       const moe_shape* shape, const moe_layout* layout,
                                       void* stream);

/* Self-test of the device-side wait limit that guards every wait of the
 * kernels (no counterpart in the pages: it checks the library's own failure
 * reporting).  Launches one warp that waits on an mbarrier that nothing
 * completes; after limit_cycles SM clock cycles (1 .. 2^32) the wait gives
 * up, MOE_ERR_TIMEOUT is recorded in the workspace error word (read it with
 * moe_get_error) and the kernel returns, leaving the context usable. */
moe_status moe_selftest_wait_timeout(void* ws, int64_t limit_cycles, void* stream);

/* Synchronizes `stream`, reads the workspace error word, clears it, and
 * returns it (MOE_OK if no device-side problem was recorded). */
moe_status moe_get_error(void* ws, void* stream);

/* Static description of a status code. */
const char* moe_status_str(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
