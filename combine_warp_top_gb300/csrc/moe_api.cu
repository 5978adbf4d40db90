// C ABI entry points of libmoe: argument checks, workspace sizing, and the
// chaining of the kernels of the other files on the caller's stream.
// Declarations and the contract of every call are in include/moe.h.
#include <nvtx3/nvToolsExt.h>

#include "moe_internal.cuh"

namespace moe {

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 1;
    if (dev < 64) cached[dev] = n;
    return n;
}

namespace {

moe_status check_shape(const moe_shape* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->N < 0 || s->H <= 0 || s->E <= 0 || s->k <= 0 || s->W <= 0 || s->I <= 0)
        return MOE_ERR_INVALID_ARG;
    if (s->k > s->E || s->E % s->W != 0) return MOE_ERR_INVALID_ARG;
    if (s->E > kMaxE || s->k > kMaxK) return MOE_ERR_UNSUPPORTED;
    if (s->H % 8 != 0 || s->I % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)s->N * s->k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (s->gemm != MOE_GEMM_AUTO && s->gemm != MOE_GEMM_SINGLE_CTA &&
        s->gemm != MOE_GEMM_CTA_PAIR && s->gemm != MOE_GEMM_FUSED)
        return MOE_ERR_INVALID_ARG;
    if (s->gemm == MOE_GEMM_FUSED && !fused_ffn_supported(s->H)) return MOE_ERR_UNSUPPORTED;
    if (s->weights != MOE_WEIGHTS_ROW_MAJOR && s->weights != MOE_WEIGHTS_PACKED)
        return MOE_ERR_INVALID_ARG;
    // the GEMMs address packed rows with 32-bit TMA coordinates
    if (s->weights == MOE_WEIGHTS_PACKED &&
        (packed_gate_up_rows(*s) >= (1LL << 31) || packed_down_rows(*s) >= (1LL << 31)))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// w_up is read only in the row-major layout (the packed gate/up weights hold both).
inline bool up_given(const moe_shape* s, const uint16_t* w_up) {
    return w_up != nullptr || s->weights == MOE_WEIGHTS_PACKED;
}

moe_status check_layout(const moe_layout* L, const moe_shape* s) {
    if (!L) return MOE_ERR_INVALID_ARG;
    if (!L->expert_counts || !L->expert_offsets || !L->rank_offsets || !L->row_token ||
        !L->pair_row)
        return MOE_ERR_INVALID_ARG;
    if (s->dedup && (!L->dedup_counts || !L->dedup_offsets || !L->dedup_row_token ||
                     !L->pair_dedup_row || !L->expand_src || !L->n_dedup_rows))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status check_ws(const moe_shape* s, void* ws, size_t ws_bytes) {
    if (!ws || ws_bytes < workspace_layout(*s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// CTA-pair (256-row) GEMM tiles pay off when experts have many rows; with few
// rows per expert the single-CTA 128-row tiles waste less.  The shape's gemm
// field can name either kernel instead of the automatic choice.
bool use_pair(long long R, int E, int32_t gemm) {
    if (gemm == MOE_GEMM_SINGLE_CTA || gemm == MOE_GEMM_FUSED) return false;
    if (gemm == MOE_GEMM_CTA_PAIR) return true;
    return R >= 512LL * E;
}

// moe_layer_forward runs the expert FFN as one kernel with h on chip when the
// shape names it, and by default for H <= 128, and for H <= 256 in the plain
// form: there it measured faster than the two GEMMs on all but two of the
// shapes tried (h never goes to HBM and one launch goes); on dedup layers
// with H = 256 the two GEMMs (gathered gate/up) were faster.  One CTA walks
// all of I for its 128-row tile, so a layer with few rows and a long I
// (N*k < 4096 rows and I > 256) keeps the two GEMMs, which spread over I.
constexpr int kAutoFusedMaxH = 128;        // any form
constexpr int kAutoFusedMaxHPlain = 256;   // the plain form
constexpr long long kAutoFusedMinRows = 4096;
constexpr int kAutoFusedShortI = 256;
bool layer_fuses_ffn(const moe_shape& s) {
    if (s.gemm == MOE_GEMM_FUSED) return true;
    if (s.gemm != MOE_GEMM_AUTO || !fused_ffn_supported(s.H)) return false;
    if (s.H > (s.dedup ? kAutoFusedMaxH : kAutoFusedMaxHPlain)) return false;
    return (long long)s.N * s.k >= kAutoFusedMinRows || s.I <= kAutoFusedShortI;
}

// The routed experts' GEMM problem: the plain expert-major rows of the layout.
GemmGroup routed_group(const moe_layout& L, const moe_shape& s, void* ws) {
    const Workspace wl = workspace_layout(s);
    return GemmGroup{L.expert_counts, L.expert_offsets, s.E, (long long)s.N * s.k,
                     ws_ptr<int32_t>(ws, wl.mblk_prefix), ws_ptr<int>(ws, wl.err),
                     s.weights == MOE_WEIGHTS_PACKED};
}

// The shared expert's GEMM problem: all N token rows as one segment.
GemmGroup dense_group(const moe_shape& s, void* ws) {
    const Workspace wl = workspace_layout(s);
    int32_t* d = ws_ptr<int32_t>(ws, wl.dense);
    return GemmGroup{d, d + 1, 1, (long long)s.N, d + 4, ws_ptr<int>(ws, wl.err)};
}

inline cudaStream_t as_stream(void* p) { return reinterpret_cast<cudaStream_t>(p); }

// The kernels move bf16 rows (and the fp32 accumulator) in 16-byte vectors,
// by TMA, cp.async or plain vector loads: a base address that is not 16-byte
// aligned is refused here instead of faulting on the device.  NULL passes
// (whether NULL is allowed is checked separately).
template <typename... T>
inline bool aligned16(const T*... p) {
    return ((((uintptr_t)p & 15u) == 0) && ...);
}

// An NVTX range named after the entry point around every call that enqueues
// work: profilers (Nsight Systems, ncu's NVTX filters) show the C ABI calls on
// the timeline.  With no tool attached a push/pop is a check of one function
// pointer.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define MOE_RANGE() const NvtxRange _moe_nvtx_range(__func__)

#define MOE_TRY(expr)                     \
    do {                                  \
        const moe_status _st = (expr);    \
        if (_st != MOE_OK) return _st;    \
    } while (0)

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    return workspace_layout(*shape).total;
}

size_t moe_packed_gate_up_bytes(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    return (size_t)packed_gate_up_rows(*shape) * 64 * sizeof(uint16_t);
}

size_t moe_packed_down_bytes(const moe_shape* shape) {
    if (check_shape(shape) != MOE_OK) return 0;
    return (size_t)packed_down_rows(*shape) * 64 * sizeof(uint16_t);
}

moe_status moe_pack_weights(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                            const moe_shape* shape, uint16_t* gate_up_packed,
                            uint16_t* down_packed, void* stream) {
    MOE_RANGE();
    if (!shape) return MOE_ERR_INVALID_ARG;
    moe_shape s = *shape;
    s.weights = MOE_WEIGHTS_ROW_MAJOR;  // not read here
    MOE_TRY(check_shape(&s));
    if (gate_up_packed && (!w_gate || !w_up)) return MOE_ERR_INVALID_ARG;
    if (down_packed && !w_down) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate, w_up, w_down, gate_up_packed, down_packed)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pack(w_gate, w_up, w_down, s, gate_up_packed, down_packed,
                                   as_stream(stream)));
}

moe_status moe_route(const float* logits, const moe_shape* shape, int32_t* topk_ids,
                     float* topk_w, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    if (shape->N == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route(logits, shape->N, shape->E, shape->k, topk_ids, topk_w, true,
                                    as_stream(stream)));
}

moe_status moe_route_full_softmax(const float* logits, const moe_shape* shape, int32_t* topk_ids,
                                  float* topk_w, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    if (shape->N == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route(logits, shape->N, shape->E, shape->k, topk_ids, topk_w, false,
                                    as_stream(stream)));
}

moe_status moe_route_sigmoid_bias(const float* logits, const float* bias, const moe_shape* shape,
                                  int32_t* topk_ids, float* topk_w, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    if (shape->N == 0) return MOE_OK;
    if (!logits || !bias || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route_sigmoid(logits, bias, shape->N, shape->E, shape->k, topk_ids,
                                            topk_w, as_stream(stream)));
}

moe_status moe_dispatch_layout(const int32_t* topk_ids, const int32_t* placement,
                               const moe_shape* shape, const moe_layout* layout, void* ws,
                               size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N > 0 && !topk_ids) return MOE_ERR_INVALID_ARG;
    return cuda_status(
        launch_layout(topk_ids, placement, *shape, *layout, ws, as_stream(stream)));
}

moe_status moe_dispatch(const uint16_t* x, const moe_layout* layout, const moe_shape* shape,
                        uint16_t* xd, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    if (shape->N == 0) return MOE_OK;
    if (!x || !xd) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x, xd)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_dispatch(x, *layout, *shape, xd, as_stream(stream)));
}

moe_status moe_expand(const uint16_t* xd, const moe_layout* layout, const moe_shape* shape,
                      uint16_t* xe, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    if (!shape->dedup) return MOE_ERR_INVALID_ARG;
    if (shape->N == 0) return MOE_OK;
    if (!xd || !xe) return MOE_ERR_INVALID_ARG;
    if (!aligned16(xd, xe)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_expand(xd, *layout, *shape, xe, as_stream(stream)));
}

moe_status moe_ffn_gate_up(const uint16_t* rows, const moe_layout* layout, const moe_shape* shape,
                           const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h, void* ws,
                           size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    if (!rows || !w_gate || !up_given(shape, w_up) || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned16(rows, w_gate, w_up, h)) return MOE_ERR_INVALID_ARG;
    const GemmGroup g = routed_group(*layout, *shape, ws);
    if (use_pair(g.R, g.E, shape->gemm))
        return launch_gate_up_pair(rows, g, shape->H, shape->I, w_gate, w_up, h, as_stream(stream));
    return launch_gate_up(rows, g, shape->H, shape->I, w_gate, w_up, h, as_stream(stream));
}

moe_status moe_ffn_gate_up_gather(const uint16_t* src, const int32_t* row_index, int64_t src_rows,
                                  const moe_layout* layout, const moe_shape* shape,
                                  const uint16_t* w_gate, const uint16_t* w_up, uint16_t* h,
                                  void* ws, size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    if (!src || !row_index || !w_gate || !up_given(shape, w_up) || !h)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(src, w_gate, w_up, h)) return MOE_ERR_INVALID_ARG;
    if (src_rows <= 0 || src_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
    return launch_gate_up(src, routed_group(*layout, *shape, ws), shape->H, shape->I, w_gate, w_up,
                          h, as_stream(stream), row_index, src_rows);
}

moe_status moe_ffn_down(const uint16_t* h, const moe_layout* layout, const moe_shape* shape,
                        const uint16_t* w_down, uint16_t* y, void* ws, size_t ws_bytes,
                        void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    if (!h || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h, w_down, y)) return MOE_ERR_INVALID_ARG;
    const GemmGroup g = routed_group(*layout, *shape, ws);
    if (use_pair(g.R, g.E, shape->gemm))
        return launch_down_pair(h, g, shape->H, shape->I, w_down, y, as_stream(stream));
    return launch_down(h, g, shape->H, shape->I, w_down, y, as_stream(stream));
}

moe_status moe_ffn_down_combine(const uint16_t* h, const float* topk_w, const moe_layout* layout,
                                const moe_shape* shape, const uint16_t* w_down,
                                const uint16_t* residual, float* acc, uint16_t* out, void* ws,
                                size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    if (!h || !topk_w || !w_down || !acc || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(h, w_down, residual, acc, out)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(acc, 0, (size_t)shape->N * shape->H * sizeof(float), st) != cudaSuccess)
        return MOE_ERR_CUDA;
    const CombineArgs cmb{layout->row_token, layout->pair_row, topk_w, acc, shape->N, shape->k};
    MOE_TRY(launch_down_combine(h, routed_group(*layout, *shape, ws), shape->H, shape->I, w_down,
                                cmb, st));
    return cuda_status(launch_acc_finish(acc, residual, shape->N, shape->H, out, st));
}

moe_status moe_ffn_fused(const uint16_t* src, const int32_t* row_index, int64_t src_rows,
                         const moe_layout* layout, const moe_shape* shape, const uint16_t* w_gate,
                         const uint16_t* w_up, const uint16_t* w_down, uint16_t* y, void* ws,
                         size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (!fused_ffn_supported(shape->H)) return MOE_ERR_UNSUPPORTED;
    if (shape->N == 0) return MOE_OK;
    if (!src || !w_gate || !up_given(shape, w_up) || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(src, w_gate, w_up, w_down, y)) return MOE_ERR_INVALID_ARG;
    if (src_rows <= 0 || src_rows >= ((int64_t)1 << 31)) return MOE_ERR_INVALID_ARG;
    // without an index the problem's rows are the first N*k rows of src
    if (!row_index && src_rows < (int64_t)shape->N * shape->k) return MOE_ERR_INVALID_ARG;
    return launch_ffn_fused(src, row_index, src_rows, routed_group(*layout, *shape, ws), shape->H,
                            shape->I, w_gate, w_up, w_down, y, as_stream(stream));
}

int32_t moe_ffn_fused_supported(const moe_shape* shape) {
    return shape && check_shape(shape) == MOE_OK && fused_ffn_supported(shape->H) ? 1 : 0;
}

moe_status moe_expert_ffn(const uint16_t* xd, const moe_layout* layout, const moe_shape* shape,
                          const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          uint16_t* xe, uint16_t* h, uint16_t* y, void* ws, size_t ws_bytes,
                          void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    const bool fused = shape->gemm == MOE_GEMM_FUSED;  // h stays on chip: not written
    if (!xd || !w_gate || !up_given(shape, w_up) || !w_down || (!h && !fused) || !y)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(xd, w_gate, w_up, w_down, h, y)) return MOE_ERR_INVALID_ARG;
    (void)xe;
    const int64_t rd_max = (int64_t)shape->N * (shape->k < shape->W ? shape->k : shape->W);
    if (fused)
        return shape->dedup ? moe_ffn_fused(xd, layout->expand_src, rd_max, layout, shape, w_gate,
                                            w_up, w_down, y, ws, ws_bytes, stream)
                            : moe_ffn_fused(xd, nullptr, (int64_t)shape->N * shape->k, layout,
                                            shape, w_gate, w_up, w_down, y, ws, ws_bytes, stream);
    if (shape->dedup) {
        // the expansion to expert-major order is done by the GEMM's gather
        // warps: cheaper than writing the N*k rows out and reading them back
        MOE_TRY(moe_ffn_gate_up_gather(xd, layout->expand_src, rd_max, layout, shape, w_gate,
                                       w_up, h, ws, ws_bytes, stream));
    } else {
        MOE_TRY(moe_ffn_gate_up(xd, layout, shape, w_gate, w_up, h, ws, ws_bytes, stream));
    }
    return moe_ffn_down(h, layout, shape, w_down, y, ws, ws_bytes, stream);
}

moe_status moe_combine(const uint16_t* y, const float* topk_w, const moe_layout* layout,
                       const moe_shape* shape, uint16_t* partial, const uint16_t* residual,
                       uint16_t* out, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    if (shape->N == 0) return MOE_OK;
    if (!y || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y, partial, residual, out)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(y, topk_w, *layout, *shape, partial, nullptr, residual, out,
                                      as_stream(stream)));
}

moe_status moe_shared_expert_ffn(const uint16_t* x, const moe_shape* shape, int32_t I_shared,
                                 const uint16_t* w_gate_s, const uint16_t* w_up_s,
                                 const uint16_t* w_down_s, uint16_t* h_s, uint16_t* y_s, void* ws,
                                 size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (I_shared <= 0) return MOE_ERR_INVALID_ARG;
    if (I_shared % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (shape->N == 0) return MOE_OK;
    if (!x || !w_gate_s || !w_up_s || !w_down_s || !h_s || !y_s) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x, w_gate_s, w_up_s, w_down_s, h_s, y_s)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    const GemmGroup g = dense_group(*shape, ws);
    MOE_TRY(cuda_status(launch_dense_group(shape->N, const_cast<int32_t*>(g.counts),
                                           const_cast<int32_t*>(g.offsets), st)));
    if (use_pair(g.R, g.E, shape->gemm)) {
        MOE_TRY(launch_gate_up_pair(x, g, shape->H, I_shared, w_gate_s, w_up_s, h_s, st));
        return launch_down_pair(h_s, g, shape->H, I_shared, w_down_s, y_s, st);
    }
    MOE_TRY(launch_gate_up(x, g, shape->H, I_shared, w_gate_s, w_up_s, h_s, st));
    return launch_down(h_s, g, shape->H, I_shared, w_down_s, y_s, st);
}

moe_status moe_combine_shared(const uint16_t* y, const float* topk_w, const moe_layout* layout,
                              const moe_shape* shape, uint16_t* partial, const uint16_t* y_shared,
                              const uint16_t* residual, uint16_t* out, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    if (shape->N == 0) return MOE_OK;
    if (!y || !topk_w || !out || !y_shared) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y, partial, y_shared, residual, out)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(y, topk_w, *layout, *shape, partial, y_shared, residual, out,
                                      as_stream(stream)));
}

moe_status moe_layer_forward(const float* logits, const uint16_t* x, const int32_t* placement,
                             const uint16_t* w_gate, const uint16_t* w_up,
                             const uint16_t* w_down, const uint16_t* residual,
                             const moe_shape* shape, int32_t* topk_ids, float* topk_w,
                             const moe_layout* layout, uint16_t* xd, uint16_t* xe, uint16_t* h,
                             uint16_t* y, uint16_t* partial, uint16_t* out, void* ws,
                             size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_layout(layout, shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (shape->N == 0) return MOE_OK;
    const bool fused = layer_fuses_ffn(*shape);  // h stays on chip: not written
    if (!logits || !x || !w_gate || !up_given(shape, w_up) || !w_down || !topk_ids ||
        !topk_w || !xd || (!h && !fused) || !y || !out)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x, w_gate, w_up, w_down, residual, xd, xe, h, y, partial, out))
        return MOE_ERR_INVALID_ARG;
    MOE_TRY(moe_route(logits, shape, topk_ids, topk_w, stream));
    MOE_TRY(moe_dispatch_layout(topk_ids, placement, shape, layout, ws, ws_bytes, stream));
    if (moe_layer_skips_dispatch(shape) && fused) {
        // dispatch copy, both GEMMs and SwiGLU in one kernel: rows of x through row_token
        MOE_TRY(moe_ffn_fused(x, layout->row_token, shape->N, layout, shape, w_gate, w_up, w_down,
                              y, ws, ws_bytes, stream));
    } else if (moe_layer_skips_dispatch(shape)) {
        // the dispatch copy fused into the gate/up GEMM: rows of x through row_token
        MOE_TRY(moe_ffn_gate_up_gather(x, layout->row_token, shape->N, layout, shape, w_gate,
                                       w_up, h, ws, ws_bytes, stream));
        MOE_TRY(moe_ffn_down(h, layout, shape, w_down, y, ws, ws_bytes, stream));
    } else if (fused) {
        // only the dedup form dispatches before the fused FFN: its dedup rows
        // are expanded to expert-major order by the kernel's gather warps
        MOE_TRY(moe_dispatch(x, layout, shape, xd, stream));
        const int64_t rd_max = (int64_t)shape->N * (shape->k < shape->W ? shape->k : shape->W);
        MOE_TRY(moe_ffn_fused(xd, layout->expand_src, rd_max, layout, shape, w_gate, w_up,
                              w_down, y, ws, ws_bytes, stream));
    } else {
        MOE_TRY(moe_dispatch(x, layout, shape, xd, stream));
        MOE_TRY(moe_expert_ffn(xd, layout, shape, w_gate, w_up, w_down, xe, h, y, ws, ws_bytes,
                               stream));
    }
    return moe_combine(y, topk_w, layout, shape, partial, residual, out, stream);
}

int32_t moe_layer_fuses_ffn(const moe_shape* shape) {
    return shape && check_shape(shape) == MOE_OK && layer_fuses_ffn(*shape) ? 1 : 0;
}

int32_t moe_layer_skips_dispatch(const moe_shape* shape) {
    if (!shape || check_shape(shape) != MOE_OK || shape->dedup) return 0;
    // the fused FFN gathers its plain rows from x itself
    if (layer_fuses_ffn(*shape)) return 1;
    // plain rows are gathered when the single-CTA GEMM runs (the weight-streaming
    // regime, where fusing the copy saves its HBM traffic); the CTA-pair kernel
    // has no gather mode
    return use_pair((long long)shape->N * shape->k, shape->E, shape->gemm) ? 0 : 1;
}

moe_status moe_coselection(const int32_t* topk_ids, const moe_shape* shape, int32_t* coselect,
                           void* ws, size_t ws_bytes, void* stream) {
    MOE_RANGE();
    MOE_TRY(check_shape(shape));
    MOE_TRY(check_ws(shape, ws, ws_bytes));
    if (!coselect || (shape->N > 0 && !topk_ids)) return MOE_ERR_INVALID_ARG;
    int* err = ws_ptr<int>(ws, workspace_layout(*shape).err);
    return cuda_status(
        launch_coselection(topk_ids, *shape, coselect, err, as_stream(stream)));
}

moe_status moe_placement_search(const int32_t* coselect, int32_t E, int32_t ranks, int32_t nodes,
                                int64_t max_swaps, int32_t* placement, int64_t* swaps_made) {
    MOE_RANGE();
    if (!coselect || !placement || E <= 0 || ranks <= 0 || nodes <= 0 || max_swaps < 0)
        return MOE_ERR_INVALID_ARG;
    if (ranks % nodes != 0 || E % ranks != 0) return MOE_ERR_INVALID_ARG;
    long long made = 0;
    const moe_status st = placement_search(coselect, E, ranks, nodes, max_swaps, placement, &made);
    if (swaps_made) *swaps_made = made;
    return st;
}

moe_status moe_selftest_wait_timeout(void* ws, int64_t limit_cycles, void* stream) {
    MOE_RANGE();
    if (!ws) return MOE_ERR_WORKSPACE;
    if (limit_cycles <= 0 || limit_cycles > (int64_t)1 << 32) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_wait_selftest(limit_cycles, ws_ptr<int>(ws, 0), as_stream(stream)));
}

moe_status moe_get_error(void* ws, void* stream) {
    MOE_RANGE();
    if (!ws) return MOE_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    int code = 0;
    if (cudaMemcpyAsync(&code, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (code != 0) {
        if (cudaMemsetAsync(ws, 0, sizeof(int), st) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return (moe_status)code;
}

const char* moe_status_str(moe_status status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_DEVICE_ASSERT: return "device-side check failed";
    }
    return "unknown status";
}

}  // extern "C"
