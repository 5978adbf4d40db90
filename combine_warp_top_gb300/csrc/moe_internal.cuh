// Internal declarations of libmoe: workspace layout, launch helpers shared by
// the kernel files, and the inline-PTX wrappers (mbarrier, TMA, tcgen05) used
// by the grouped GEMM.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kLayoutWarps = 8;                  // warps per layout block
constexpr int kLayoutTokens = 32 * kLayoutWarps;  // tokens per layout block
constexpr int kGemmBM = 128;                      // rows per GEMM tile

// Workspace layout (byte offsets, each 256-aligned).
struct Workspace {
    size_t err;          // int32 error word
    size_t blk_counts;   // int32 [nblk][E]  per-block counts by placement slot
    size_t blk_rcounts;  // int32 [nblk][W]  per-block dedup counts by rank
    size_t slot_start;   // int32 [E+1]      first row of each slot
    size_t mblk_prefix;  // int32 [E+3]      [E+1]: tile counter of the CTA-pair GEMM, [E+2]: its
                         //                  exit counter (both return to 0 after every launch)
    size_t dense;        // int32 [8]        shared expert: count, offsets, tile counters
    size_t total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline int layout_blocks(int N) { return (N + kLayoutTokens - 1) / kLayoutTokens; }

inline Workspace workspace_layout(const moe_shape& s) {
    Workspace w;
    size_t nb = (size_t)layout_blocks(s.N);
    size_t o = 0;
    w.err = o;         o += 256;
    w.blk_counts = o;  o = align256(o + nb * s.E * 4);
    w.blk_rcounts = o; o = align256(o + nb * s.W * 4);
    w.slot_start = o;  o = align256(o + (size_t)(s.E + 1) * 4);
    w.mblk_prefix = o; o = align256(o + (size_t)(s.E + 3) * 4);
    w.dense = o;       o = align256(o + 8 * 4);
    w.total = o;
    return w;
}

template <typename T>
inline T* ws_ptr(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// prefix[e] = sum over experts e' < e of ceil(cnts[e'] / bm) (the GEMM m-blocks
// before expert e), prefix[E] = the total; run by one whole warp over arrays in
// shared memory (each lane scans a contiguous run of experts, then the 32 run
// sums are scanned by shuffles).
__device__ __forceinline__ void warp_mblk_prefix(const int* cnts, int E, int bm, int* prefix) {
    const int lane = threadIdx.x & 31;
    const int per = (E + 31) / 32;
    const int e0 = lane * per, e1 = e0 + per < E ? e0 + per : E;
    int sum = 0;
    for (int e = e0; e < e1; ++e) sum += (cnts[e] + bm - 1) / bm;
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    int run = incl - sum;
    for (int e = e0; e < e1; ++e) {
        prefix[e] = run;
        run += (cnts[e] + bm - 1) / bm;
    }
    if (lane == 31) prefix[E] = incl;
}

// Device-side status recording: the first error sticks.
__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// ---- kernel launchers (one per .cu file) -------------------------------------------

// renorm: softmax over the selected k (true) or the full softmax over E (false).
cudaError_t launch_route(const float* logits, int N, int E, int k, int32_t* ids, float* w,
                         bool renorm, cudaStream_t st);

cudaError_t launch_route_sigmoid(const float* logits, const float* bias, int N, int E, int k,
                                 int32_t* ids, float* w, cudaStream_t st);

cudaError_t launch_layout(const int32_t* ids, const int32_t* placement, const moe_shape& s,
                          const moe_layout& L, void* ws, cudaStream_t st);

cudaError_t launch_dispatch(const uint16_t* x, const moe_layout& L, const moe_shape& s,
                            uint16_t* xd, cudaStream_t st);

cudaError_t launch_expand(const uint16_t* xd, const moe_layout& L, const moe_shape& s,
                          uint16_t* xe, cudaStream_t st);

// shared: nullable [N, H] rows added to every token's output (shared expert).
cudaError_t launch_combine(const uint16_t* y, const float* w, const moe_layout& L,
                           const moe_shape& s, uint16_t* partial, const uint16_t* shared,
                           const uint16_t* residual, uint16_t* out, cudaStream_t st);

// One grouped GEMM problem: R rows in E expert segments (device arrays
// counts[E], offsets[E] of the segments), plus device scratch for the CTA-pair
// kernel's tile counter (prefix[E+1]) and exit counter (prefix[E+2]), both zero
// between launches, and the error word.  Each GEMM derives its tile schedule
// from the counts in its own prologue.
struct GemmGroup {
    const int32_t* counts;
    const int32_t* offsets;
    int E;
    long long R;
    int32_t* prefix;
    int* err;
    bool packed = false;  // weights in the packed layout (moe_pack_weights)
};

// Packed expert weights: blocks of kPackRows x 64 bf16 (32 KB), one per
// (expert, n-block, 64-deep k-block), as rows of a [rows, 64] matrix.  An
// n-block is 128 gate + 128 up columns (gate/up) or 256 output columns (down).
constexpr int kPackRows = 256;
inline long long packed_rows(int E, int n_blocks, int K) {
    return (long long)E * n_blocks * ((K + 63) / 64) * kPackRows;
}
inline long long packed_gate_up_rows(const moe_shape& s) {
    return packed_rows(s.E, (s.I + 127) / 128, s.H);
}
inline long long packed_down_rows(const moe_shape& s) {
    return packed_rows(s.E, (s.H + 255) / 256, s.I);
}

// Inputs of the combine fused into the down GEMM's epilogue: row i of y is
// added, times its routing weight, into acc[row_token[i], :] (fp32 [N, H]).
struct CombineArgs {
    const int32_t* row_token;  // [N*k]
    const int32_t* pair_row;   // [N*k]
    const float* topk_w;       // [N*k]
    float* acc;                // [N, H]
    int N;
    int k;
};

// Return MOE_OK, or an error status when a host-side step (tensor-map
// encoding, launch) failed.
// gather != nullptr: problem row i is row gather[i] of `rows` ([src_rows, H]),
// copied into shared memory by the GEMM's gather warps instead of a prior copy.
moe_status launch_gate_up(const uint16_t* rows, const GemmGroup& g, int H, int I,
                          const uint16_t* wg, const uint16_t* wu, uint16_t* h, cudaStream_t st,
                          const int32_t* gather = nullptr, long long src_rows = 0);
moe_status launch_down_combine(const uint16_t* h, const GemmGroup& g, int H, int I,
                               const uint16_t* wd, const CombineArgs& cmb, cudaStream_t st);
cudaError_t launch_acc_finish(const float* acc, const uint16_t* residual, int N, int H,
                              uint16_t* out, cudaStream_t st);
moe_status launch_down(const uint16_t* h, const GemmGroup& g, int H, int I, const uint16_t* wd,
                       uint16_t* y, cudaStream_t st);
// One warp waits on an mbarrier that never completes, up to limit_cycles.
cudaError_t launch_wait_selftest(long long limit_cycles, int* err, cudaStream_t st);
// counts = {N}, offsets = {0, N}: one dense segment of N rows.
cudaError_t launch_dense_group(int N, int32_t* counts, int32_t* offsets, cudaStream_t st);

// moe_pack_weights (pack.cu): either output may be null.
cudaError_t launch_pack(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                        const moe_shape& s, uint16_t* gate_up, uint16_t* down, cudaStream_t st);

cudaError_t launch_coselection(const int32_t* ids, const moe_shape& s, int32_t* W, int* err,
                               cudaStream_t st);

// Host-only: balanced best-swap partition of Algorithm 1 (placement.cu).
moe_status placement_search(const int32_t* W, int E, int ranks, int nodes, long long max_swaps,
                            int32_t* placement, long long* swaps_made);

// Tensor maps (bf16, 128-byte swizzle, zero fill; grouped_gemm.cu), shared by
// the single-CTA and the CTA-pair GEMMs.
bool map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
bool map_3d(CUtensorMap* m, const void* ptr, uint64_t E, uint64_t rows, uint64_t cols,
            uint32_t box_rows);
bool map_packed(CUtensorMap* m, CUtensorMap* second, const void* ptr, int E, int n_blocks, int K,
                uint32_t box_rows);

// CTA-pair GEMMs (grouped_gemm_2sm.cu): 256-row tiles on tcgen05 cta_group::2.
moe_status launch_gate_up_pair(const uint16_t* rows, const GemmGroup& g, int H, int I,
                               const uint16_t* wg, const uint16_t* wu, uint16_t* h,
                               cudaStream_t st);
moe_status launch_down_pair(const uint16_t* h, const GemmGroup& g, int H, int I,
                            const uint16_t* wd, uint16_t* y, cudaStream_t st);

// The expert FFN in one kernel with h kept on chip (fused_ffn.cu): y for the
// problem's rows, gathered like launch_gate_up's (row_index == nullptr: row i
// of src).  Needs H <= kFusedMaxH (the 128 x H fp32 y tile lives in TMEM).
// From I = kFusedWideMinI on, the form on 128-column chunks of I
// (fused_ffn_wide.cu) runs instead of the 64-column one; same results.
constexpr int kFusedMaxH = 256;
constexpr int kFusedWideMinI = 1024;
bool fused_ffn_supported(int H);
moe_status launch_ffn_fused(const uint16_t* src, const int32_t* row_index, long long src_rows,
                            const GemmGroup& g, int H, int I, const uint16_t* wg,
                            const uint16_t* wu, const uint16_t* wd, uint16_t* y,
                            cudaStream_t st);
moe_status launch_ffn_fused_wide(const uint16_t* src, const int32_t* row_index,
                                 long long src_rows, const GemmGroup& g, int H, int I,
                                 const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                                 uint16_t* y, cudaStream_t st);

int sm_count();

}  // namespace moe
