// Dispatch: copy token rows into the per-expert (plain) or per-rank (dedup)
// receive buffers, and the receiver's expansion of dedup rows into
// expert-major order.
//
// "Kernel fusion for expert parallelism", section "Expert parallelism:
// dispatch and combine" (the dispatch sends each token to the ranks that hold
// its experts) and the Baseline's "pack" stage of "Fusing the layer into one
// kernel"; "Expert Coupling" Sec. V-A (one copy per unique (token, rank)) and
// Appendix A-A2 (the receiver expands the rows into expert-major order).
//
// The copy is source-major: a token's row is read once with 16-byte loads and
// stored to each destination, so x is read from HBM exactly once whatever k
// is.  One warp handles one slice of 32*kUnroll chunks of one row, so a long
// row is spread over several warps that each make a single round trip.  Rows
// are bit-exact copies.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte chunks in flight per lane

__device__ __forceinline__ int clamp_row(int r, int bound) {
    return (unsigned)r < (unsigned)bound ? r : 0;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// dest_of_pair: pair_row (plain) or pair_dedup_row (dedup), [N*k].  Warp g
// copies slice g % slices of token g / slices.
__global__ void __launch_bounds__(kThreads)
    dispatch_kernel(const uint4* __restrict__ x, int N, int C, int k,
                    const int32_t* __restrict__ dest_of_pair, int dedup, int row_bound,
                    uint4* __restrict__ xd) {
    const int lane = threadIdx.x & 31;
    const long long g = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const int slices = (C + 32 * kUnroll - 1) / (32 * kUnroll);
    const int t = (int)(g / slices);
    const int cs = (int)(g % slices) * 32 * kUnroll;
    if (t >= N) return;
    int d = lane < k ? clamp_row(dest_of_pair[(size_t)t * k + lane], row_bound) : -1;
    bool keep = lane < k;
    if (dedup) {
        // several experts of the token on one rank share one dedup row: copy once
        for (int jj = 0; jj < k; ++jj) {
            const int o = __shfl_sync(0xffffffffu, d, jj);
            if (jj < lane && o == d) keep = false;
        }
    }
    const uint32_t dests = __ballot_sync(0xffffffffu, keep);
    const uint4* src = x + (size_t)t * C;
    {
        const int c0 = cs;
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) v[u] = ld_stream(src + c);
        }
        uint32_t m = dests;
        while (m) {
            const int j = __ffs(m) - 1;
            m &= m - 1;
            const int dj = __shfl_sync(0xffffffffu, d, j);
            uint4* dst = xd + (size_t)dj * C;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < C) dst[c] = v[u];
            }
        }
    }
}

// xe[i] = xd[expand_src[i]] for the R = N*k expert-major rows.
__global__ void __launch_bounds__(kThreads) expand_kernel(const uint4* __restrict__ xd, int R,
                                                          int C,
                                                          const int32_t* __restrict__ expand_src,
                                                          int src_bound, uint4* __restrict__ xe) {
    const int lane = threadIdx.x & 31;
    const int i = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    if (i >= R) return;
    const int s = clamp_row(expand_src[i], src_bound);
    const uint4* src = xd + (size_t)s * C;
    uint4* dst = xe + (size_t)i * C;
    for (int c0 = 0; c0 < C; c0 += 32 * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) v[u] = src[c];
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) dst[c] = v[u];
        }
    }
}

inline int warps_grid(long long n) { return (int)((n + kThreads / 32 - 1) / (kThreads / 32)); }

}  // namespace

cudaError_t launch_dispatch(const uint16_t* x, const moe_layout& L, const moe_shape& s,
                            uint16_t* xd, cudaStream_t st) {
    if (s.N == 0) return cudaSuccess;
    const int C = s.H / 8;
    const int rows = s.dedup ? s.N * (s.k < s.W ? s.k : s.W) : s.N * s.k;
    const long long slices = (C + 32 * kUnroll - 1) / (32 * kUnroll);
    dispatch_kernel<<<warps_grid(s.N * slices), kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(x), s.N, C, s.k, s.dedup ? L.pair_dedup_row : L.pair_row,
        s.dedup, rows, reinterpret_cast<uint4*>(xd));
    return cudaGetLastError();
}

cudaError_t launch_expand(const uint16_t* xd, const moe_layout& L, const moe_shape& s,
                          uint16_t* xe, cudaStream_t st) {
    const int R = s.N * s.k;
    if (R == 0) return cudaSuccess;
    const int C = s.H / 8;
    const int bound = s.N * (s.k < s.W ? s.k : s.W);
    expand_kernel<<<warps_grid(R), kThreads, 0, st>>>(reinterpret_cast<const uint4*>(xd), R, C,
                                                      L.expand_src, bound,
                                                      reinterpret_cast<uint4*>(xe));
    return cudaGetLastError();
}

}  // namespace moe
