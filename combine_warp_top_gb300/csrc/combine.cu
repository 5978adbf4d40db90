// Combine: the router-weighted sum of each token's k expert outputs, fused
// with the residual add.
//
// "Kernel fusion for expert parallelism", section "Expert parallelism:
// dispatch and combine" (the combine returns the weighted outputs to the token's
// owner, which sums them; Sigma_t = sigma^0_t + ... + sigma^{W-1}_t) and stage 7
// "reduce" of "Fusing the layer into one kernel" (each expert output scaled by
// its routing weight and accumulated into the rank's partial); "Expert
// Coupling" Sec. V-A (dedup: one partial per (token, rank), summed by the
// owner); FarSkip-Collective Sec. 3 (the layer output is added into the
// residual stream).
//
// The plain combine runs on persistent warps that each walk units of (token,
// 2 x 512-byte column stripes; 4 when k <= 2), with the next unit's row
// indices loaded while the current unit's rows are in flight.  The dedup
// kernels take one warp per output row; each lane owns U 16-byte chunks (8
// bf16 each) per step along the row, the source rows of a chunk are loaded
// together, then accumulated in fp32 in j order.  These are latency-bound
// chains of loads, so the kernels are compiled with register caps that keep
// 16-32 warps per SM in flight.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;  // source rows loaded together
// Dedup combine: one 16-byte chunk per lane and step, up to eight source rows
// loaded together, at 60 registers (32 warps per SM).  Wider chunks need a
// second set of fp32 partials and halve the warps per SM; at four chunks the
// kernel ran 1.85x slower on the k = 6 correlated shape.
constexpr int kDedupU = 1;
constexpr int kDedupB = 8;

__device__ __forceinline__ int clamp_row(int r, int bound) {
    return (unsigned)r < (unsigned)bound ? r : 0;
}

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4& v, float w) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
    }
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
    uint4 o;
    __nv_bfloat162* q = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    return o;
}

// acc[u] += sum over the set bits j of `srcs` (ascending) of w_j * rows[row_j][c_u]
// for U chunks c_u = c0 + u*32 + lane at once, where lane j holds row_j / w_j.
// Loads of up to kLoads (row, chunk) pairs are issued before any is used.
// Warp-uniform control flow.
template <int U>
__device__ __forceinline__ void gather_weighted(float (&acc)[U][8], const uint4* __restrict__ rows,
                                                int C, int c0, uint32_t srcs, int my_row,
                                                float my_w) {
    constexpr int kRows = kBatch / U > 0 ? kBatch / U : 1;  // source rows per batch
    const int lane = threadIdx.x & 31;
    while (srcs) {
        uint4 v[kRows][U];
        int js[kRows];
        int n = 0;
#pragma unroll
        for (int b = 0; b < kRows; ++b) {
            js[b] = 0;
            if (srcs) {
                js[b] = __ffs(srcs) - 1;
                srcs &= srcs - 1;
                n = b + 1;
            }
        }
#pragma unroll
        for (int b = 0; b < kRows; ++b) {
            if (b < n) {
                const int r = __shfl_sync(0xffffffffu, my_row, js[b]);
                const uint4* src = rows + (size_t)r * C;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * 32 + lane;
                    if (c < C) v[b][u] = src[c];
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kRows; ++b) {
            if (b < n) {
                const float w = __shfl_sync(0xffffffffu, my_w, js[b]);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + u * 32 + lane;
                    if (c < C) acc_bf16x8(acc[u], v[b][u], w);
                }
            }
        }
    }
}

template <int U>
__device__ __forceinline__ void zero(float (&acc)[U][8]) {
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
}

// out[c] = bf16(acc (+ shared[c]) (+ residual[c])) for the U chunks of this lane.
// With several chunks per lane all their loads are issued before any add;
// with one, the load-add-store chain per chunk measured faster.
template <int U>
__device__ __forceinline__ void finish(float (&acc)[U][8], const uint4* shared,
                                       const uint4* residual, uint4* out, size_t row_base, int C,
                                       int c0) {
    const int lane = threadIdx.x & 31;
    if constexpr (U == 1) {
        const int c = c0 + lane;
        if (c < C) {
            if (shared) add_bf16x8(acc[0], shared[row_base + c]);
            if (residual) add_bf16x8(acc[0], residual[row_base + c]);
            out[row_base + c] = pack_bf16x8(acc[0]);
        }
    } else {
        uint4 r[U], sh[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) {
                if (shared) sh[u] = shared[row_base + c];
                if (residual) r[u] = residual[row_base + c];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) {
                if (shared) add_bf16x8(acc[u], sh[u]);
                if (residual) add_bf16x8(acc[u], r[u]);
                out[row_base + c] = pack_bf16x8(acc[u]);
            }
        }
    }
}

// Plain combine, persistent: warps walk units (token t, group of kU stripes of
// 32 lanes x 16 bytes); lane l covers chunks s*32*kU + q*32 + l (q < kU) of the
// token's k source rows, the shared row and the residual.  All loads of a unit
// are issued before any is used (source rows kKB at a time), and the pair_row
// and topk_w entries of the warp's NEXT unit are loaded while this unit's rows
// are in flight, so no unit waits on its own index load.  Sums in j order in
// fp32, then + shared, then + residual:
// out[t] = bf16(residual[t] + shared[t] + sum_j w[t,j] * y[pair_row[t,j]]).
template <int kU, int kKB, bool kShared, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) combine_rows_kernel(
    const uint4* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ pair_row, int N, int C, int k, int R, int groups,
    const uint4* __restrict__ shared, const uint4* __restrict__ residual,
    uint4* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long units = (long long)N * groups;
    long long u = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    int next_row = 0;
    float next_w = 0.f;
    if (u < units && lane < k) {
        const size_t i = (size_t)(u / groups) * k + lane;
        next_row = clamp_row(pair_row[i], R);
        next_w = topk_w[i];
    }
    for (; u < units; u += nwarps) {
        const int t = (int)(u / groups);
        const int c0 = (int)(u % groups) * 32 * kU + lane;
        const int my_row = next_row;
        const float my_w = next_w;
        const size_t base = (size_t)t * C;
        uint4 r[kU], sh[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int c = c0 + q * 32;
            if (c < C) {
                if (kShared) sh[q] = shared[base + c];
                if (residual) r[q] = residual[base + c];
            }
        }
        float acc[kU][8];
        zero(acc);
        for (int j0 = 0; j0 < k; j0 += kKB) {
            uint4 v[kKB][kU];
#pragma unroll
            for (int b = 0; b < kKB; ++b) {
                if (j0 + b < k) {
                    const int row = __shfl_sync(0xffffffffu, my_row, j0 + b);
                    const uint4* src = y + (size_t)row * C;
#pragma unroll
                    for (int q = 0; q < kU; ++q) {
                        const int c = c0 + q * 32;
                        if (c < C) v[b][q] = src[c];
                    }
                }
            }
            if (j0 == 0) {
                // the next unit's indices, while this unit's rows are in flight
                const long long un = u + nwarps;
                if (un < units && lane < k) {
                    const size_t i = (size_t)(un / groups) * k + lane;
                    next_row = clamp_row(pair_row[i], R);
                    next_w = topk_w[i];
                }
            }
#pragma unroll
            for (int b = 0; b < kKB; ++b) {
                if (j0 + b < k) {
                    const float w = __shfl_sync(0xffffffffu, my_w, j0 + b);
#pragma unroll
                    for (int q = 0; q < kU; ++q) {
                        const int c = c0 + q * 32;
                        if (c < C) acc_bf16x8(acc[q], v[b][q], w);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int c = c0 + q * 32;
            if (c < C) {
                if (kShared) add_bf16x8(acc[q], sh[q]);
                if (residual) add_bf16x8(acc[q], r[q]);
                out[base + c] = pack_bf16x8(acc[q]);
            }
        }
    }
}

// Dedup, expert-rank side: partial[d] = bf16(sum over the j of token t carried
// by dedup row d of w[t,j] * y[pair_row[t,j]]), j ascending.
template <int U>
__global__ void __launch_bounds__(kThreads, 3) rank_reduce_kernel(
    const uint4* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ pair_row, const int32_t* __restrict__ pair_dedup_row,
    const int32_t* __restrict__ dedup_row_token, const int32_t* __restrict__ n_dedup_rows, int N,
    int C, int k, int R, uint4* __restrict__ partial) {
    const int lane = threadIdx.x & 31;
    const int d = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    const int Rd = *n_dedup_rows;
    if (d >= Rd) return;
    const int t = clamp_row(dedup_row_token[d], N);
    const int my_row = lane < k ? clamp_row(pair_row[(size_t)t * k + lane], R) : 0;
    const float my_w = lane < k ? topk_w[(size_t)t * k + lane] : 0.f;
    const bool mine = lane < k && pair_dedup_row[(size_t)t * k + lane] == d;
    const uint32_t srcs = __ballot_sync(0xffffffffu, mine);
    for (int c0 = 0; c0 < C; c0 += 32 * U) {
        float acc[U][8];
        zero(acc);
        gather_weighted<U>(acc, y, C, c0, srcs, my_row, my_w);
        finish<U>(acc, nullptr, nullptr, partial, (size_t)d * C, C, c0);
    }
}

// Dedup, owner side: out[t] = bf16(residual[t] + sum of the token's partial
// rows in ascending rank order).
template <int U>
__global__ void __launch_bounds__(kThreads, U == 4 ? 2 : 3) owner_sum_kernel(
    const uint4* __restrict__ partial, const int32_t* __restrict__ pair_dedup_row, int N, int C,
    int k, int Rd_bound, const uint4* shared, const uint4* residual, uint4* out) {
    const int lane = threadIdx.x & 31;
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    if (t >= N) return;
    const int my_d = lane < k ? clamp_row(pair_dedup_row[(size_t)t * k + lane], Rd_bound) : -1;
    // distinct rows of the token; their order among themselves is ascending d,
    // which is ascending rank because dedup rows are stored rank-major
    bool first = lane < k;
    int below = 0;
    for (int jj = 0; jj < k; ++jj) {
        const int o = __shfl_sync(0xffffffffu, my_d, jj);
        if (jj < lane && o == my_d) first = false;
    }
    const uint32_t firsts = __ballot_sync(0xffffffffu, first);
    for (int jj = 0; jj < k; ++jj) {
        const int o = __shfl_sync(0xffffffffu, my_d, jj);
        if (((firsts >> jj) & 1u) && o < my_d) ++below;
    }
    const int nd = __popc(firsts);
    // lane q receives the q-th smallest distinct row
    int sorted_d = 0;
    for (int jj = 0; jj < k; ++jj) {
        const int b = __shfl_sync(0xffffffffu, below, jj);
        const int o = __shfl_sync(0xffffffffu, my_d, jj);
        if (((firsts >> jj) & 1u) && b == lane) sorted_d = o;
    }
    const uint32_t srcs = nd >= 32 ? 0xffffffffu : ((1u << nd) - 1u);
    for (int c0 = 0; c0 < C; c0 += 32 * U) {
        float acc[U][8];
        zero(acc);
        gather_weighted<U>(acc, partial, C, c0, srcs, sorted_d, 1.0f);
        finish<U>(acc, shared, residual, out, (size_t)t * C, C, c0);
    }
}

// Dedup combine in one pass: the two levels of rank_reduce_kernel and
// owner_sum_kernel with the partial rows kept in registers.  For each of the
// token's dedup rows d in ascending order (= ascending rank), the partial is
// the fp32 sum of w[t, j] * y[pair_row[t, j]] over the j carried by d (j
// ascending), rounded to bf16 as the materialised partial would be; the
// partials are summed in fp32 in that order, then the shared row and the
// residual are added.  Bit-identical to the two-kernel form, without writing
// the partials out and reading them back.
//
// The token's k source rows are put in that (d, j) order once; the row loop
// then loads B of them at a time whatever the groups, and a partial is
// rounded and added where its group ends, so the loads of several dedup rows
// are in flight together.  The residual chunk of the next step along the row
// is loaded together with this step's first source rows, so a step waits on
// one round of loads instead of two.
template <int U, int B>
__global__ void __launch_bounds__(kThreads, U == 1 ? 4 : (U == 2 ? 2 : 1)) dedup_combine_kernel(
    const uint4* __restrict__ y, const float* __restrict__ topk_w,
    const int32_t* __restrict__ pair_row, const int32_t* __restrict__ pair_dedup_row, int N,
    int C, int k, int R, int Rd_bound, const uint4* shared, const uint4* residual, uint4* out) {
    const int lane = threadIdx.x & 31;
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    if (t >= N) return;
    const bool live = lane < k;
    const int my_row = live ? clamp_row(pair_row[(size_t)t * k + lane], R) : 0;
    const float my_w = live ? topk_w[(size_t)t * k + lane] : 0.f;
    const int my_d = live ? clamp_row(pair_dedup_row[(size_t)t * k + lane], Rd_bound) : -1;
    // position of lane j in the (d, j) order: rows of smaller d, then the
    // lanes below j with the same d
    int pos = 0;
    for (int jj = 0; jj < k; ++jj) {
        const int o = __shfl_sync(0xffffffffu, my_d, jj);
        if (o < my_d || (o == my_d && jj < lane)) ++pos;
    }
    // lane p takes the row, weight and dedup row at position p
    int src = 0;
    for (int jj = 0; jj < k; ++jj) {
        const int q = __shfl_sync(0xffffffffu, pos, jj);
        if (q == lane) src = jj;
    }
    const int s_row = __shfl_sync(0xffffffffu, my_row, src);
    const float s_w = __shfl_sync(0xffffffffu, my_w, src);
    const int s_d = __shfl_sync(0xffffffffu, my_d, src);
    const int next_d = __shfl_down_sync(0xffffffffu, s_d, 1);
    // bit p: position p is the last row of its dedup row
    const uint32_t ends = __ballot_sync(0xffffffffu, live && (lane == k - 1 || next_d != s_d));
    const size_t base = (size_t)t * C;
    uint4 res_next[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = u * 32 + lane;
        if (residual && c < C) res_next[u] = residual[base + c];
    }
    for (int c0 = 0; c0 < C; c0 += 32 * U) {
        float acc[U][8], part[U][8];
        zero(acc);
        zero(part);
        uint4 res_here[U];
#pragma unroll
        for (int u = 0; u < U; ++u) res_here[u] = res_next[u];
        for (int p0 = 0; p0 < k; p0 += B) {
            uint4 v[B][U];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (p0 + b < k) {
                    const int r = __shfl_sync(0xffffffffu, s_row, p0 + b);
                    const uint4* row = y + (size_t)r * C;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + u * 32 + lane;
                        if (c < C) v[b][u] = row[c];
                    }
                }
            }
            if (p0 == 0) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * U + u * 32 + lane;
                    if (residual && c < C) res_next[u] = residual[base + c];
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int p = p0 + b;
                if (p < k) {
                    const float w = __shfl_sync(0xffffffffu, s_w, p);
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + u * 32 + lane;
                        if (c < C) acc_bf16x8(part[u], v[b][u], w);
                    }
                    if ((ends >> p) & 1u) {
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            add_bf16x8(acc[u], pack_bf16x8(part[u]));
#pragma unroll
                            for (int i = 0; i < 8; ++i) part[u][i] = 0.f;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < C) {
                if (shared) add_bf16x8(acc[u], shared[base + c]);
                if (residual) add_bf16x8(acc[u], res_here[u]);
                out[base + c] = pack_bf16x8(acc[u]);
            }
        }
    }
}

// out = bf16(acc (+ residual)) for the fp32 accumulator of the combine fused
// into the down GEMM; one thread per 8 elements, grid-stride.
__global__ void __launch_bounds__(kThreads) acc_finish_kernel(const float4* __restrict__ acc,
                                                              const uint4* residual, long long n8,
                                                              uint4* out) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8;
         i += (long long)gridDim.x * blockDim.x) {
        const float4 a0 = acc[2 * i], a1 = acc[2 * i + 1];
        float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        if (residual) add_bf16x8(a, residual[i]);
        out[i] = pack_bf16x8(a);
    }
}

inline int warps_grid(long long n) { return (int)((n + kThreads / 32 - 1) / (kThreads / 32)); }

// combine_rows_kernel on a persistent grid of at most kMinBlocks blocks per SM.
template <int kU, int kKB, bool kShared, int kMinBlocks>
cudaError_t rows(const uint4* y, const float* w, const int32_t* pair_row, const moe_shape& s,
                 int C, int R, const uint4* sh, const uint4* res, uint4* o, cudaStream_t st) {
    const int groups = (C + 32 * kU - 1) / (32 * kU);
    const long long units = (long long)s.N * groups;
    long long blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
    const long long cap = (long long)sm_count() * kMinBlocks;
    if (blocks > cap) blocks = cap;
    combine_rows_kernel<kU, kKB, kShared, kMinBlocks><<<(int)blocks, kThreads, 0, st>>>(
        y, w, pair_row, s.N, C, s.k, R, groups, sh, res, o);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_acc_finish(const float* acc, const uint16_t* residual, int N, int H,
                              uint16_t* out, cudaStream_t st) {
    const long long n8 = (long long)N * (H / 8);
    if (n8 == 0) return cudaSuccess;
    long long blocks = (n8 + kThreads - 1) / kThreads;
    const long long cap = (long long)sm_count() * 8;
    acc_finish_kernel<<<(int)(blocks < cap ? blocks : cap), kThreads, 0, st>>>(
        reinterpret_cast<const float4*>(acc), reinterpret_cast<const uint4*>(residual), n8,
        reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* y, const float* w, const moe_layout& L,
                           const moe_shape& s, uint16_t* partial, const uint16_t* shared,
                           const uint16_t* residual, uint16_t* out, cudaStream_t st) {
    if (s.N == 0) return cudaSuccess;
    const int C = s.H / 8;
    const int R = s.N * s.k;
    const uint4* res = reinterpret_cast<const uint4*>(residual);
    const uint4* sh = reinterpret_cast<const uint4*>(shared);
    // chunks per lane per iteration: keep ~8 source loads in flight per lane
    const int kk = s.dedup ? (s.k < s.W ? s.k : s.W) : s.k;
    const int U = kk <= 2 ? 4 : (kk <= 4 ? 2 : 1);
    if (!s.dedup) {
        const uint4* yy = reinterpret_cast<const uint4*>(y);
        uint4* o = reinterpret_cast<uint4*>(out);
        // persistent warps, two 16-byte chunks per lane, source rows two at a
        // time, the next unit's indices prefetched (measured against
        // combine_kernel<4>: 0.86 -> 0.935 of HBM on the DeepSeek-V3 shape,
        // 0.76 -> 0.84 on Mixtral's k = 2, 0.97 -> 1.0 on the skewed shape)
        if (sh) return rows<2, 2, true, 3>(yy, w, L.pair_row, s, C, R, sh, res, o, st);
        // k <= 2: four chunks per lane (a unit is 2 KB of each source row) at
        // two blocks per SM, so a warp keeps as many rows in flight as with
        // larger k (Mixtral's k = 2: 0.052 -> 0.050 ms, 0.78 -> 0.82 of HBM)
        if (s.k <= 2) return rows<4, 2, false, 2>(yy, w, L.pair_row, s, C, R, nullptr, res, o, st);
        return rows<2, 2, false, 4>(yy, w, L.pair_row, s, C, R, nullptr, res, o, st);
    }
    const int Rd_max = s.N * (s.k < s.W ? s.k : s.W);
    const uint4* yy = reinterpret_cast<const uint4*>(y);
    if (!partial) {
        // one pass, partials in registers (bit-identical to the two kernels below)
        uint4* o = reinterpret_cast<uint4*>(out);
        dedup_combine_kernel<kDedupU, kDedupB><<<warps_grid(s.N), kThreads, 0, st>>>(
            yy, w, L.pair_row, L.pair_dedup_row, s.N, C, s.k, R, Rd_max, sh, res, o);
        return cudaGetLastError();
    }
    uint4* pp = reinterpret_cast<uint4*>(partial);
    // a dedup row carries the token's experts on one rank: at most min(k, E/W) rows
    const int per_rank = s.E / s.W;
    const int kr = s.k < per_rank ? s.k : per_rank;
    const int Ur = kr <= 2 ? 4 : (kr <= 4 ? 2 : 1);
    if (Ur == 4)
        rank_reduce_kernel<4><<<warps_grid(Rd_max), kThreads, 0, st>>>(
            yy, w, L.pair_row, L.pair_dedup_row, L.dedup_row_token, L.n_dedup_rows, s.N, C, s.k,
            R, pp);
    else if (Ur == 2)
        rank_reduce_kernel<2><<<warps_grid(Rd_max), kThreads, 0, st>>>(
            yy, w, L.pair_row, L.pair_dedup_row, L.dedup_row_token, L.n_dedup_rows, s.N, C, s.k,
            R, pp);
    else
        rank_reduce_kernel<1><<<warps_grid(Rd_max), kThreads, 0, st>>>(
            yy, w, L.pair_row, L.pair_dedup_row, L.dedup_row_token, L.n_dedup_rows, s.N, C, s.k,
            R, pp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    uint4* o = reinterpret_cast<uint4*>(out);
    const uint4* cp = reinterpret_cast<const uint4*>(partial);
    if (U == 4)
        owner_sum_kernel<4><<<warps_grid(s.N), kThreads, 0, st>>>(
            cp, L.pair_dedup_row, s.N, C, s.k, Rd_max, sh, res, o);
    else if (U == 2)
        owner_sum_kernel<2><<<warps_grid(s.N), kThreads, 0, st>>>(
            cp, L.pair_dedup_row, s.N, C, s.k, Rd_max, sh, res, o);
    else
        owner_sum_kernel<1><<<warps_grid(s.N), kThreads, 0, st>>>(
            cp, L.pair_dedup_row, s.N, C, s.k, Rd_max, sh, res, o);
    return cudaGetLastError();
}

}  // namespace moe
