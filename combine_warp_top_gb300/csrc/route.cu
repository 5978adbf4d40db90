// Router: top-k over fp32 logits, then a softmax over the k selected logits.
//
// "Expert Coupling" (arXiv 2610.09372), Appendix A-A1, Table II: the router is
// an FP32 linear gate whose top-k experts carry the selected probabilities;
// FarSkip-Collective (arXiv 2511.11505) Sec. 2.1: G(A) is a sparse top-k
// selection.  The weights are renormalised over the k selected experts.
//
// One warp per token.  Lane l holds logits l, l+32, l+64, ... (coalesced
// 128-byte loads).  k rounds of a warp arg-max pick the experts in descending
// order; ties go to the lower expert index.  Each round compares order-
// preserving integer keys with the warp-wide redux max / min instructions.
// Lane j keeps the j-th pick, so the k results are written with one coalesced
// store per array.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

// Order-preserving map of a finite float to uint32: a < b as floats iff
// key(a) < key(b).  -0.0 is folded into +0.0 so that the two tie (and the
// lower index wins, as for any tie).  Every key is at least 0x007FFFFF (the
// key of -inf), so 0 marks an empty slot.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// One round of the warp's selection: the largest key over every lane's slots,
// ties to the lowest expert index (slot * 32 + lane); the winning slot is
// emptied.  Lane-local best first (strict '>' over ascending slots keeps the
// lowest index), then one warp max and one warp min (redux) instead of a
// shuffle tree.  Requires at least one non-empty slot in the warp.
template <int VPL>
__device__ __forceinline__ int take_max(uint32_t (&key)[VPL], int lane, uint32_t& won) {
    uint32_t best = 0;
    int bslot = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        if (key[i] > best) {
            best = key[i];
            bslot = i;
        }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, best);
    const uint32_t cand = best == m ? (uint32_t)(bslot * 32 + lane) : 0xffffffffu;
    const uint32_t idx = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(idx & 31u) == lane) {
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i == (int)(idx >> 5)) key[i] = 0;
    }
    won = m;
    return (int)idx;
}

// One compare-exchange of a sorting network: position a ends with the larger
// key, ties to the lower slot (the lower expert index of the lane).
__device__ __forceinline__ void cex(uint32_t& ka, int& sa, uint32_t& kb, int& sb) {
    const bool swap = kb > ka || (kb == ka && sb < sa);
    const uint32_t k0 = swap ? kb : ka, k1 = swap ? ka : kb;
    const int s0 = swap ? sb : sa, s1 = swap ? sa : sb;
    ka = k0;
    kb = k1;
    sa = s0;
    sb = s1;
}

// The lane's VPL (key, slot) pairs in descending key order (Batcher's
// odd-even merge networks for 2, 4 and 8 entries).
template <int VPL>
__device__ __forceinline__ void sort_lane(uint32_t (&key)[VPL], int (&slot)[VPL]) {
    if constexpr (VPL == 2) {
        cex(key[0], slot[0], key[1], slot[1]);
    } else if constexpr (VPL == 4) {
        constexpr int net[5][2] = {{0, 1}, {2, 3}, {0, 2}, {1, 3}, {1, 2}};
#pragma unroll
        for (int c = 0; c < 5; ++c)
            cex(key[net[c][0]], slot[net[c][0]], key[net[c][1]], slot[net[c][1]]);
    } else if constexpr (VPL == 8) {
        constexpr int net[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                                    {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                                    {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
        for (int c = 0; c < 19; ++c)
            cex(key[net[c][0]], slot[net[c][0]], key[net[c][1]], slot[net[c][1]]);
    }
}

// One round over lanes whose slots are sorted (sort_lane): the largest head key
// over the warp, ties to the lowest expert index (slot * 32 + lane); the
// winning lane pops its head.  m receives the key, head this lane's head slot
// before the round (the caller can read a per-slot value of the winner from
// it).  The same picks in the same order as take_max.
template <int VPL>
__device__ __forceinline__ uint32_t take_head(uint32_t (&key)[VPL], int (&slot)[VPL], int lane,
                                              uint32_t& m, int& head) {
    m = __reduce_max_sync(0xffffffffu, key[0]);
    head = slot[0];
    const uint32_t cand = key[0] == m ? (uint32_t)(slot[0] * 32 + lane) : 0xffffffffu;
    const uint32_t idx = __reduce_min_sync(0xffffffffu, cand);
    if ((int)(idx & 31u) == lane) {
#pragma unroll
        for (int i = 0; i + 1 < VPL; ++i) {
            key[i] = key[i + 1];
            slot[i] = slot[i + 1];
        }
        key[VPL - 1] = 0;
    }
    return idx;
}

// kRenorm: weights are a softmax over the k selected logits; otherwise the
// full softmax over all E logits, read at the selected experts.
//
// For E <= 256 (VPL <= 8) each lane first sorts its own slots, so a round
// compares the lanes' heads only and the winner pops its head (take_head),
// a shorter chain per round than take_max's scan of every slot.
template <int VPL, bool kRenorm>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int N, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    if (t >= N) return;
    const float* row = logits + (size_t)t * E;

    float v[VPL];
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? __ldg(row + e) : 0.f;
        key[i] = e < E ? order_key(v[i]) : 0u;
    }

    // k <= E: every round finds a non-empty slot
    int my_id = -1;
    float my_val = 0.f;
    if constexpr (VPL <= 8) {
        int slot[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) slot[i] = i;
        sort_lane<VPL>(key, slot);
        for (int j = 0; j < k; ++j) {
            uint32_t m;
            int head;
            const uint32_t idx = take_head<VPL>(key, slot, lane, m, head);
            if (lane == j) {
                my_id = (int)idx;
                my_val = key_value(m);
            }
        }
    } else {
        for (int j = 0; j < k; ++j) {
            uint32_t m;
            const int idx = take_max<VPL>(key, lane, m);
            if (lane == j) {
                my_id = idx;
                my_val = key_value(m);
            }
        }
    }

    // softmax; the first pick holds the maximum of all E logits
    const float m = __shfl_sync(0xffffffffu, my_val, 0);
    const float z = lane < k ? expf(my_val - m) : 0.f;
    float s = z;
    if (!kRenorm) {
        s = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i * 32 + lane < E) s += expf(v[i] - m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = z / s;
    }
}

// Sigmoid router with a per-expert selection bias (the auxiliary-loss-free
// router of "Expert Coupling" Appendix A-B): score s_e = sigmoid(L_e),
// evaluated in double and rounded once to fp32; the k largest s_e + bias_e
// (fp32 add; ties to the lower expert index) are selected; the weights are
// s_e / sum of the selected s_e (the bias only steers the selection).
template <int VPL>
__global__ void __launch_bounds__(256) route_sigmoid_kernel(const float* __restrict__ logits,
                                                            const float* __restrict__ bias, int N,
                                                            int E, int k,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
    if (t >= N) return;
    const float* row = logits + (size_t)t * E;
    float sc[VPL];
    uint32_t key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        if (e < E) {
            const double L = (double)__ldg(row + e);
            sc[i] = (float)(1.0 / (1.0 + exp(-L)));
            key[i] = order_key(sc[i] + __ldg(bias + e));
        } else {
            sc[i] = 0.f;
            key[i] = 0u;
        }
    }
    int my_id = -1;
    float my_s = 0.f;
    if constexpr (VPL <= 8) {
        // as in route_kernel: each lane sorts its slots once, rounds compare heads
        int slot[VPL];
#pragma unroll
        for (int i = 0; i < VPL; ++i) slot[i] = i;
        sort_lane<VPL>(key, slot);
        for (int j = 0; j < k; ++j) {
            uint32_t m;
            int head;
            const uint32_t idx = take_head<VPL>(key, slot, lane, m, head);
            // the winner's score, from the lane that holds it (its head slot)
            float s_head = 0.f;
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == head) s_head = sc[i];
            const float bs = __shfl_sync(0xffffffffu, s_head, (int)(idx & 31u));
            if (lane == j) {
                my_id = (int)idx;
                my_s = bs;
            }
        }
    } else {
        for (int j = 0; j < k; ++j) {
            uint32_t m;
            const int idx = take_max<VPL>(key, lane, m);
            // the winner's score, from the lane that holds it
            float s_slot = 0.f;
#pragma unroll
            for (int i = 0; i < VPL; ++i)
                if (i == (idx >> 5)) s_slot = sc[i];
            const float bs = __shfl_sync(0xffffffffu, s_slot, idx & 31);
            if (lane == j) {
                my_id = idx;
                my_s = bs;
            }
        }
    }
    float sum = lane < k ? my_s : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = my_s / sum;
    }
}

template <int VPL>
cudaError_t go_sigmoid(const float* logits, const float* bias, int N, int E, int k, int32_t* ids,
                       float* w, cudaStream_t st) {
    const int blocks = (N + 7) / 8;
    route_sigmoid_kernel<VPL><<<blocks, 256, 0, st>>>(logits, bias, N, E, k, ids, w);
    return cudaGetLastError();
}

template <int VPL>
cudaError_t go(const float* logits, int N, int E, int k, int32_t* ids, float* w, bool renorm,
               cudaStream_t st) {
    const int threads = 256;
    const int tokens_per_block = threads / 32;
    const int blocks = (N + tokens_per_block - 1) / tokens_per_block;
    if (renorm)
        route_kernel<VPL, true><<<blocks, threads, 0, st>>>(logits, N, E, k, ids, w);
    else
        route_kernel<VPL, false><<<blocks, threads, 0, st>>>(logits, N, E, k, ids, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const float* logits, int N, int E, int k, int32_t* ids, float* w,
                         bool renorm, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    if (E <= 32) return go<1>(logits, N, E, k, ids, w, renorm, st);
    if (E <= 64) return go<2>(logits, N, E, k, ids, w, renorm, st);
    if (E <= 128) return go<4>(logits, N, E, k, ids, w, renorm, st);
    if (E <= 256) return go<8>(logits, N, E, k, ids, w, renorm, st);
    if (E <= 512) return go<16>(logits, N, E, k, ids, w, renorm, st);
    return go<32>(logits, N, E, k, ids, w, renorm, st);
}

cudaError_t launch_route_sigmoid(const float* logits, const float* bias, int N, int E, int k,
                                 int32_t* ids, float* w, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    if (E <= 32) return go_sigmoid<1>(logits, bias, N, E, k, ids, w, st);
    if (E <= 64) return go_sigmoid<2>(logits, bias, N, E, k, ids, w, st);
    if (E <= 128) return go_sigmoid<4>(logits, bias, N, E, k, ids, w, st);
    if (E <= 256) return go_sigmoid<8>(logits, bias, N, E, k, ids, w, st);
    if (E <= 512) return go_sigmoid<16>(logits, bias, N, E, k, ids, w, st);
    return go_sigmoid<32>(logits, bias, N, E, k, ids, w, st);
}

}  // namespace moe
