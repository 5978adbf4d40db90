// Correlated expert placement ("Expert Coupling", arXiv 2610.09372, Sec. V-A
// and Appendix A-D, Algorithm 1).
//
// moe_coselection (device): W[e, e'] = number of tokens whose selected experts
// include both e and e'.  One thread per token adds its k*k (e_j, e_j') pairs
// (diagonal included) with integer atomics, so the counts do not depend on the
// order of the additions.  When E*E counts fit in shared memory, each block
// first accumulates its tokens there and then adds its non-zero counts to the
// global matrix.
//
// moe_placement_search (host, C++): the balanced partition of Algorithm 1.
// Start from contiguous groups of E/G experts and repeatedly apply the swap of
// two experts of different groups with the largest gain in within-group
// co-selection (ties: the pair (a, b), a < b, first in lexicographic order)
// until no swap gains or the swap budget is spent.  On several nodes the
// experts are first partitioned across nodes, then each node's experts
// (ascending ids) across its ranks.  The result is written as a placement
// permutation: slot p holds expert placement[p]; rank r owns slots
// [r*E/P, (r+1)*E/P), its experts in ascending id order.
#include <stdint.h>

#include <vector>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kSmemCounts = 16384;  // E*E counts that fit in 64 KB of shared memory

__global__ void __launch_bounds__(kThreads) coselect_smem_kernel(const int32_t* __restrict__ ids,
                                                                 int N, int k, int E,
                                                                 int32_t* __restrict__ W,
                                                                 int* err) {
    extern __shared__ int32_t cnt[];
    const int EE = E * E;
    for (int i = threadIdx.x; i < EE; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < N; t += gridDim.x * blockDim.x) {
        int e[kMaxK];
        for (int j = 0; j < k; ++j) {
            int v = ids[(size_t)t * k + j];
            if (v < 0 || v >= E) {
                set_error(err, MOE_ERR_INVALID_ARG);
                v = 0;
            }
            e[j] = v;
        }
        for (int j = 0; j < k; ++j)
            for (int j2 = 0; j2 < k; ++j2) atomicAdd(&cnt[e[j] * E + e[j2]], 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < EE; i += blockDim.x)
        if (cnt[i]) atomicAdd(&W[i], cnt[i]);
}

__global__ void __launch_bounds__(kThreads) coselect_global_kernel(
    const int32_t* __restrict__ ids, int N, int k, int E, int32_t* __restrict__ W, int* err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= N) return;
    int e[kMaxK];
    for (int j = 0; j < k; ++j) {
        int v = ids[(size_t)t * k + j];
        if (v < 0 || v >= E) {
            set_error(err, MOE_ERR_INVALID_ARG);
            v = 0;
        }
        e[j] = v;
    }
    for (int j = 0; j < k; ++j)
        for (int j2 = 0; j2 < k; ++j2) atomicAdd(&W[(size_t)e[j] * E + e[j2]], 1);
}

// ---- host search --------------------------------------------------------------------

// Balanced best-swap partition of the experts `members` (indices into W, an
// E_full x E_full row-major matrix) into G groups; returns each member's group.
std::vector<int> partition(const int32_t* W, int E_full, const std::vector<int>& members, int G,
                           long long max_swaps, long long* swaps_made) {
    const int n = (int)members.size();
    const int size = n / G;
    std::vector<int> group(n);
    for (int i = 0; i < n; ++i) group[i] = i / size;
    auto w = [&](int i, int j) -> long long {
        return W[(size_t)members[i] * E_full + members[j]];
    };
    // conn[i*G + g] = sum over members x != i of group g of W[i, x]
    std::vector<long long> conn((size_t)n * G);
    auto rebuild = [&]() {
        std::fill(conn.begin(), conn.end(), 0LL);
        for (int i = 0; i < n; ++i)
            for (int x = 0; x < n; ++x)
                if (x != i) conn[(size_t)i * G + group[x]] += w(i, x);
    };
    rebuild();
    long long swaps = 0;
    for (long long it = 0; it < max_swaps; ++it) {
        long long best = 0;
        int ba = -1, bb = -1;
        for (int a = 0; a < n; ++a) {
            const int A = group[a];
            const long long* ca = &conn[(size_t)a * G];
            for (int b = a + 1; b < n; ++b) {
                const int B = group[b];
                if (A == B) continue;
                const long long* cb = &conn[(size_t)b * G];
                const long long gain = ca[B] - ca[A] + cb[A] - cb[B] - 2 * w(a, b);
                if (gain > best) {
                    best = gain;
                    ba = a;
                    bb = b;
                }
            }
        }
        if (ba < 0) break;
        // move ba to group B and bb to group A; update every row's two sums
        const int A = group[ba], B = group[bb];
        for (int i = 0; i < n; ++i) {
            long long* ci = &conn[(size_t)i * G];
            const long long wa = (i == ba) ? 0 : w(i, ba);
            const long long wb = (i == bb) ? 0 : w(i, bb);
            ci[A] += wb - wa;
            ci[B] += wa - wb;
        }
        group[ba] = B;
        group[bb] = A;
        ++swaps;
    }
    if (swaps_made) *swaps_made += swaps;
    return group;
}

}  // namespace

cudaError_t launch_coselection(const int32_t* ids, const moe_shape& s, int32_t* W, int* err,
                               cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(W, 0, sizeof(int32_t) * (size_t)s.E * s.E, st);
    if (e != cudaSuccess || s.N == 0) return e;
    if (s.E * s.E <= kSmemCounts) {
        const size_t smem = sizeof(int32_t) * (size_t)s.E * s.E;
        if (smem > 48 * 1024) {
            e = cudaFuncSetAttribute(coselect_smem_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        int blocks = (s.N + kThreads - 1) / kThreads;
        const int cap = 2 * sm_count();
        if (blocks > cap) blocks = cap;
        coselect_smem_kernel<<<blocks, kThreads, smem, st>>>(ids, s.N, s.k, s.E, W, err);
    } else {
        coselect_global_kernel<<<(s.N + kThreads - 1) / kThreads, kThreads, 0, st>>>(
            ids, s.N, s.k, s.E, W, err);
    }
    return cudaGetLastError();
}

moe_status placement_search(const int32_t* W, int E, int ranks, int nodes, long long max_swaps,
                            int32_t* placement, long long* swaps_made) {
    std::vector<int> rank_of(E);
    long long swaps = 0;
    std::vector<int> all(E);
    for (int e = 0; e < E; ++e) all[e] = e;
    if (nodes == 1) {
        std::vector<int> g = partition(W, E, all, ranks, max_swaps, &swaps);
        for (int e = 0; e < E; ++e) rank_of[e] = g[e];
    } else {
        std::vector<int> node = partition(W, E, all, nodes, max_swaps, &swaps);
        const int per = ranks / nodes;
        for (int n = 0; n < nodes; ++n) {
            std::vector<int> members;
            for (int e = 0; e < E; ++e)
                if (node[e] == n) members.push_back(e);
            std::vector<int> rho = partition(W, E, members, per, max_swaps, &swaps);
            for (size_t i = 0; i < members.size(); ++i) rank_of[members[i]] = n * per + rho[i];
        }
    }
    int p = 0;
    for (int r = 0; r < ranks; ++r)
        for (int e = 0; e < E; ++e)
            if (rank_of[e] == r) placement[p++] = e;
    if (swaps_made) *swaps_made = swaps;
    return p == E ? MOE_OK : MOE_ERR_DEVICE_ASSERT;
}

}  // namespace moe
