// Dispatch layout: a stable counting sort of the (token, expert) pairs by the
// placement slot of the expert, plus the deduplicated (token, rank) rows.
//
// "Kernel fusion for expert parallelism", section "Expert parallelism:
// dispatch and combine" (W ranks of E/W experts; receivers must know their
// per-sender counts) and "Expert Coupling" (arXiv 2610.09372) Sec. V-A (one row
// per unique (token, destination rank); a placement is a permutation of global
// expert IDs) and Appendix A-A2 (the receiver expands rows to expert-major
// order).
//
// Two launches (three when the count tables exceed kScanTableBytes, one when
// all tokens fit one block of 256), all deterministic:
//  1. count:   per block of 256 tokens, one 32-bit mask per (warp, slot) and
//              per (warp, rank) records which lanes (tokens) hit it; the block
//              count of a key is the sum of the popcounts.  OR-ing the rank
//              bits merges a token's experts on one rank for free, which is the
//              deduplication.
//  2. scatter: each block rebuilds its masks and derives its own bases: it
//              copies the whole per-block count table into shared memory, sums
//              every column (the slot and rank totals, scanned into the slot
//              and rank offsets) and the part of it above its own row (the
//              blocks before it in token order).  Block 0 also writes the
//              layout's count and offset tables.  A pair's row is its warp's
//              base plus the popcount of the lower lanes' bits, so tokens
//              ascend inside every segment exactly as in a stable sort.
//     With larger tables a one-block scan launch between the two turns the
//     table into bases once, and the scatter blocks read theirs.  With one
//     block (N <= 256) the scatter block's own masks are the whole table, so
//     it counts them itself and the count launch is skipped.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 32 * kLayoutWarps;
// Largest per-block count table ([nb][E] + [nb][W] int32) that every scatter
// block scans for itself in its shared memory.  Measured against the separate
// scan launch: 2 to 4.5 us faster at 32 bytes to 64 KB (1 to 128 count blocks,
// the tables copied by cp.async while the masks are built, tall columns summed
// in parts).
constexpr size_t kScanTableBytes = 64 * 1024;

// slot_of[e] = the placement slot holding expert e.  Invalid placements are
// reported and resolved deterministically (lowest slot wins, unplaced experts
// fall back to slot 0) so that every block derives the same table.
__device__ void build_slot_of(int* slot_of, const int32_t* placement, int E, int* err) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) slot_of[e] = 0x7fffffff;
    __syncthreads();
    for (int p = threadIdx.x; p < E; p += blockDim.x) {
        const int e = placement ? placement[p] : p;
        if (e < 0 || e >= E) {
            set_error(err, MOE_ERR_INVALID_ARG);
            continue;
        }
        const int old = atomicMin(&slot_of[e], p);
        if (old != 0x7fffffff) set_error(err, MOE_ERR_INVALID_ARG);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        if (slot_of[e] == 0x7fffffff) {
            set_error(err, MOE_ERR_INVALID_ARG);
            slot_of[e] = 0;
        }
    }
    __syncthreads();
}

struct Smem {
    int* slot_of;     // [E]
    uint32_t* mask;   // [kLayoutWarps][E]
    uint32_t* rmask;  // [kLayoutWarps][W]
    int* base;        // [kLayoutWarps][E]
    int* rbase;       // [kLayoutWarps][W]
};

// Word offset of the scatter kernel's copy of the count tables in its dynamic
// shared memory: after the Smem arrays, rounded up to 16 bytes.
__host__ __device__ inline size_t table_offset_words(int E, int W) {
    return ((size_t)E + 2 * (size_t)kLayoutWarps * (E + W) + 3) & ~(size_t)3;
}
// Words that a [nb][ncol] table takes there: it is copied in whole 16-byte
// pieces, so nb * ncol rounded up to 4.  The [nb][E] slot table comes first,
// the [nb][W] rank table right after it.
__host__ __device__ inline size_t padded_table_words(int nb, int ncol) {
    return ((size_t)nb * ncol + 3) & ~(size_t)3;
}

__device__ Smem carve(uint32_t* sm, int E, int W) {
    Smem s;
    s.slot_of = reinterpret_cast<int*>(sm);
    s.mask = sm + E;
    s.rmask = s.mask + kLayoutWarps * E;
    s.base = reinterpret_cast<int*>(s.rmask + kLayoutWarps * W);
    s.rbase = s.base + kLayoutWarps * E;
    return s;
}

// This thread's token's k expert ids, all loads issued at once (one memory
// round trip instead of k); entries j >= k and tokens past N are 0.
__device__ __forceinline__ void load_token_ids(int (&ids_t)[kMaxK],
                                               const int32_t* __restrict__ ids, int N, int k) {
    const int t = blockIdx.x * kLayoutTokens + threadIdx.x;
    const int32_t* row = ids + (size_t)t * k;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) ids_t[j] = (t < N && j < k) ? __ldg(row + j) : 0;
}

// Fill this block's lane masks from the token ids in ids_t.  Masks are valid
// after the trailing __syncthreads.
__device__ void build_masks(const Smem& s, const int (&ids_t)[kMaxK], int N, int E, int k, int W,
                            int dedup, int* err) {
    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s.mask[i] = 0;
    if (dedup)
        for (int i = threadIdx.x; i < kLayoutWarps * W; i += blockDim.x) s.rmask[i] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kLayoutTokens + threadIdx.x;
    const int per_rank = E / W;
    if (t < N) {
        const uint32_t bit = 1u << lane;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (j >= k) break;
            int e = ids_t[j];
            if (e < 0 || e >= E) {
                set_error(err, MOE_ERR_INVALID_ARG);
                e = 0;
            }
            const int p = s.slot_of[e];
            const uint32_t old = atomicOr(&s.mask[warp * E + p], bit);
            if (old & bit) set_error(err, MOE_ERR_INVALID_ARG);  // expert repeated in a token
            if (dedup) atomicOr(&s.rmask[warp * W + p / per_rank], bit);
        }
    }
    __syncthreads();
}

// Exclusive scan of one value per thread over a block of up to 1024 threads.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        int ws = lane < nw ? warp_sums[lane] : 0;
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) warp_sums[lane] = wi - ws;  // exclusive prefix of the warps
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int r = warp_sums[warp] + incl - v;
    __syncthreads();
    return r;
}

// Exclusive scan of n values by the whole block: each thread takes a run of
// consecutive values.  out[i] = sum of in[0..i); *total = the sum.
__device__ void block_scan_values(const int* in, int n, int* out, int* warp_sums, int* total) {
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = threadIdx.x * per, i1 = min(n, i0 + per);
    int sum = 0;
    for (int i = i0; i < i1; ++i) sum += in[i];
    int run = block_exclusive_scan(sum, warp_sums, total);
    for (int i = i0; i < i1; ++i) {
        const int v = in[i];
        out[i] = run;
        run += v;
    }
    __syncthreads();
}

// Exclusive scan down every column of a [nb][ncol] table in global memory, in
// place, by the whole block (ncol <= blockDim): the rows of a column are split
// into P = blockDim / ncol parts; each thread sums its part (independent
// loads), the parts of a column are scanned through part_sums, and each
// thread rewrites its rows with the running prefix.  totals[c] receives the
// column sum.  part_sums holds blockDim ints.
__device__ void columns_scan(int32_t* __restrict__ tab, int nb, int ncol, int* part_sums,
                             int* totals) {
    const int P = blockDim.x / ncol;
    const int c = threadIdx.x % ncol, part = threadIdx.x / ncol;
    const int L = (nb + P - 1) / P;
    const int b0 = part * L, b1 = min(nb, b0 + L);
    int sum = 0;
    if (part < P)
        for (int b = b0; b < b1; ++b) sum += tab[(size_t)b * ncol + c];
    if (part < P) part_sums[part * ncol + c] = sum;
    __syncthreads();
    if (threadIdx.x < ncol) {
        int run = 0;
        for (int q = 0; q < P; ++q) {
            const int v = part_sums[q * ncol + threadIdx.x];
            part_sums[q * ncol + threadIdx.x] = run;
            run += v;
        }
        totals[threadIdx.x] = run;
    }
    __syncthreads();
    if (part < P) {
        int run = part_sums[part * ncol + c];
        for (int b = b0; b < b1; ++b) {
            const int v = tab[(size_t)b * ncol + c];
            tab[(size_t)b * ncol + c] = run;
            run += v;
        }
    }
    __syncthreads();
}

// Scratch of the scan, in the block's shared memory.
struct ScanSmem {
    int part_sums[1024];
    int totals[kMaxE];
    int starts[kMaxE];
    int warp_sums[32];
    int total;
};

// The scan proper: per-block counts -> exclusive bases in place; column totals
// -> slot and rank offsets, the layout's counts and offsets, and (dedup) the
// dedup row counts and offsets.  tab / rtab: [nb][E] / [nb][W] tables in
// global memory; every thread of a block of at least E threads calls it.
__device__ void scan_counts(const int32_t* __restrict__ placement, int nb, int E, int W,
                            int dedup, int32_t* tab, int32_t* rtab,
                            int32_t* __restrict__ slot_start, const moe_layout& L, ScanSmem& ss) {
    columns_scan(tab, nb, E, ss.part_sums, ss.totals);
    block_scan_values(ss.totals, E, ss.starts, ss.warp_sums, &ss.total);
    const int R = ss.total;
    const int per_rank = E / W;
    for (int p = threadIdx.x; p < E; p += blockDim.x) {
        const int start = ss.starts[p];
        slot_start[p] = start;
        int e = placement ? placement[p] : p;
        if (e < 0 || e >= E) e = 0;  // reported by the count kernel
        L.expert_counts[e] = ss.totals[p];
        L.expert_offsets[e] = start;
        if (p % per_rank == 0) L.rank_offsets[p / per_rank] = start;
    }
    if (threadIdx.x == 0) {
        slot_start[E] = R;
        L.expert_offsets[E] = R;
        L.rank_offsets[W] = R;
    }
    __syncthreads();
    if (!dedup) return;
    columns_scan(rtab, nb, W, ss.part_sums, ss.totals);
    block_scan_values(ss.totals, W, ss.starts, ss.warp_sums, &ss.total);
    for (int r = threadIdx.x; r < W; r += blockDim.x) {
        L.dedup_counts[r] = ss.totals[r];
        L.dedup_offsets[r] = ss.starts[r];
    }
    if (threadIdx.x == 0) {
        L.dedup_offsets[W] = ss.total;
        *L.n_dedup_rows = ss.total;
    }
}

// The scan as its own one-block launch, on the tables in global memory (for
// tables larger than kScanSmemBytes).
__global__ void __launch_bounds__(1024) layout_scan_kernel(
    const int32_t* __restrict__ placement, int nb, int E, int W, int dedup,
    int32_t* __restrict__ blk_counts, int32_t* __restrict__ blk_rcounts,
    int32_t* __restrict__ slot_start, moe_layout L) {
    __shared__ ScanSmem ss;
    scan_counts(placement, nb, E, W, dedup, blk_counts, blk_rcounts, slot_start, L, ss);
}

__global__ void __launch_bounds__(kThreads) layout_count_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ placement, int N, int E, int k,
    int W, int dedup, int32_t* __restrict__ blk_counts, int32_t* __restrict__ blk_rcounts,
    int* err) {
    extern __shared__ uint32_t sm[];
    const Smem s = carve(sm, E, W);
    int ids_t[kMaxK];
    load_token_ids(ids_t, ids, N, k);
    build_slot_of(s.slot_of, placement, E, err);
    build_masks(s, ids_t, N, E, k, W, dedup, err);
    for (int p = threadIdx.x; p < E; p += blockDim.x) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) c += __popc(s.mask[w * E + p]);
        blk_counts[(size_t)blockIdx.x * E + p] = c;
    }
    if (dedup) {
        for (int r = threadIdx.x; r < W; r += blockDim.x) {
            int c = 0;
#pragma unroll
            for (int w = 0; w < kLayoutWarps; ++w) c += __popc(s.rmask[w * W + r]);
            blk_rcounts[(size_t)blockIdx.x * W + r] = c;
        }
    }
}

// Scatter-side scan of one [nb][ncol] count table held in shared memory:
// col_base[c] = first row of this block's part of column c (the column
// offset plus the counts of the blocks before this one); totals[c] and
// starts[c] = the column sums and their exclusive scan.  Tall tables split
// the rows of a column into P parts of at least 8 rows, summed by different
// threads (P <= blockDim / ncol; the part sums wait in ss.starts until the
// scan overwrites it); otherwise a thread walks a whole column.
__device__ void block_bases(const int32_t* tab, int nb, int ncol, int* col_base, ScanSmem& ss) {
    const int P = min((int)blockDim.x / ncol, nb / 8);
    if (P > 1) {
        const int c = threadIdx.x % ncol, part = threadIdx.x / ncol;
        const int L = (nb + P - 1) / P, b0 = part * L, b1 = min(nb, b0 + L);
        int* psum = ss.starts;                // [P][ncol]
        int* pbefore = ss.starts + P * ncol;  // [P][ncol]
        if (part < P) {
            int tot = 0, before = 0;
            for (int b = b0; b < b1; ++b) {
                const int v = tab[(size_t)b * ncol + c];
                if (b < (int)blockIdx.x) before += v;
                tot += v;
            }
            psum[part * ncol + c] = tot;
            pbefore[part * ncol + c] = before;
        }
        __syncthreads();
        if (threadIdx.x < ncol) {
            int tot = 0, before = 0;
            for (int q = 0; q < P; ++q) {
                tot += psum[q * ncol + threadIdx.x];
                before += pbefore[q * ncol + threadIdx.x];
            }
            ss.totals[threadIdx.x] = tot;
            col_base[threadIdx.x] = before;
        }
    } else {
        for (int c = threadIdx.x; c < ncol; c += blockDim.x) {
            int tot = 0, before = 0;
            for (int b = 0; b < nb; ++b) {
                const int v = tab[(size_t)b * ncol + c];
                if (b < (int)blockIdx.x) before += v;
                tot += v;
            }
            ss.totals[c] = tot;
            col_base[c] = before;
        }
    }
    __syncthreads();
    block_scan_values(ss.totals, ncol, ss.starts, ss.warp_sums, &ss.total);
    for (int c = threadIdx.x; c < ncol; c += blockDim.x) col_base[c] += ss.starts[c];
    __syncthreads();
}

// scan_here: derive this block's bases from the whole count table (copied
// into shared memory after the masks) instead of reading the bases that a
// separate scan launch wrote.  self_count (a grid of one block, with
// scan_here): the table is this block's own mask popcounts, no count launch
// ran, and the invalid ids / placement it would have reported are reported
// here (err).
__global__ void __launch_bounds__(kThreads) layout_scatter_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ placement, int N, int E, int k,
    int W, int dedup, const int32_t* __restrict__ blk_counts,
    const int32_t* __restrict__ blk_rcounts, const int32_t* __restrict__ slot_start, moe_layout L,
    int scan_here, int self_count, int* err) {
    extern __shared__ uint32_t sm[];
    __shared__ ScanSmem ss;
    const Smem s = carve(sm, E, W);
    // every global load of the prologue in flight at once: the token ids (to
    // registers) and, with scan_here, the count tables (16-byte asynchronous
    // copies to shared memory, waited for after the masks are built)
    int ids_t[kMaxK];
    load_token_ids(ids_t, ids, N, k);
    const int nb = gridDim.x;
    int32_t* tab = reinterpret_cast<int32_t*>(sm + table_offset_words(E, W));  // [nb][E]
    int32_t* rtab = tab + padded_table_words(nb, E);                            // [nb][W]
    if (scan_here && !self_count) {
        const int nE = nb * E, nW = dedup ? nb * W : 0;
        const uint32_t t0 = ptx::smem_u32(tab), r0 = ptx::smem_u32(rtab);
        for (int i = threadIdx.x; 4 * i < nE; i += blockDim.x)
            ptx::cp_async_16(t0 + 16u * i, blk_counts + 4 * i, 4u * min(4, nE - 4 * i));
        for (int i = threadIdx.x; 4 * i < nW; i += blockDim.x)
            ptx::cp_async_16(r0 + 16u * i, blk_rcounts + 4 * i, 4u * min(4, nW - 4 * i));
    }
    // errors were reported by the count pass, unless there was none
    int* const perr = self_count ? err : nullptr;
    build_slot_of(s.slot_of, placement, E, perr);
    build_masks(s, ids_t, N, E, k, W, dedup, perr);
    int* col_base = ss.part_sums;  // first row of this block's part of each slot / rank
    const int per_rank = E / W;
    if (scan_here) {
        if (self_count) {
            // the only block: its mask popcounts are the count table
            for (int p = threadIdx.x; p < E; p += blockDim.x) {
                int c = 0;
#pragma unroll
                for (int w = 0; w < kLayoutWarps; ++w) c += __popc(s.mask[w * E + p]);
                tab[p] = c;
            }
            if (dedup) {
                for (int r = threadIdx.x; r < W; r += blockDim.x) {
                    int c = 0;
#pragma unroll
                    for (int w = 0; w < kLayoutWarps; ++w) c += __popc(s.rmask[w * W + r]);
                    rtab[r] = c;
                }
            }
        } else {
            ptx::cp_async_wait_all();
        }
        __syncthreads();
        block_bases(tab, nb, E, col_base, ss);
        if (blockIdx.x == 0) {
            for (int p = threadIdx.x; p < E; p += blockDim.x) {
                int e = placement ? placement[p] : p;
                if (e < 0 || e >= E) e = 0;  // reported by the count kernel
                L.expert_counts[e] = ss.totals[p];
                L.expert_offsets[e] = ss.starts[p];
                if (p % per_rank == 0) L.rank_offsets[p / per_rank] = ss.starts[p];
            }
            if (threadIdx.x == 0) {
                L.expert_offsets[E] = ss.total;
                L.rank_offsets[W] = ss.total;
            }
        }
    } else {
        for (int p = threadIdx.x; p < E; p += blockDim.x)
            col_base[p] = slot_start[p] + blk_counts[(size_t)blockIdx.x * E + p];
        __syncthreads();
    }
    for (int p = threadIdx.x; p < E; p += blockDim.x) {
        int run = col_base[p];
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            s.base[w * E + p] = run;
            run += __popc(s.mask[w * E + p]);
        }
    }
    __syncthreads();
    if (dedup) {
        if (scan_here) {
            block_bases(rtab, nb, W, col_base, ss);
            if (blockIdx.x == 0) {
                for (int r = threadIdx.x; r < W; r += blockDim.x) {
                    L.dedup_counts[r] = ss.totals[r];
                    L.dedup_offsets[r] = ss.starts[r];
                }
                if (threadIdx.x == 0) {
                    L.dedup_offsets[W] = ss.total;
                    *L.n_dedup_rows = ss.total;
                }
            }
        } else {
            for (int r = threadIdx.x; r < W; r += blockDim.x)
                col_base[r] = L.dedup_offsets[r] + blk_rcounts[(size_t)blockIdx.x * W + r];
            __syncthreads();
        }
        for (int r = threadIdx.x; r < W; r += blockDim.x) {
            int run = col_base[r];
#pragma unroll
            for (int w = 0; w < kLayoutWarps; ++w) {
                s.rbase[w * W + r] = run;
                run += __popc(s.rmask[w * W + r]);
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kLayoutTokens + threadIdx.x;
    if (t >= N) return;
    const uint32_t lower = (1u << lane) - 1u;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j >= k) break;
        int e = ids_t[j];
        if (e < 0 || e >= E) e = 0;
        const int p = s.slot_of[e];
        const int row = s.base[warp * E + p] + __popc(s.mask[warp * E + p] & lower);
        L.row_token[row] = t;
        L.pair_row[(size_t)t * k + j] = row;
        if (dedup) {
            const int r = p / per_rank;
            const int d = s.rbase[warp * W + r] + __popc(s.rmask[warp * W + r] & lower);
            L.pair_dedup_row[(size_t)t * k + j] = d;
            L.dedup_row_token[d] = t;
            L.expand_src[row] = d;
        }
    }
}

inline size_t smem_bytes(int E, int W) {
    return sizeof(uint32_t) * ((size_t)E + 2 * (size_t)kLayoutWarps * (E + W));
}

}  // namespace

cudaError_t launch_layout(const int32_t* ids, const int32_t* placement, const moe_shape& s,
                          const moe_layout& L, void* ws, cudaStream_t st) {
    const Workspace wl = workspace_layout(s);
    int* err = ws_ptr<int>(ws, wl.err);
    int32_t* blk_counts = ws_ptr<int32_t>(ws, wl.blk_counts);
    int32_t* blk_rcounts = ws_ptr<int32_t>(ws, wl.blk_rcounts);
    int32_t* slot_start = ws_ptr<int32_t>(ws, wl.slot_start);
    const int nb = layout_blocks(s.N);
    const size_t smem = smem_bytes(s.E, s.W);
    // the scatter blocks scan the count tables themselves when they are small
    // (they copy them in 16-byte pieces, so a workspace that does not start on
    // 16 bytes takes the separate scan instead)
    const size_t table = sizeof(int32_t) * (padded_table_words(nb, s.E) +
                                            (s.dedup ? padded_table_words(nb, s.W) : 0));
    const bool aligned = ((reinterpret_cast<uintptr_t>(blk_counts) |
                           reinterpret_cast<uintptr_t>(blk_rcounts)) & 15u) == 0;
    const bool scan_here = nb > 0 && table <= kScanTableBytes && aligned;
    // one block: it counts its own masks (no count launch)
    const bool self_count = scan_here && nb == 1;
    const size_t scatter_smem =
        scan_here ? sizeof(int32_t) * table_offset_words(s.E, s.W) + table : smem;
    cudaError_t e;
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
    }
    if (scatter_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(layout_scatter_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scatter_smem);
        if (e != cudaSuccess) return e;
    }
    if (nb > 0 && !self_count) {
        layout_count_kernel<<<nb, kThreads, smem, st>>>(ids, placement, s.N, s.E, s.k, s.W,
                                                        s.dedup, blk_counts, blk_rcounts, err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (!scan_here) {
        layout_scan_kernel<<<1, 1024, 0, st>>>(placement, nb, s.E, s.W, s.dedup, blk_counts,
                                                blk_rcounts, slot_start, L);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (nb > 0) {
        layout_scatter_kernel<<<nb, kThreads, scatter_smem, st>>>(
            ids, placement, s.N, s.E, s.k, s.W, s.dedup, blk_counts, blk_rcounts, slot_start, L,
            scan_here ? 1 : 0, self_count ? 1 : 0, err);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
