// Grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2): the same
// computation as grouped_gemm.cu -- gate/up with the SwiGLU epilogue, and down
// -- on 256-row tiles that two CTAs of a cluster share.
//
// FarSkip-Collective (arXiv 2511.11505) Sec. 2.1 and "Kernel fusion for expert
// parallelism", section "Fusing the layer into one kernel", stages 4-6.
//
// Why pairs: one 128x256 tile per CTA makes the tensor core read 48 KB of
// operands from shared memory per 64-deep k-block while TMA writes the next
// 48 KB; with a pair, each CTA holds its 128 rows of A and half of B (N/2 =
// 128 rows), so 32 KB per CTA and k-block feed a 256x256 MMA.  That halves
// the B traffic per flop and leaves room for six pipeline stages.
//
// Roles per CTA (224 threads): warp 0 loads this CTA's A rows and B half by
// TMA, counting the bytes on the LEADER's full barrier; warp 1 allocates TMEM
// (collectively for the pair) and, in the leader only, issues
// tcgen05.mma.cta_group::2 (M=256, N=256) and commits each stage to the empty
// barriers and each tile to the tmem-full barriers of both CTAs; warps 2-5 of
// each CTA drain its own 128 accumulator rows (as in the single-CTA kernel)
// and release the accumulator on the leader's tmem-empty barrier (8 arrivals:
// 4 local, 4 from the peer).  Every wait is bounded.
//
// Tiles are handed out dynamically: a scheduler warp of the leader (warp 6)
// takes tile indices from a global counter and publishes them in a small
// queue in both CTAs' shared memory, one tile ahead of the leader's producer
// (so the tiles in flight over the whole GPU stay about two per pair).  In the
// leader the producer, the MMA thread and the epilogue warps read that queue;
// in the peer only the producer does, and it forwards each tile to its
// epilogue warps through a second, CTA-local queue, so a tile costs one
// cluster-scope release each way and none on a loading thread.
// Pairs that run faster simply take more tiles, so the tiles in flight stay
// close to consecutive in the schedule's order and blocks that neighbouring
// tiles share are still in L2 when they are needed (a static round-robin
// assignment lets pairs drift apart over a long launch).
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BMP = 256;          // rows per pair tile (128 per CTA)
constexpr int BMC = 128;          // rows per CTA
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int kStages = 6;
constexpr int kMmaN = 256;
constexpr int kAccs = 2;
constexpr int kTmemCols = kMmaN * kAccs;
constexpr int A_BYTES = BMC * BK * 2;          // 16 KB
constexpr int B_BYTES = (kMmaN / 2) * BK * 2;  // 16 KB: this CTA's half of N
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 224;  // 6 warps + the tile scheduler warp
constexpr int kEpilogueWarps = 4;
constexpr int kStageCols = 64;
constexpr int kQ = 8;  // slots of the tile queues
// Readers of each slot of the leader's queue: its producer, MMA thread and 4
// epilogue warps, and the peer's producer.
constexpr int kQueueReaders = 2 + kEpilogueWarps + 1;
constexpr int kStageWarpBytes = 32 * kStageCols * 2;

struct Ctl {
    uint64_t full[kStages];    // leader: both CTAs' bytes of a stage
    uint64_t empty[kStages];   // each CTA: its stage may be refilled
    uint64_t tfull[kAccs];     // each CTA: accumulator ready
    uint64_t tempty[kAccs];    // leader: accumulator drained by both CTAs
    uint64_t done;             // leader: every issued MMA retired
    uint64_t tq_full[kQ];      // each CTA: queue slot written
    uint64_t tq_empty[kQ];     // leader: queue slot read by every reader of both CTAs
    int tile_q[kQ];            // each CTA: tile index (-1: no more tiles)
    uint64_t tq_taken[kQ];     // leader: its producer has taken the slot's tile
    uint64_t lq_full[kQ];      // peer: local queue slot written by its producer
    uint64_t lq_empty[kQ];     // peer: local queue slot read by its 4 epilogue warps
    int local_q[kQ];           // peer: the tiles forwarded to its epilogue
    uint32_t tmem_base;
    int abort;
    int prefix[kMaxE + 1];
    int offs[kMaxE];
    int cnts[kMaxE];
};

constexpr size_t kCtlBytes = (sizeof(Ctl) + 15) & ~size_t(15);
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * STAGE_BYTES +
                              (size_t)kEpilogueWarps * kStageWarpBytes + kCtlBytes;

// Leader's scheduler thread: wait until queue slot i % kQ is free in both CTAs, take
// the next tile from the counter (-1 once every tile is taken) and publish it
// to both CTAs.  Returns the tile, or -2 if the wait gave up.
__device__ __forceinline__ int queue_publish(Ctl* ctl, int i, int* counter, int total,
                                             volatile int* abort, int* err) {
    const int slot = i % kQ;
    const uint32_t ph = (uint32_t)(i / kQ) & 1u;
    if (!wait_bar(smem_u32(&ctl->tq_empty[slot]), ph ^ 1u, abort, err)) return -2;
    int t = atomicAdd(counter, 1);
    if (t >= total) t = -1;
    ctl->tile_q[slot] = t;
    st_shared_cluster(mapa_shared(smem_u32(&ctl->tile_q[slot]), 1), t);
    mbar_arrive(smem_u32(&ctl->tq_full[slot]));
    // release.cluster: the store into the peer's slot is visible before its arrival
    mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tq_full[slot]), 1));
    return t;
}

// Peer's producer: forward tile t to the peer's epilogue warps (local queue).
// Returns false if the wait gave up.
__device__ __forceinline__ bool local_publish(Ctl* ctl, int i, int t, volatile int* abort,
                                              int* err) {
    const int slot = i % kQ;
    const uint32_t ph = (uint32_t)(i / kQ) & 1u;
    if (!wait_bar(smem_u32(&ctl->lq_empty[slot]), ph ^ 1u, abort, err)) return false;
    ctl->local_q[slot] = t;
    mbar_arrive(smem_u32(&ctl->lq_full[slot]));
    return true;
}

// Peer's epilogue warp (lane 0): the tile in local queue slot i % kQ.
__device__ __forceinline__ int local_take(Ctl* ctl, int i, volatile int* abort, int* err) {
    const int slot = i % kQ;
    const uint32_t ph = (uint32_t)(i / kQ) & 1u;
    if (!wait_bar(smem_u32(&ctl->lq_full[slot]), ph, abort, err)) return -2;
    const int t = *reinterpret_cast<volatile int*>(&ctl->local_q[slot]);
    mbar_arrive(smem_u32(&ctl->lq_empty[slot]));
    return t;
}

// Reader of the leader's queue (the leader's producer, MMA thread and
// epilogue warps, the peer's producer): the tile in slot i % kQ (-1: none left), after which
// the slot is released to the leader.  Returns -2 if the wait gave up.
__device__ __forceinline__ int queue_take(Ctl* ctl, int i, bool leader, volatile int* abort,
                                          int* err) {
    const int slot = i % kQ;
    const uint32_t ph = (uint32_t)(i / kQ) & 1u;
    const uint32_t full = smem_u32(&ctl->tq_full[slot]);
    // the peer's copy was written by the leader: acquire at cluster scope
    if (!(leader ? wait_bar(full, ph, abort, err) : wait_bar_cluster(full, ph, abort, err)))
        return -2;
    const int t = *reinterpret_cast<volatile int*>(&ctl->tile_q[slot]);
    const uint32_t empty = smem_u32(&ctl->tq_empty[slot]);
    if (leader)
        mbar_arrive(empty);
    else
        mbar_arrive_cluster(mapa_shared(empty, 0));
    return t;
}

// Spin for about `cycles` SM clocks (lets copies in flight land on abort).
__device__ __forceinline__ void spin(long long cycles) {
    const long long t0 = clock64();
    while (clock64() - t0 < cycles) {
    }
}

template <bool kSwiGLU>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB0,
                             const __grid_constant__ CUtensorMap tmB1,
                             const __grid_constant__ CUtensorMap tmOut,
                             const int32_t* __restrict__ expert_offsets,
                             const int32_t* __restrict__ expert_counts,
                             int E, int K, int n_out, __nv_bfloat16* __restrict__ out,
                             int* err, int* tile_counter, int b_packed) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t tiles_addr = smem_u32(tiles);
    uint8_t* stage_area = tiles + (size_t)kStages * STAGE_BYTES;
    Ctl* ctl = reinterpret_cast<Ctl*>(stage_area + (size_t)kEpilogueWarps * kStageWarpBytes);
    volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();  // 0 = leader
    const bool leader = rank == 0;
    constexpr int BNo = kSwiGLU ? kMmaN / 2 : kMmaN;  // output columns per tile
    const int NB = (n_out + BNo - 1) / BNo;
    const int KB = (K + BK - 1) / BK;

    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        ctl->offs[i] = expert_offsets[i];
        ctl->cnts[i] = expert_counts[i];
    }
    __syncthreads();
    // the tile schedule: m-blocks of 256 rows before each expert, from the
    // counts (an epilogue warp, idle until the first accumulator is ready)
    if (warp == 2) warp_mblk_prefix(ctl->cnts, E, BMP, ctl->prefix);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < kAccs; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), 2 * kEpilogueWarps);
        }
        mbar_init(smem_u32(&ctl->done), 1);
        for (int q = 0; q < kQ; ++q) {
            mbar_init(smem_u32(&ctl->tq_full[q]), 1);
            mbar_init(smem_u32(&ctl->tq_empty[q]), kQueueReaders);
            mbar_init(smem_u32(&ctl->lq_full[q]), 1);
            mbar_init(smem_u32(&ctl->tq_taken[q]), 1);
            mbar_init(smem_u32(&ctl->lq_empty[q]), kEpilogueWarps);
        }
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmA);
        prefetch_map(&tmB0);
        if (kSwiGLU) prefetch_map(&tmB1);
        prefetch_map(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any remote signal
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const int total = ctl->prefix[E] * NB;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                int tile = queue_take(ctl, i, leader, abort_flag, err);
                if (leader && tile != -2) mbar_arrive(smem_u32(&ctl->tq_taken[i % kQ]));
                if (!leader && tile != -2 && !local_publish(ctl, i, tile, abort_flag, err))
                    tile = -2;
                if (tile == -2) ok = false;
                if (tile < 0) break;
                int e, mb, nb;
                decode_tile(ctl->prefix, E, NB, BMP, kMmaN, tile, e, mb, nb);
                const int row0 = ctl->offs[e] + mb * BMP + (int)rank * BMC;
                const int n0 = nb * BNo;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_local = smem_u32(&ctl->full[stage]);
                    const uint32_t full = mapa_shared(full_local, 0);
                    const uint32_t a_s = tiles_addr + stage * STAGE_BYTES;
                    const uint32_t b_s = a_s + A_BYTES;
                    if (leader) {
                        mbar_expect_tx(full_local, 2 * STAGE_BYTES);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    tma_load_2d_pair(a_s, &tmA, full, kb * BK, row0);
                    if (b_packed) {
                        // packed weights: this CTA's 128 rows of the tile's 256 x 64
                        // operand slice (gate rows in the leader, up rows in the peer)
                        tma_load_2d_pair(b_s, &tmB0, full, 0,
                                         ((e * NB + nb) * KB + kb) * kPackRows +
                                             (int)rank * (kMmaN / 2));
                    } else if (kSwiGLU) {
                        // leader holds the gate half of N, the peer the up half
                        tma_load_3d_pair(b_s, leader ? &tmB0 : &tmB1, full, kb * BK, n0, e);
                    } else {
                        tma_load_3d_pair(b_s, &tmB0, full, kb * BK, n0 + (int)rank * (kMmaN / 2),
                                         e);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                if (leader) {
                    for (int s = 0; s < kStages; ++s)
                        if ((armed >> s) & 1u)
                            wait_bar_drain(smem_u32(&ctl->full[s]), (armed_parity >> s) & 1u);
                } else {
                    spin(4000000);  // the leader holds the barrier of this CTA's copies
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader only) ----------------
        if (leader && lane == 0) {
            constexpr uint32_t idesc = make_idesc(BMP, kMmaN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int i = 0; ok; ++i) {
                if (queue_take(ctl, i, true, abort_flag, err) < 0) break;
                if (!wait_bar(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kMmaN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = tiles_addr + stage * STAGE_BYTES;
                    const uint64_t ad = sw128_desc(a_s);
                    const uint64_t bd = sw128_desc(a_s + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        umma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit_pair_multicast(smem_u32(&ctl->empty[stage]), 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_multicast(smem_u32(&ctl->tfull[acc]), 0x3);
                if (++acc == kAccs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair_multicast(smem_u32(&ctl->done), 0x1);
            wait_bar_drain(smem_u32(&ctl->done), 0);
        }
    } else if (warp < 2 + kEpilogueWarps) {
        // ---------------- epilogue (both CTAs): own 128 rows ----------------
        const int q = warp & 3;
        uint8_t* stage = stage_area + (size_t)(warp - 2) * kStageWarpBytes;
        const uint32_t stage_addr = smem_u32(stage);
        uint8_t* my_row = stage + lane * 128;
        const int sw = lane & 7;
        const uint32_t tempty_leader0 = mapa_shared(smem_u32(&ctl->tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_u32(&ctl->tempty[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int i = 0;; ++i) {
            int tile = 0;
            if (lane == 0)
                tile = leader ? queue_take(ctl, i, true, abort_flag, err)
                              : local_take(ctl, i, abort_flag, err);
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0) break;
            int e, mb, nb;
            decode_tile(ctl->prefix, E, NB, BMP, kMmaN, tile, e, mb, nb);
            const int row_base = ctl->offs[e] + mb * BMP + (int)rank * BMC + q * 32;
            int rows_valid = ctl->offs[e] + ctl->cnts[e] - row_base;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > 32 ? 32 : rows_valid);
            const int n0 = nb * BNo;
            int ready = 0;
            if (lane == 0) ready = wait_bar(smem_u32(&ctl->tfull[acc]), acc_phase, abort_flag, err);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kMmaN);
#pragma unroll 1
            for (int c = 0; c < BNo / kStageCols; ++c) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint32_t col_t = (uint32_t)(c * kStageCols + half * 32);
                    uint32_t g[32], u[32];
                    tmem_ld32(tbase + col_t, g);
                    if (kSwiGLU) tmem_ld32(tbase + BNo + col_t, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int grp = 0; grp < 4; ++grp) {
                        uint4 o;
                        uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int j = grp * 8 + 2 * i;
                            if (kSwiGLU) {
                                const float h0 = silu(__uint_as_float(g[j])) * __uint_as_float(u[j]);
                                const float h1 =
                                    silu(__uint_as_float(g[j + 1])) * __uint_as_float(u[j + 1]);
                                op[i] = pack2(h0, h1);
                            } else {
                                op[i] = pack2(__uint_as_float(g[j]), __uint_as_float(g[j + 1]));
                            }
                        }
                        const int chunk = half * 4 + grp;
                        *reinterpret_cast<uint4*>(my_row + ((chunk ^ sw) << 4)) = o;
                    }
                }
                const int col0 = n0 + c * kStageCols;
                if (rows_valid == 32) {
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOut, stage_addr, col0, row_base);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    const int qq = lane & 7;
                    const int col = col0 + qq * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = i * 4 + (lane >> 3);
                        if (rr < rows_valid && col < n_out) {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                stage + rr * 128 + ((qq ^ (rr & 7)) << 4));
                            *reinterpret_cast<uint4*>(out + (size_t)(row_base + rr) * n_out + col) =
                                v;
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc == 0 ? tempty_leader0 : tempty_leader1);
            if (++acc == kAccs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if (leader && lane == 0) {
        // ---------------- tile scheduler (leader) ----------------
        // index i is published once the producer has taken index i - 1
        for (int i = 0;; ++i) {
            if (i > 0) {
                const int j = i - 1;
                if (!wait_bar(smem_u32(&ctl->tq_taken[j % kQ]), (uint32_t)(j / kQ) & 1u,
                              abort_flag, err))
                    break;
            }
            if (queue_publish(ctl, i, tile_counter, total, abort_flag, err) < 0) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
    // The tile counter returns to zero for the next launch: every pair counts
    // itself out once its scheduler is past its last fetch (the barriers
    // above), and the last pair out resets both counters.  Nothing waits here.
    if (leader && threadIdx.x == 0) {
        __threadfence();
        const int before = atomicAdd(tile_counter + 1, 1);
        if (before == (int)(gridDim.x / 2) - 1) {
            atomicExch(tile_counter, 0);
            atomicExch(tile_counter + 1, 0);
        }
    }
}

bool set_pair_smem_attr() {
    return cudaFuncSetAttribute(grouped_gemm_pair_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(grouped_gemm_pair_kernel<false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess;
}

// Grid of the 256-row tiles: 2 CTAs per pair, at most one CTA per SM.  (The
// kernel derives the tile schedule itself from the expert counts.)
moe_status pair_schedule(const GemmGroup& g, long long n_blocks, cudaStream_t st, int* grid) {
    (void)st;
    const long long tiles = n_blocks * ((g.R + BMP - 1) / BMP + g.E);
    const long long pairs_max = sm_count() / 2;
    const long long pairs = tiles < pairs_max ? tiles : pairs_max;
    *grid = (int)(2 * (pairs > 0 ? pairs : 1));
    return MOE_OK;
}

}  // namespace

moe_status launch_gate_up_pair(const uint16_t* rows, const GemmGroup& g, int H, int I,
                               const uint16_t* wg, const uint16_t* wu, uint16_t* h,
                               cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    CUtensorMap a, bg, bu, o;
    const bool ok_b = g.packed ? map_packed(&bg, &bu, wg, g.E, (I + 127) / 128, H, kMmaN / 2)
                               : map_3d(&bg, wg, g.E, I, H, kMmaN / 2) &&
                                     map_3d(&bu, wu, g.E, I, H, kMmaN / 2);
    if (!map_2d(&a, rows, g.R, H, BMC) || !ok_b || !map_2d(&o, h, g.R, I, 32))
        return MOE_ERR_UNSUPPORTED;
    if (!set_pair_smem_attr()) return MOE_ERR_CUDA;
    int grid;
    const moe_status ss = pair_schedule(g, (I + kMmaN / 2 - 1) / (kMmaN / 2), st, &grid);
    if (ss != MOE_OK) return ss;
    grouped_gemm_pair_kernel<true><<<grid, kThreads, kSmemBytes, st>>>(
        a, bg, bu, o, g.offsets, g.counts, g.E, H, I,
        reinterpret_cast<__nv_bfloat16*>(h), g.err, g.prefix + g.E + 1, g.packed ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_down_pair(const uint16_t* h, const GemmGroup& g, int H, int I,
                            const uint16_t* wd, uint16_t* y, cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    CUtensorMap a, bd, unused, o;
    const bool ok_b = g.packed ? map_packed(&bd, &unused, wd, g.E, (H + 255) / 256, I, kMmaN / 2)
                               : map_3d(&bd, wd, g.E, H, I, kMmaN / 2);
    if (!map_2d(&a, h, g.R, I, BMC) || !ok_b || !map_2d(&o, y, g.R, H, 32))
        return MOE_ERR_UNSUPPORTED;
    if (!set_pair_smem_attr()) return MOE_ERR_CUDA;
    int grid;
    const moe_status ss = pair_schedule(g, (H + kMmaN - 1) / kMmaN, st, &grid);
    if (ss != MOE_OK) return ss;
    grouped_gemm_pair_kernel<false><<<grid, kThreads, kSmemBytes, st>>>(
        a, bd, bd, o, g.offsets, g.counts, g.E, I, H,
        reinterpret_cast<__nv_bfloat16*>(y), g.err, g.prefix + g.E + 1, g.packed ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
