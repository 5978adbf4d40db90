// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// FarSkip-Collective (arXiv 2511.11505) Sec. 2.1: the gated expert MLP; "Kernel
// fusion for expert parallelism", section "Fusing the layer into one kernel",
// stages 4-6: the gate/up MatMul, the SwiGLU activation and the down MatMul of
// every expert over its expert-contiguous rows ("Expert Coupling" Appendix
// A-A1: dispatch feeds a grouped GEMM).
//
// Two launches of one persistent, warp-specialised kernel:
//   gate/up:  one 128x256 MMA tile holds 128 gate columns and the matching 128
//             up columns of the same rows, so the epilogue can apply
//             h = SiLU(g) * u straight out of TMEM and store bf16 h.
//   down:     a 128x256 tile of y = h Wd^T, stored as bf16.
// The weight operand B comes from the row-major [E, rows, K] matrices (a 3-D
// map, 256 strided 128-byte pieces per k-block) or from their packed copy
// (moe_pack_weights: each k-block of a 256-row tile one contiguous 32 KB
// block of a [rows, 64] map), which the HBM-bound shapes stream faster.
// Roles (192 threads, 320 with gathered rows): warp 0 issues TMA loads into a
// 4-stage shared-memory ring (128B swizzle; with gathered rows only B, while
// warps 6-9 copy the A rows in with cp.async), warp 1 owns TMEM and issues
// tcgen05.mma from one thread
// (fp32 accumulators, two 256-column buffers so the epilogue of one tile
// overlaps the main loop of the next), warps 2-5 read the accumulators back
// with tcgen05.ld, stage 64 output columns of their 32 rows in shared memory
// and write them out with a TMA store (or masked row-line stores at the ragged
// end of an expert's segment).  Tiles of an expert never cross into
// the next expert's rows on store: rows past the segment end are masked, so
// no padding of the expert-major layout is needed.  Every wait is bounded; a
// wait that runs out of time records MOE_ERR_TIMEOUT, the CTA drains what it
// has in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <cstring>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = kGemmBM;       // rows per tile (TMEM lanes)
constexpr int BK = 64;            // bf16 elements per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 16;        // K of one kind::f16 MMA
constexpr int kStages = 4;
constexpr int kMmaN = 256;        // columns per MMA and per accumulator
constexpr int kAccs = 2;
constexpr int kTmemCols = kMmaN * kAccs;  // 512: the whole TMEM of the SM
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BYTES = kMmaN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr int kEpilogueWarps = 4;
// Gathered A rows (kGather): row i of the problem is row a_rows[i] of a
// source matrix (x through row_token, or the dedup rows through expand_src),
// copied by 4 extra gather warps with 16-byte cp.async into the 128B-swizzled
// layout a TMA box would have produced; B still comes by TMA.  This replaces
// a separate copy kernel that would write the rows out and read them back.
constexpr int kGatherWarps = 4;
constexpr int kGatherThreads = kGatherWarps * 32;
__host__ __device__ constexpr int threads_for(bool gather) {
    return gather ? kThreads + kGatherThreads : kThreads;
}

struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[kAccs];
    uint64_t tempty[kAccs];
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    int prefix[kMaxE + 1];
    int offs[kMaxE];
    int cnts[kMaxE];
};

// Epilogue staging: each epilogue warp writes its 32 rows x 64 output columns
// (bf16, 4 KB) into shared memory in the 128-byte swizzled layout of a TMA
// box; a slice whose 32 rows all belong to the tile's expert leaves by one
// asynchronous TMA tensor store, a ragged slice at the end of an expert's
// segment by masked 16-byte stores of whole row lines.
constexpr int kStageCols = 64;
constexpr int kStageWarpBytes = 32 * kStageCols * 2;  // 4 KB, 1024-byte aligned
constexpr size_t kCtlBytes = (sizeof(Ctl) + 15) & ~size_t(15);

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * STAGE_BYTES +
                              (size_t)kEpilogueWarps * kStageWarpBytes + kCtlBytes;

using namespace ptx;

// kGather: A row i of the problem is row a_rows[i] of a_src (rows >= a_total
// and indices outside [0, a_src_rows) read row 0; such rows are masked on
// store); otherwise row i of tmA's tensor.
// kCombine (down only): instead of storing y, the epilogue scales row i by its
// routing weight and adds it into cmb.acc[token of row i] with fp32 vector
// atomics (the combine of "Kernel fusion for expert parallelism", stage 7,
// moved into the MatMul's epilogue).
template <bool kSwiGLU, bool kGather, bool kCombine>
__global__ void __launch_bounds__(threads_for(kGather), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmOut,
                        const int32_t* __restrict__ expert_offsets,
                        const int32_t* __restrict__ expert_counts,
                        int E, int K, int n_out,
                        __nv_bfloat16* __restrict__ out, int* err,
                        const int32_t* __restrict__ a_rows, int a_total, int a_src_rows,
                        const uint16_t* __restrict__ a_src, int a_keep, const CombineArgs cmb,
                        int b_packed) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* tiles = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t tiles_addr = smem_u32(tiles);
    uint8_t* stage_area = tiles + (size_t)kStages * STAGE_BYTES;  // 1024-byte aligned
    Ctl* ctl = reinterpret_cast<Ctl*>(stage_area + (size_t)kEpilogueWarps * kStageWarpBytes);
    volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int BNo = kSwiGLU ? kMmaN / 2 : kMmaN;  // output columns per tile
    const int NB = (n_out + BNo - 1) / BNo;
    const int KB = (K + BK - 1) / BK;

    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        ctl->offs[i] = expert_offsets[i];
        ctl->cnts[i] = expert_counts[i];
    }
    __syncthreads();
    // the tile schedule: m-blocks before each expert, from the counts (an
    // epilogue warp, idle until the first accumulator is ready)
    if (warp == 2) warp_mblk_prefix(ctl->cnts, E, BM, ctl->prefix);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // kGather: the producer's arrive plus one cp.async arrival per gather thread
            mbar_init(smem_u32(&ctl->full[s]), kGather ? 1 + kGatherThreads : 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < kAccs; ++a) {
            mbar_init(smem_u32(&ctl->tfull[a]), 1);
            mbar_init(smem_u32(&ctl->tempty[a]), kEpilogueWarps);
        }
        mbar_init(smem_u32(&ctl->done), 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        if (!kGather) prefetch_map(&tmA);
        prefetch_map(&tmB0);
        if (kSwiGLU) prefetch_map(&tmB1);
        if (!kCombine) prefetch_map(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const int total = ctl->prefix[E] * NB;

    if (warp == 0) {
        // ---------------- TMA producer (A unless gathered, and B) ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int e, mb, nb;
                decode_tile(ctl->prefix, E, NB, BM, kMmaN, tile, e, mb, nb);
                const int row0 = ctl->offs[e] + mb * BM;
                const int n0 = nb * BNo;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&ctl->full[stage]);
                    const uint32_t a_s = tiles_addr + stage * STAGE_BYTES;
                    const uint32_t b_s = a_s + A_BYTES;
                    mbar_expect_tx(full, kGather ? B_BYTES : STAGE_BYTES);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (b_packed) {
                        // packed weights: the tile's 256 x 64 operand slice is one
                        // contiguous block of the [rows, 64] map
                        tma_load_2d(b_s, &tmB0, full, 0, ((e * NB + nb) * KB + kb) * kPackRows);
                    } else if (kSwiGLU) {
                        tma_load_3d(b_s, &tmB0, full, kb * BK, n0, e);
                        tma_load_3d(b_s + B_BYTES / 2, &tmB1, full, kb * BK, n0, e);
                    } else {
                        tma_load_3d(b_s, &tmB0, full, kb * BK, n0, e);
                    }
                    if (!kGather) tma_load_2d(a_s, &tmA, full, kb * BK, row0);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort_flag) {
                // let every copy still in flight land before the CTA exits
                for (int s = 0; s < kStages; ++s)
                    if ((armed >> s) & 1u)
                        wait_bar_drain(smem_u32(&ctl->full[s]), (armed_parity >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(BM, kMmaN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                if (!wait_bar(smem_u32(&ctl->tempty[acc]), acc_phase ^ 1u, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kMmaN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // A rows written through the generic proxy (cp.async) are
                    // read by the MMA through the async proxy
                    if (kGather) fence_async_shared();
                    const uint32_t a_s = tiles_addr + stage * STAGE_BYTES;
                    const uint64_t ad = sw128_desc(a_s);
                    const uint64_t bd = sw128_desc(a_s + A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        // advance 16 elements = 32 bytes along K inside the swizzle row
                        umma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                  (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&ctl->tfull[acc]));
                if (++acc == kAccs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // every MMA issued by this thread has retired once `done` fires
            umma_commit(smem_u32(&ctl->done));
            wait_bar_drain(smem_u32(&ctl->done), 0);
        }
    } else if (warp < 2 + kEpilogueWarps) {
        // ---------------- epilogue: TMEM -> registers -> smem -> global ----------------
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        uint8_t* stage = stage_area + (size_t)(warp - 2) * kStageWarpBytes;
        const uint32_t stage_addr = smem_u32(stage);
        // lane r's row; 16-byte chunk j of it sits at chunk (j ^ (r & 7)) (128B swizzle)
        uint8_t* my_row = stage + lane * 128;
        const int sw = lane & 7;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int e, mb, nb;
            decode_tile(ctl->prefix, E, NB, BM, kMmaN, tile, e, mb, nb);
            const int row_base = ctl->offs[e] + mb * BM + q * 32;  // this warp's first row
            int rows_valid = ctl->offs[e] + ctl->cnts[e] - row_base;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > 32 ? 32 : rows_valid);
            const int n0 = nb * BNo;
            int ready = 0;
            if (lane == 0) ready = wait_bar(smem_u32(&ctl->tfull[acc]), acc_phase, abort_flag, err);
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kMmaN);
            if constexpr (kCombine) {
                // this lane's row: its token and routing weight (the j with
                // pair_row[t, j] == row)
                const int i = row_base + lane;
                int t = 0;
                float wr = 0.f;
                if (lane < rows_valid) {
                    const int tt = cmb.row_token[i];
                    t = (unsigned)tt < (unsigned)cmb.N ? tt : 0;
                    for (int j = 0; j < cmb.k; ++j) {
                        if (cmb.pair_row[(size_t)t * cmb.k + j] == i) {
                            wr = cmb.topk_w[(size_t)t * cmb.k + j];
                            break;
                        }
                    }
                }
                // 32 columns at a time: each lane stages its scaled row (128 B,
                // swizzled), then 8 lanes per row add whole 128-byte lines
                const int qq = lane & 7;
#pragma unroll 1
                for (int c = 0; c < BNo / 32; ++c) {
                    uint32_t g[32];
                    tmem_ld32(tbase + (uint32_t)(c * 32), g);
                    tmem_wait_ld();
                    __syncwarp();  // the previous slice's reads of the staging tile are done
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const float4 v = make_float4(wr * __uint_as_float(g[4 * ch]),
                                                     wr * __uint_as_float(g[4 * ch + 1]),
                                                     wr * __uint_as_float(g[4 * ch + 2]),
                                                     wr * __uint_as_float(g[4 * ch + 3]));
                        *reinterpret_cast<float4*>(my_row + ((ch ^ sw) << 4)) = v;
                    }
                    __syncwarp();
                    const int col = n0 + c * 32 + qq * 4;  // n_out % 8 == 0: 4 columns in or out
#pragma unroll
                    for (int pp = 0; pp < 8; ++pp) {
                        const int rr = pp * 4 + (lane >> 3);
                        const int tr = __shfl_sync(0xffffffffu, t, rr);
                        if (rr < rows_valid && col < n_out) {
                            const float4 v = *reinterpret_cast<const float4*>(
                                stage + rr * 128 + ((qq ^ (rr & 7)) << 4));
                            atomicAdd(reinterpret_cast<float4*>(cmb.acc + (size_t)tr * n_out + col),
                                      v);
                        }
                    }
                }
            } else {
#pragma unroll 1
            for (int c = 0; c < BNo / kStageCols; ++c) {
                // the staging tile is free once the previous TMA store has read it
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                // 1) this lane's row: 64 bf16 values into its staged row
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
                    // 2a) whole slice inside the expert: one TMA store (columns past
                    // n_out are clipped by the tensor map)
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOut, stage_addr, col0, row_base);
                        bulk_commit();
                    }
                } else {
                    // 2b) ragged slice: whole row lines, masked; pass i stores rows 4i..4i+3
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
            }  // kCombine
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
            if (++acc == kAccs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if (kGather) {
        // ---------------- gather warps (kGather): A rows by cp.async ----------------
        // Instruction i of a stage covers rows 16i + 4g .. 16i + 4g + 3 (g = gather
        // warp); 8 lanes copy the 8 16-byte chunks of one row's 128-byte k-block,
        // so every instruction reads 4 whole 128-byte lines.
        const int g = warp - 2 - kEpilogueWarps;
        const int chunk = lane & 7;
        const int rsub = g * 4 + (lane >> 3);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            int e, mb, nb;
            decode_tile(ctl->prefix, E, NB, BM, kMmaN, tile, e, mb, nb);
            const int row0 = ctl->offs[e] + mb * BM;
            const uint16_t* src[BM / 16];
#pragma unroll
            for (int i = 0; i < BM / 16; ++i) {
                const int r = row0 + i * 16 + rsub;  // rows past the data read row 0
                const int v = r < a_total ? a_rows[r] : 0;
                src[i] = a_src + (size_t)((unsigned)v < (unsigned)a_src_rows ? v : 0) * K;
            }
            for (int kb = 0; kb < KB; ++kb) {
                int go = 1;
                if (lane == 0)
                    go = wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, err);
                go = __shfl_sync(0xffffffffu, go, 0);
                if (!go) {
                    ok = false;
                    break;
                }
                const uint32_t a_s = tiles_addr + stage * STAGE_BYTES;
                const int col = kb * BK + chunk * 8;
                const bool in = col < K;  // K % 8 == 0: a chunk is wholly in or out
                if (a_keep) {
                    // a source small enough to stay in L2 is read there by the
                    // later experts of each token, not from HBM again
                    const uint64_t pol = policy_evict_last(1.0f);
#pragma unroll
                    for (int i = 0; i < BM / 16; ++i) {
                        const int r = i * 16 + rsub;
                        cp_async_16_hint(a_s + r * 128 + ((chunk ^ (r & 7)) << 4),
                                         src[i] + (in ? col : 0), in ? 16u : 0u, pol);
                    }
                } else {
#pragma unroll
                for (int i = 0; i < BM / 16; ++i) {
                    const int r = i * 16 + rsub;
                    cp_async_16(a_s + r * 128 + ((chunk ^ (r & 7)) << 4), src[i] + (in ? col : 0),
                                in ? 16u : 0u);
                }
                }
                cp_async_arrive_noinc(smem_u32(&ctl->full[stage]));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // no copy may land after the CTA has gone
        cp_async_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// 2-D bf16 map over a row-major [rows, cols] matrix; box = 64 columns x box_rows.
bool map_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [E, rows, cols]; box = 64 columns x box_rows x 1 expert.
bool map_3d(CUtensorMap* m, const void* ptr, uint64_t E, uint64_t rows, uint64_t cols,
            uint32_t box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {cols, rows, E};
    cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over packed weights (E experts x n_blocks n-blocks x ceil(K/64) k-blocks
// of 256 x 64 bf16) as a [rows, 64] matrix; box = box_rows rows.  *second is
// set to the same map (the kernels take a second B map for row-major up
// weights).
bool map_packed(CUtensorMap* m, CUtensorMap* second, const void* ptr, int E, int n_blocks, int K,
                uint32_t box_rows) {
    const long long rows = packed_rows(E, n_blocks, K);
    if (rows >= (1LL << 31) || !map_2d(m, ptr, (uint64_t)rows, 64, box_rows)) return false;
    *second = *m;
    return true;
}

namespace {

bool set_smem_attr() {
    return cudaFuncSetAttribute(grouped_gemm_kernel<true, false, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(grouped_gemm_kernel<true, true, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(grouped_gemm_kernel<false, false, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(grouped_gemm_kernel<false, false, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess;
}

// The persistent grid size for a GEMM with `n_blocks` n-blocks: never more
// CTAs than tiles, never more than one per SM.  (The kernel derives the tile
// schedule itself from the expert counts.)
moe_status schedule(const GemmGroup& g, long long n_blocks, cudaStream_t st, int* grid) {
    (void)st;
    // tiles <= n_blocks * (ceil(R / BM) + E): each expert adds at most one ragged m-block
    const long long tiles = n_blocks * ((g.R + BM - 1) / BM + g.E);
    const int sms = sm_count();
    *grid = (int)(tiles < sms ? tiles : sms);
    return MOE_OK;
}

}  // namespace

moe_status launch_gate_up(const uint16_t* rows, const GemmGroup& g, int H, int I,
                          const uint16_t* wg, const uint16_t* wu, uint16_t* h, cudaStream_t st,
                          const int32_t* gather, long long src_rows) {
    if (g.R == 0) return MOE_OK;
    CUtensorMap a, bg, bu, o;
    bool ok_a = true;
    // gathered rows are re-read by every expert of their token: ask L2 to keep
    // the source when it is at most half of L2 (x of the DeepSeek-V3 shape:
    // 59 MB), never for the larger dedup sources
    const bool keep_src = gather && src_rows * (long long)H * 2 <= (64LL << 20);
    if (gather)
        memset(&a, 0, sizeof(a));  // unused: the gather warps read `rows` directly
    else
        ok_a = map_2d(&a, rows, g.R, H, BM);
    const bool ok_b = g.packed ? map_packed(&bg, &bu, wg, g.E, (I + 127) / 128, H, kMmaN)
                               : map_3d(&bg, wg, g.E, I, H, kMmaN / 2) &&
                                     map_3d(&bu, wu, g.E, I, H, kMmaN / 2);
    if (!ok_a || !ok_b || !map_2d(&o, h, g.R, I, 32)) return MOE_ERR_UNSUPPORTED;
    if (!set_smem_attr()) return MOE_ERR_CUDA;
    int grid;
    const moe_status ss = schedule(g, (I + kMmaN / 2 - 1) / (kMmaN / 2), st, &grid);
    if (ss != MOE_OK) return ss;
    __nv_bfloat16* hb = reinterpret_cast<__nv_bfloat16*>(h);
    if (gather)
        grouped_gemm_kernel<true, true, false><<<grid, threads_for(true), kSmemBytes, st>>>(
            a, bg, bu, o, g.offsets, g.counts, g.E, H, I, hb, g.err, gather, (int)g.R,
            (int)src_rows, rows, keep_src ? 1 : 0, CombineArgs{}, g.packed ? 1 : 0);
    else
        grouped_gemm_kernel<true, false, false><<<grid, kThreads, kSmemBytes, st>>>(
            a, bg, bu, o, g.offsets, g.counts, g.E, H, I, hb, g.err, nullptr, 0, 0,
            nullptr, 0, CombineArgs{}, g.packed ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_down(const uint16_t* h, const GemmGroup& g, int H, int I, const uint16_t* wd,
                       uint16_t* y, cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    CUtensorMap a, bd, unused, o;
    const bool ok_b = g.packed ? map_packed(&bd, &unused, wd, g.E, (H + 255) / 256, I, kMmaN)
                               : map_3d(&bd, wd, g.E, H, I, kMmaN);
    if (!map_2d(&a, h, g.R, I, BM) || !ok_b || !map_2d(&o, y, g.R, H, 32))
        return MOE_ERR_UNSUPPORTED;
    if (!set_smem_attr()) return MOE_ERR_CUDA;
    int grid;
    const moe_status ss = schedule(g, (H + kMmaN - 1) / kMmaN, st, &grid);
    if (ss != MOE_OK) return ss;
    grouped_gemm_kernel<false, false, false><<<grid, kThreads, kSmemBytes, st>>>(
        a, bd, bd, o, g.offsets, g.counts, g.E, I, H,
        reinterpret_cast<__nv_bfloat16*>(y), g.err, nullptr, 0, 0, nullptr, 0, CombineArgs{},
        g.packed ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_down_combine(const uint16_t* h, const GemmGroup& g, int H, int I,
                               const uint16_t* wd, const CombineArgs& cmb, cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    CUtensorMap a, bd, unused, o;
    memset(&o, 0, sizeof(o));  // unused: the epilogue adds into cmb.acc
    const bool ok_b = g.packed ? map_packed(&bd, &unused, wd, g.E, (H + 255) / 256, I, kMmaN)
                               : map_3d(&bd, wd, g.E, H, I, kMmaN);
    if (!map_2d(&a, h, g.R, I, BM) || !ok_b) return MOE_ERR_UNSUPPORTED;
    if (!set_smem_attr()) return MOE_ERR_CUDA;
    int grid;
    const moe_status ss = schedule(g, (H + kMmaN - 1) / kMmaN, st, &grid);
    if (ss != MOE_OK) return ss;
    grouped_gemm_kernel<false, false, true><<<grid, kThreads, kSmemBytes, st>>>(
        a, bd, bd, o, g.offsets, g.counts, g.E, I, H, nullptr, g.err, nullptr, 0, 0,
        nullptr, 0, cmb, g.packed ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Self-test of the bounded wait: one warp waits on an mbarrier whose phase
// nothing completes, with the limit given in SM clock cycles.  The wait must
// give up, record MOE_ERR_TIMEOUT and let the kernel return.
__global__ void wait_selftest_kernel(long long limit_cycles, int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&bar), 0)) {
            if (clock64() - t0 > limit_cycles) {
                set_error(err, MOE_ERR_TIMEOUT);
                break;
            }
        }
    }
    __syncthreads();
}

cudaError_t launch_wait_selftest(long long limit_cycles, int* err, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_cycles, err);
    return cudaGetLastError();
}

__global__ void dense_group_kernel(int N, int32_t* counts, int32_t* offsets) {
    counts[0] = N;
    offsets[0] = 0;
    offsets[1] = N;
}

cudaError_t launch_dense_group(int N, int32_t* counts, int32_t* offsets, cudaStream_t st) {
    dense_group_kernel<<<1, 1, 0, st>>>(N, counts, offsets);
    return cudaGetLastError();
}

}  // namespace moe
