// The expert FFN with h kept on chip, wide form: the kernel of fused_ffn.cu
// on 128-column chunks of I, for layers with a large I.
//
// "Kernel fusion for expert parallelism", section "Fusing the layer into one
// kernel" (expert intermediates kept in the SM's local memory between the two
// MatMuls); FarSkip-Collective (arXiv 2511.11505) Sec. 2.1 (h = SiLU(x Wg^T) *
// (x Wu^T), y = h Wd^T).  Same results, bit for bit, as fused_ffn.cu's
// 64-column form and as the two GEMMs.
//
// Why a second form: one thread issues every MMA, and each ring stage costs
// it a fixed few hundred cycles (barrier wait, four MMA issues, commit)
// whatever the stage carries.  The 64-column form's stages are 128 x 128 x 64
// MMA chains, 256 tensor cycles, so on a long I its tensor pipe waits on the
// issuing thread; here a stage is a 128 x 256 x 64 chain (g and u of 128
// columns of I at once), 512 tensor cycles.  The price is TMEM: the 256-column
// gate/up accumulator and y's H <= 256 columns fill all 512, so the
// accumulator is single-buffered.  The epilogue warps read it out of TMEM
// while the tensor pipe runs the previous chunk's down MMAs, then turn it into
// h while the next chunk's gate/up runs; with few chunks (small I) there is
// little to overlap, which is why the 64-column form keeps those layers.
//
// Per tile (persistent CTAs, tiles = 128-row m-blocks of each expert):
//   x tile   [128, H] bf16 gathered once into shared memory (swizzled k-blocks)
//   chunk c  g|u[128, 256] = x (Wg|Wu)[e][128c..128c+127, :]^T       (TMEM)
//            h_c = bf16(SiLU(g) * u)  -> the shared h tile (swizzled)
//            y[128, H] += h_c Wd[e][:, 128c..128c+127]^T              (TMEM, fp32)
//   y        bf16 -> HBM (16-byte stores of each lane's row, masked at the ends)
// The fp32 accumulation orders are those of the two-kernel path (k-blocks of
// x for g and u, 64-column k-blocks of h for y, 16-deep MMAs in order), and h
// is rounded to bf16 the same way.
//
// Roles (384 threads): warp 0 TMA-loads weight k-blocks into a ring of 32 KB
// stages (a 256-row gate|up k-block, or the down k-block of round_up(H, 32)
// rows); warp 1 owns TMEM and issues tcgen05.mma; warps 2-9 turn g|u into h
// and drain y, two warps per TMEM lane quadrant, each on 64 of a chunk's 128
// columns; warps 10-11 gather the x rows with 16-byte cp.async.  Every wait is
// bounded; a wait that runs out records MOE_ERR_TIMEOUT and the CTA drains
// and returns.
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = kGemmBM;        // rows per tile (TMEM lanes)
constexpr int BK = 64;             // bf16 per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kChunk = 128;        // columns of I per chunk
constexpr int kGuN = 2 * kChunk;   // gate/up MMA N: 128 gate + 128 up columns
constexpr int kMaxStages = 6;
constexpr int kEpilogueWarps = 8;
constexpr int kGatherWarps = 2;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kThreads = (2 + kEpilogueWarps + kGatherWarps) * 32;
constexpr int kTileBytes = BM * BK * 2;      // 16 KB: 128 rows x one k-block
constexpr int kHBytes = 2 * kTileBytes;      // the h tile: 128 rows x 128 columns
constexpr int kStageBytes = kGuN * BK * 2;   // 32 KB: a gate|up k-block (>= any down k-block)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kYCol = kGuN;             // y accumulator: TMEM columns 256..511
constexpr int kSmemLimit = 227 * 1024;

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t x_full, x_empty;  // x tile gathered / read by the last gate/up MMA
    uint64_t a_full, a_empty;  // gate/up accumulator computed / read out
    uint64_t h_full, h_empty;  // h tile written / read by the down MMA
    uint64_t y_full, y_empty;  // y accumulator complete / read out
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    int prefix[kMaxE + 1];
};
constexpr size_t kCtlBytes = (sizeof(Ctl) + 15) & ~size_t(15);

// Shared memory after the 1024-byte alignment: x tile, h tile, the weight
// ring, Ctl.
struct SmemPlan {
    int stages;
    size_t bytes;
};

__host__ __device__ inline int y_cols(int H) { return (H + 31) / 32 * 32; }

SmemPlan smem_plan(int H) {
    SmemPlan p;
    const int kbx = (H + BK - 1) / BK;
    const size_t fixed = 1024 + (size_t)kbx * kTileBytes + kHBytes + kCtlBytes;
    long long st = ((long long)kSmemLimit - (long long)fixed) / kStageBytes;
    if (st > kMaxStages) st = kMaxStages;
    p.stages = (int)st;
    p.bytes = fixed + (size_t)p.stages * kStageBytes;
    return p;
}

// 8 bf16 of h = SiLU(g) * u from 8 fp32 accumulator columns of g and of u.
__device__ __forceinline__ uint4 swiglu8(const uint32_t* g, const uint32_t* u) {
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float h0 = silu(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
        const float h1 = silu(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
        op[i] = pack2(h0, h1);
    }
    return o;
}

// a_rows == nullptr: tile row i is row i of a_src.  Otherwise row a_rows[i]
// (rows >= a_total and indices outside [0, a_src_rows) read row 0; such rows
// are masked on store).
__global__ void __launch_bounds__(kThreads, 1)
    fused_ffn_wide_kernel(const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmD,
                     const int32_t* __restrict__ expert_offsets,
                     const int32_t* __restrict__ expert_counts, int E, int H, int I,
                     __nv_bfloat16* __restrict__ y, int* err,
                     const int32_t* __restrict__ a_rows, int a_total, int a_src_rows,
                     const uint16_t* __restrict__ a_src, int b_packed, int n_stages) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int KBX = (H + BK - 1) / BK;         // k-blocks of x
    const int NC = (I + kChunk - 1) / kChunk;  // chunks of I
    const int KBD = (I + BK - 1) / BK;         // k-blocks of the down GEMM
    const int NY = y_cols(H);
    const uint32_t x_addr = smem_u32(base);
    const uint32_t h_addr = x_addr + (uint32_t)KBX * kTileBytes;
    uint8_t* h_ptr = base + (size_t)KBX * kTileBytes;
    const uint32_t ring_addr = h_addr + (uint32_t)kHBytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(h_ptr + kHBytes + (size_t)n_stages * kStageBytes);
    volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the tile schedule: m-blocks before each expert, from the counts
    if (warp == 2) warp_mblk_prefix(expert_counts, E, BM, ctl->prefix);
    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->x_full), kGatherThreads);
        mbar_init(smem_u32(&ctl->x_empty), 1);
        mbar_init(smem_u32(&ctl->a_full), 1);
        mbar_init(smem_u32(&ctl->a_empty), kEpilogueWarps);
        mbar_init(smem_u32(&ctl->h_full), kEpilogueWarps);
        mbar_init(smem_u32(&ctl->h_empty), 1);
        mbar_init(smem_u32(&ctl->y_full), 1);
        mbar_init(smem_u32(&ctl->y_empty), kEpilogueWarps);
        mbar_init(smem_u32(&ctl->done), 1);
        ctl->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_map(&tmG);
        if (!b_packed) prefetch_map(&tmU);
        prefetch_map(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const int total = ctl->prefix[E];  // one tile per m-block: every column in one CTA

    if (warp == 0) {
        // ---------------- TMA producer: weight k-blocks in the MMA's order ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            // the next ring stage: wait until it is free, arm it for `bytes`
            auto next = [&](uint32_t bytes, uint32_t& dst, uint32_t& full) -> bool {
                if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, err))
                    return false;
                full = smem_u32(&ctl->full[stage]);
                dst = ring_addr + (uint32_t)stage * (uint32_t)kStageBytes;
                mbar_expect_tx(full, bytes);
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == n_stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return true;
            };
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int e, mb, nb;
                decode_tile(ctl->prefix, E, 1, BM, NY, tile, e, mb, nb);
                for (int c = 0; ok && c <= NC; ++c) {
                    if (c < NC) {
                        for (int kb = 0; kb < KBX; ++kb) {
                            uint32_t dst, full;
                            if (!next(kStageBytes, dst, full)) {
                                ok = false;
                                break;
                            }
                            if (b_packed) {
                                // block (e, c, kb): gate rows 0..127, up rows 128..255
                                tma_load_2d(dst, &tmG, full, 0,
                                            ((e * NC + c) * KBX + kb) * kPackRows);
                            } else {
                                tma_load_3d(dst, &tmG, full, kb * BK, c * kChunk, e);
                                tma_load_3d(dst + kStageBytes / 2, &tmU, full, kb * BK,
                                            c * kChunk, e);
                            }
                        }
                        if (!ok) break;
                    }
                    if (c >= 1) {
                        // down k-blocks 2(c-1) and 2(c-1)+1 (only the first when I ends there)
                        for (int kd = 2 * (c - 1); kd < 2 * c && kd < KBD; ++kd) {
                            uint32_t dst, full;
                            if (!next((uint32_t)NY * BK * 2, dst, full)) {
                                ok = false;
                                break;
                            }
                            if (b_packed)  // H <= 256: one n-block, block (e, 0, kd)
                                tma_load_2d(dst, &tmD, full, 0, (e * KBD + kd) * kPackRows);
                            else
                                tma_load_3d(dst, &tmD, full, kd * BK, 0, e);
                        }
                    }
                }
            }
            if (*abort_flag) {
                for (int s = 0; s < n_stages; ++s)
                    if ((armed >> s) & 1u)
                        wait_bar_drain(smem_u32(&ctl->full[s]), (armed_parity >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_gu = make_idesc(BM, kGuN);
            const uint32_t idesc_y = make_idesc(BM, NY);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t cpar = 0;  // parity of this CTA's chunk count over all its tiles
            uint32_t tpar = 0;  // parity of this CTA's tile count
            bool ok = true;
            // the next ring stage once TMA has filled it (0 if the wait gave up);
            // the MMAs read it through the async proxy that wrote it, ordered by
            // the stage's mbarrier
            auto take = [&]() -> uint32_t {
                if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, err)) return 0;
                return ring_addr + (uint32_t)stage * (uint32_t)kStageBytes;
            };
            auto release = [&]() {
                umma_commit(smem_u32(&ctl->empty[stage]));
                if (++stage == n_stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                if (!wait_bar(smem_u32(&ctl->x_full), tpar, abort_flag, err)) break;
                tc_fence_after();
                fence_async_shared();  // x rows came through cp.async (generic proxy)
                for (int c = 0; ok && c <= NC; ++c) {
                    // here cpar is the parity of chunk c (flipped after each gate/up)
                    if (c < NC) {
                        // the epilogue has read chunk c-1's accumulator out of TMEM
                        if (!wait_bar(smem_u32(&ctl->a_empty), cpar ^ 1u, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        for (int kb = 0; kb < KBX; ++kb) {
                            const uint32_t b_s = take();
                            if (!b_s) {
                                ok = false;
                                break;
                            }
                            const uint64_t ad = sw128_desc(x_addr + (uint32_t)kb * kTileBytes);
                            const uint64_t bd = sw128_desc(b_s);
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk)
                                umma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                          idesc_gu, (kb | kk) != 0 ? 1u : 0u);
                            release();
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&ctl->a_full));
                        if (c == NC - 1) umma_commit(smem_u32(&ctl->x_empty));
                    }
                    if (c >= 1) {
                        const int d = c - 1;
                        if (d == 0) {
                            // the previous tile's y has been read out of TMEM
                            if (!wait_bar(smem_u32(&ctl->y_empty), tpar ^ 1u, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                        }
                        // h of chunk d (parity: one chunk before c)
                        if (!wait_bar(smem_u32(&ctl->h_full), cpar ^ 1u, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        fence_async_shared();  // h was written by the epilogue (generic proxy)
                        for (int kd = 2 * d; kd < 2 * d + 2 && kd < KBD; ++kd) {
                            const uint32_t b_s = take();
                            if (!b_s) {
                                ok = false;
                                break;
                            }
                            const uint64_t ad =
                                sw128_desc(h_addr + (uint32_t)(kd - 2 * d) * kTileBytes);
                            const uint64_t bd = sw128_desc(b_s);
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk)
                                umma_bf16(tmem + kYCol, ad + (uint64_t)(kk * 2),
                                          bd + (uint64_t)(kk * 2), idesc_y,
                                          (kd | kk) != 0 ? 1u : 0u);
                            release();
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&ctl->h_empty));
                    }
                    if (c < NC) cpar ^= 1u;
                }
                if (!ok) break;
                umma_commit(smem_u32(&ctl->y_full));
                tpar ^= 1u;
            }
            umma_commit(smem_u32(&ctl->done));
            wait_bar_drain(smem_u32(&ctl->done), 0);
        }
    } else if (warp < 2 + kEpilogueWarps) {
        // ---------------- epilogue: g|u -> h (shared), y -> HBM ----------------
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;        // which 64 of a chunk's 128 columns
        const int r = q * 32 + lane;             // this lane's tile row
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        // this warp's half of the h tile is k-block `half` of the down MMA's A
        uint8_t* hrow = h_ptr + (size_t)half * kTileBytes + (size_t)r * 128;
        uint32_t cpar = 0, tpar = 0;
        bool ok = true;
        // lane 0 waits, the warp follows
        auto wait_warp = [&](uint32_t bar, uint32_t par) -> bool {
            int v = 0;
            if (lane == 0) v = wait_bar(bar, par, abort_flag, err);
            return __shfl_sync(0xffffffffu, v, 0) != 0;
        };
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            int e, mb, nb;
            decode_tile(ctl->prefix, E, 1, BM, NY, tile, e, mb, nb);
            const bool row_ok = mb * BM + r < expert_counts[e];
            const long long row = (long long)expert_offsets[e] + mb * BM + r;  // output row
            for (int c = 0; c < NC; ++c) {
                if (!wait_warp(smem_u32(&ctl->a_full), cpar)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t g0[32], g1[32], u0[32], u1[32];
                const uint32_t col = (uint32_t)(half * 64);
                tmem_ld32(lane_base + col, g0);
                tmem_ld32(lane_base + col + 32, g1);
                tmem_ld32(lane_base + kChunk + col, u0);
                tmem_ld32(lane_base + kChunk + col + 32, u1);
                tmem_wait_ld();
                // the accumulator is free for the next chunk once read
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->a_empty));
                uint4 hv[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) hv[j] = swiglu8(g0 + 8 * j, u0 + 8 * j);
#pragma unroll
                for (int j = 0; j < 4; ++j) hv[4 + j] = swiglu8(g1 + 8 * j, u1 + 8 * j);
                // the h tile is free once the down MMA of chunk c - 1 is done
                if (!wait_warp(smem_u32(&ctl->h_empty), cpar ^ 1u)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(hrow + ((j ^ (r & 7)) << 4)) = hv[j];
                fence_async_shared();  // seen by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->h_full));
                cpar ^= 1u;
            }
            if (!ok) break;
            if (!wait_warp(smem_u32(&ctl->y_full), tpar)) break;
            tc_fence_after();
            // y: this lane's row, 64 columns per slice, the two warps of a
            // quadrant taking alternate slices
#pragma unroll 1
            for (int s = half; s * 64 < NY; s += 2) {
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + kYCol + (uint32_t)(s * 64), v0);
                tmem_ld32(lane_base + kYCol + (uint32_t)(s * 64 + 32), v1);
                tmem_wait_ld();
                if (row_ok) {
                    __nv_bfloat16* yrow = y + row * H;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int cc = s * 64 + j * 8;  // H % 8 == 0: 8 columns in or out
                        if (cc < H) {
                            const uint32_t* v = j < 4 ? v0 + 8 * j : v1 + 8 * (j - 4);
                            uint4 o;
                            o.x = pack2(__uint_as_float(v[0]), __uint_as_float(v[1]));
                            o.y = pack2(__uint_as_float(v[2]), __uint_as_float(v[3]));
                            o.z = pack2(__uint_as_float(v[4]), __uint_as_float(v[5]));
                            o.w = pack2(__uint_as_float(v[6]), __uint_as_float(v[7]));
                            *reinterpret_cast<uint4*>(yrow + cc) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->y_empty));
            tpar ^= 1u;
        }
    } else {
        // ---------------- gather warps: the tile's x rows by cp.async ----------------
        // Instruction i covers rows 8i + 4g .. 8i + 4g + 3 (g = gather warp);
        // 8 lanes copy the 8 16-byte chunks of one row's 128-byte k-block.
        const int gw = warp - 2 - kEpilogueWarps;
        const int chunk = lane & 7;
        const int rsub = gw * 4 + (lane >> 3);
        uint32_t tpar = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int e, mb, nb;
            decode_tile(ctl->prefix, E, 1, BM, NY, tile, e, mb, nb);
            const int row0 = expert_offsets[e] + mb * BM;
            // the previous tile's gate/up MMAs are done with the x tile
            int go = 1;
            if (lane == 0) go = wait_bar(smem_u32(&ctl->x_empty), tpar ^ 1u, abort_flag, err);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
#pragma unroll 1
            for (int i = 0; i < BM / 8; ++i) {
                const int rr = i * 8 + rsub;
                int v = row0 + rr < a_total ? (a_rows ? a_rows[row0 + rr] : row0 + rr) : 0;
                v = (unsigned)v < (unsigned)a_src_rows ? v : 0;
                const uint16_t* src = a_src + (size_t)v * H;
                for (int kb = 0; kb < KBX; ++kb) {
                    const int colx = kb * BK + chunk * 8;
                    const bool in = colx < H;  // H % 8 == 0: a chunk is wholly in or out
                    cp_async_16(x_addr + (uint32_t)kb * kTileBytes + rr * 128 +
                                    ((chunk ^ (rr & 7)) << 4),
                                src + (in ? colx : 0), in ? 16u : 0u);
                }
            }
            cp_async_arrive_noinc(smem_u32(&ctl->x_full));
            tpar ^= 1u;
        }
        cp_async_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

moe_status launch_ffn_fused_wide(const uint16_t* src, const int32_t* row_index, long long src_rows,
                            const GemmGroup& g, int H, int I, const uint16_t* wg,
                            const uint16_t* wu, const uint16_t* wd, uint16_t* y,
                            cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    const SmemPlan plan = smem_plan(H);
    if (H <= 0 || H > kFusedMaxH || plan.stages < 2) return MOE_ERR_UNSUPPORTED;
    const int NY = y_cols(H);
    CUtensorMap mg, mu, md, unused;
    bool ok_b;
    if (g.packed)
        ok_b = map_packed(&mg, &mu, wg, g.E, (I + 127) / 128, H, kPackRows) &&
               map_packed(&md, &unused, wd, g.E, 1, I, (uint32_t)NY);
    else
        ok_b = map_3d(&mg, wg, g.E, I, H, kChunk) && map_3d(&mu, wu, g.E, I, H, kChunk) &&
               map_3d(&md, wd, g.E, H, I, (uint32_t)NY);
    if (!ok_b) return MOE_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fused_ffn_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)plan.bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
    // tiles <= ceil(R / 128) + E (each expert adds at most one ragged m-block)
    const long long tiles = (g.R + BM - 1) / BM + g.E;
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    fused_ffn_wide_kernel<<<grid, kThreads, plan.bytes, st>>>(
        mg, mu, md, g.offsets, g.counts, g.E, H, I, reinterpret_cast<__nv_bfloat16*>(y), g.err,
        row_index, (int)g.R, (int)src_rows, src, g.packed ? 1 : 0, plan.stages);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
