// The expert FFN in one kernel with h kept on chip: gate/up, SwiGLU and down
// for a 128-row tile of an expert's rows, without writing h to HBM.
//
// "Kernel fusion for expert parallelism", section "Fusing the layer into one
// kernel": the MegaKernel keeps each expert's intermediate activations in the
// SM's local memory between the two MatMuls instead of a round trip through
// device memory.  FarSkip-Collective (arXiv 2511.11505) Sec. 2.1: the gated
// expert MLP h = SiLU(x Wg^T) * (x Wu^T), y = h Wd^T.
//
// On one SM this works when a whole output row of the tile stays in TMEM: y
// for 128 rows and H columns takes H of the 512 fp32 TMEM columns, next to two
// 128-column gate/up accumulators, so H <= 256.  I is then free: h is made 64
// columns at a time (one 128-byte k-block of the down MatMul's A operand) and
// consumed by the down MMA right away, so only two 16 KB h buffers exist.
//
// Per tile (persistent CTAs, tiles = 128-row m-blocks of each expert):
//   x tile   [128, H] bf16 gathered once into shared memory (swizzled k-blocks)
//   chunk c  g|u[128, 128] = x Wg|Wu[e][64c..64c+63, :]^T   (TMEM buffer c & 1)
//            h_c = bf16(SiLU(g) * u)  -> shared h buffer c & 1 (swizzled)
//            y[128, H] += h_c Wd[e][:, 64c..64c+63]^T        (TMEM, fp32)
//   y        bf16 -> HBM (TMA store; masked row lines at a segment's end)
// The MMA thread issues gate/up(c+1) before down(c), so the tensor pipe runs
// the next chunk while the epilogue warps turn chunk c into h.  The fp32
// accumulation orders are those of the two-kernel path (k-blocks of x for g
// and u, 64-column k-blocks of h for y, 16-deep MMAs in order), and h is
// rounded to bf16 the same way.
//
// This 64-column form runs for I < 1024; from I = 1024 on the wide form of
// fused_ffn_wide.cu (128-column chunks, N = 256 gate/up MMAs) takes over,
// whose stages are long enough that the one MMA-issuing thread keeps up.
//
// Roles (320 threads): warp 0 TMA-loads weight k-blocks into a ring (gate and
// up halves of 64 rows, or the down k-block of round_up(H, 32) rows); warp 1
// owns TMEM and issues tcgen05.mma; warps 2-5 turn g|u into h and drain y;
// warps 6-9 gather the x rows with 16-byte cp.async.  Every wait is bounded;
// a wait that runs out records MOE_ERR_TIMEOUT and the CTA drains and returns.
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = kGemmBM;        // rows per tile (TMEM lanes)
constexpr int BK = 64;             // bf16 per k-block: one 128-byte swizzle row
constexpr int UMMA_K = 16;
constexpr int kChunk = 64;         // columns of I per chunk
constexpr int kGuN = 2 * kChunk;   // gate/up MMA N: 64 gate + 64 up columns
constexpr int kMaxStages = 6;
constexpr int kEpilogueWarps = 4;
constexpr int kGatherWarps = 4;
constexpr int kGatherThreads = kGatherWarps * 32;
constexpr int kThreads = (2 + kEpilogueWarps + kGatherWarps) * 32;
constexpr int kTileBytes = BM * BK * 2;  // 16 KB: 128 rows x one k-block (x or h)
constexpr int kGuBytes = kGuN * BK * 2;  // 16 KB: a gate/up weight k-block
constexpr int kStageCols = 64;
constexpr int kStageWarpBytes = 32 * kStageCols * 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kYCol = 2 * kGuN;     // y accumulator: TMEM columns 256..511
constexpr int kSmemLimit = 227 * 1024;

struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t x_full, x_empty;  // x tile gathered / read by the last gate/up MMA
    uint64_t a_full[2], a_empty[2];  // gate/up accumulators
    uint64_t h_full[2], h_empty[2];  // h buffers
    uint64_t y_full, y_empty;        // y accumulator
    uint64_t done;
    uint32_t tmem_base;
    int abort;
    int prefix[kMaxE + 1];
    int offs[kMaxE];
    int cnts[kMaxE];
};
constexpr size_t kCtlBytes = (sizeof(Ctl) + 15) & ~size_t(15);

// Shared memory after the 1024-byte alignment: x tile, two h buffers, the
// weight ring, the y staging tiles, Ctl.
struct SmemPlan {
    int kbx;          // k-blocks of x (ceil(H / 64))
    int stage_bytes;  // max(16 KB, round_up(H, 32) rows x 128 B)
    int stages;
    size_t bytes;
};

__host__ __device__ inline int y_cols(int H) { return (H + 31) / 32 * 32; }

SmemPlan smem_plan(int H) {
    SmemPlan p;
    p.kbx = (H + BK - 1) / BK;
    const int yb = y_cols(H) * BK * 2;
    p.stage_bytes = yb > kGuBytes ? yb : kGuBytes;
    const size_t fixed = 1024 + (size_t)p.kbx * kTileBytes + 2 * (size_t)kTileBytes +
                         (size_t)kEpilogueWarps * kStageWarpBytes + kCtlBytes;
    long long st = ((long long)kSmemLimit - (long long)fixed) / p.stage_bytes;
    if (st > kMaxStages) st = kMaxStages;
    p.stages = (int)st;
    p.bytes = fixed + (size_t)p.stages * p.stage_bytes;
    return p;
}

// a_rows == nullptr: tile row i is row i of a_src.  Otherwise row a_rows[i]
// (rows >= a_total and indices outside [0, a_src_rows) read row 0; such rows
// are masked on store).
__global__ void __launch_bounds__(kThreads, 1)
    fused_ffn_kernel(const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmU,
                     const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmY,
                     const int32_t* __restrict__ expert_offsets,
                     const int32_t* __restrict__ expert_counts, int E, int H, int I,
                     __nv_bfloat16* __restrict__ y, int* err,
                     const int32_t* __restrict__ a_rows, int a_total, int a_src_rows,
                     const uint16_t* __restrict__ a_src, int b_packed, int n_stages,
                     int stage_bytes) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int KBX = (H + BK - 1) / BK;
    const int NC = (I + kChunk - 1) / kChunk;
    const int NY = y_cols(H);
    const uint32_t x_addr = smem_u32(base);
    const uint32_t h_addr = x_addr + (uint32_t)KBX * kTileBytes;
    uint8_t* h_ptr = base + (size_t)KBX * kTileBytes;
    const uint32_t ring_addr = h_addr + 2u * kTileBytes;
    uint8_t* stage_area = h_ptr + 2 * kTileBytes + (size_t)n_stages * stage_bytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(stage_area + (size_t)kEpilogueWarps * kStageWarpBytes);
    volatile int* abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        ctl->offs[i] = expert_offsets[i];
        ctl->cnts[i] = expert_counts[i];
    }
    __syncthreads();
    if (warp == 2) warp_mblk_prefix(ctl->cnts, E, BM, ctl->prefix);
    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        mbar_init(smem_u32(&ctl->x_full), kGatherThreads);
        mbar_init(smem_u32(&ctl->x_empty), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->a_full[b]), 1);
            mbar_init(smem_u32(&ctl->a_empty[b]), kEpilogueWarps);
            mbar_init(smem_u32(&ctl->h_full[b]), kEpilogueWarps);
            mbar_init(smem_u32(&ctl->h_empty[b]), 1);
        }
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
        prefetch_map(&tmY);
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
            const int NBg = (I + 127) / 128;  // packed gate/up: 256-row blocks of 128 + 128
            // the next ring stage: wait until it is free, arm it for `bytes`
            auto next = [&](uint32_t bytes, uint32_t& dst, uint32_t& full) -> bool {
                if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, err))
                    return false;
                full = smem_u32(&ctl->full[stage]);
                dst = ring_addr + (uint32_t)stage * (uint32_t)stage_bytes;
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
                            if (!next(kGuBytes, dst, full)) {
                                ok = false;
                                break;
                            }
                            if (b_packed) {
                                // block (e, c / 2, kb): gate rows 0..127, up rows 128..255
                                const int blk = ((e * NBg + (c >> 1)) * KBX + kb) * kPackRows +
                                                (c & 1) * kChunk;
                                tma_load_2d(dst, &tmG, full, 0, blk);
                                tma_load_2d(dst + kGuBytes / 2, &tmG, full, 0, blk + 128);
                            } else {
                                tma_load_3d(dst, &tmG, full, kb * BK, c * kChunk, e);
                                tma_load_3d(dst + kGuBytes / 2, &tmU, full, kb * BK, c * kChunk, e);
                            }
                        }
                        if (!ok) break;
                    }
                    if (c >= 1) {
                        const int d = c - 1;
                        uint32_t dst, full;
                        if (!next((uint32_t)NY * BK * 2, dst, full)) {
                            ok = false;
                            break;
                        }
                        if (b_packed)  // H <= 256: one n-block, block (e, 0, d)
                            tma_load_2d(dst, &tmD, full, 0, (e * NC + d) * kPackRows);
                        else
                            tma_load_3d(dst, &tmD, full, d * kChunk, 0, e);
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
            long long gc = 0;  // chunks begun by this CTA over all its tiles
            uint32_t tpar = 0;  // parity of this CTA's tile count
            bool ok = true;
            auto take = [&](uint32_t& s_addr) -> bool {
                if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, err)) return false;
                tc_fence_after();
                s_addr = ring_addr + (uint32_t)stage * (uint32_t)stage_bytes;
                return true;
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
                    if (c < NC) {
                        const long long g = gc + c;
                        const int ab = (int)(g & 1);
                        const uint32_t aph = (uint32_t)(g >> 1) & 1u;
                        if (!wait_bar(smem_u32(&ctl->a_empty[ab]), aph ^ 1u, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t dacc = tmem + (uint32_t)(ab * kGuN);
                        for (int kb = 0; kb < KBX; ++kb) {
                            uint32_t b_s;
                            if (!take(b_s)) {
                                ok = false;
                                break;
                            }
                            const uint64_t ad = sw128_desc(x_addr + (uint32_t)kb * kTileBytes);
                            const uint64_t bd = sw128_desc(b_s);
#pragma unroll
                            for (int kk = 0; kk < BK / UMMA_K; ++kk)
                                umma_bf16(dacc, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                          idesc_gu, (kb | kk) != 0 ? 1u : 0u);
                            release();
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(&ctl->a_full[ab]));
                        if (c == NC - 1) umma_commit(smem_u32(&ctl->x_empty));
                    }
                    if (c >= 1) {
                        const int d = c - 1;
                        const long long g = gc + d;
                        const int hb = (int)(g & 1);
                        const uint32_t hph = (uint32_t)(g >> 1) & 1u;
                        if (d == 0) {
                            // the previous tile's y has been read out of TMEM
                            if (!wait_bar(smem_u32(&ctl->y_empty), tpar ^ 1u, abort_flag, err)) {
                                ok = false;
                                break;
                            }
                        }
                        if (!wait_bar(smem_u32(&ctl->h_full[hb]), hph, abort_flag, err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        fence_async_shared();
                        uint32_t b_s;
                        if (!take(b_s)) {
                            ok = false;
                            break;
                        }
                        const uint64_t ad = sw128_desc(h_addr + (uint32_t)hb * kTileBytes);
                        const uint64_t bd = sw128_desc(b_s);
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk)
                            umma_bf16(tmem + kYCol, ad + (uint64_t)(kk * 2),
                                      bd + (uint64_t)(kk * 2), idesc_y, (d | kk) != 0 ? 1u : 0u);
                        release();
                        umma_commit(smem_u32(&ctl->h_empty[hb]));
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&ctl->y_full));
                gc += NC;
                tpar ^= 1u;
            }
            umma_commit(smem_u32(&ctl->done));
            wait_bar_drain(smem_u32(&ctl->done), 0);
        }
    } else if (warp < 2 + kEpilogueWarps) {
        // ---------------- epilogue: g|u -> h (shared), y -> HBM ----------------
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;  // this lane's tile row
        uint8_t* stage = stage_area + (size_t)(warp - 2) * kStageWarpBytes;
        const uint32_t stage_addr = smem_u32(stage);
        uint8_t* my_row = stage + lane * 128;
        const int sw = lane & 7;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        long long gc = 0;
        uint32_t tpar = 0;
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
            const int row_base = ctl->offs[e] + mb * BM + q * 32;
            int rows_valid = ctl->offs[e] + ctl->cnts[e] - row_base;
            rows_valid = rows_valid < 0 ? 0 : (rows_valid > 32 ? 32 : rows_valid);
            for (int c = 0; c < NC; ++c) {
                const long long g = gc + c;
                const int ab = (int)(g & 1);
                const uint32_t aph = (uint32_t)(g >> 1) & 1u;
                if (!wait_warp(smem_u32(&ctl->a_full[ab]), aph)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint4 hv[8];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t gv[32], uv[32];
                    const uint32_t col = (uint32_t)(ab * kGuN + half * 32);
                    tmem_ld32(lane_base + col, gv);
                    tmem_ld32(lane_base + col + kChunk, uv);
                    tmem_wait_ld();
#pragma unroll
                    for (int grp = 0; grp < 4; ++grp) {
                        uint32_t* op = reinterpret_cast<uint32_t*>(&hv[half * 4 + grp]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int j = grp * 8 + 2 * i;
                            const float h0 = silu(__uint_as_float(gv[j])) * __uint_as_float(uv[j]);
                            const float h1 =
                                silu(__uint_as_float(gv[j + 1])) * __uint_as_float(uv[j + 1]);
                            op[i] = pack2(h0, h1);
                        }
                    }
                }
                // the accumulator is free for chunk c + 2 once read
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->a_empty[ab]));
                // h buffer ab is free once the down MMA of chunk c - 2 is done
                if (!wait_warp(smem_u32(&ctl->h_empty[ab]), aph ^ 1u)) {
                    ok = false;
                    break;
                }
                uint8_t* hrow = h_ptr + (size_t)ab * kTileBytes + (size_t)r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(hrow + ((j ^ (r & 7)) << 4)) = hv[j];
                fence_async_shared();  // seen by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->h_full[ab]));
            }
            if (!ok) break;
            if (!wait_warp(smem_u32(&ctl->y_full), tpar)) break;
            tc_fence_after();
#pragma unroll 1
            for (int s = 0; s * kStageCols < NY; ++s) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + kYCol + (uint32_t)(s * kStageCols + half * 32), v);
                    tmem_wait_ld();
#pragma unroll
                    for (int grp = 0; grp < 4; ++grp) {
                        uint4 o;
                        uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int j = grp * 8 + 2 * i;
                            op[i] = pack2(__uint_as_float(v[j]), __uint_as_float(v[j + 1]));
                        }
                        *reinterpret_cast<uint4*>(my_row + (((half * 4 + grp) ^ sw) << 4)) = o;
                    }
                }
                const int col0 = s * kStageCols;
                if (rows_valid == 32) {
                    // columns past H are clipped by the tensor map
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, stage_addr, col0, row_base);
                        bulk_commit();
                    }
                } else {
                    __syncwarp();
                    const int qq = lane & 7;
                    const int col = col0 + qq * 8;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = i * 4 + (lane >> 3);
                        if (rr < rows_valid && col < H) {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                stage + rr * 128 + ((qq ^ (rr & 7)) << 4));
                            *reinterpret_cast<uint4*>(y + (size_t)(row_base + rr) * H + col) = v;
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->y_empty));
            gc += NC;
            tpar ^= 1u;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else {
        // ---------------- gather warps: the tile's x rows by cp.async ----------------
        // Instruction i covers rows 16i + 4g .. 16i + 4g + 3 (g = gather warp);
        // 8 lanes copy the 8 16-byte chunks of one row's 128-byte k-block.
        const int gw = warp - 2 - kEpilogueWarps;
        const int chunk = lane & 7;
        const int rsub = gw * 4 + (lane >> 3);
        uint32_t tpar = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int e, mb, nb;
            decode_tile(ctl->prefix, E, 1, BM, NY, tile, e, mb, nb);
            const int row0 = ctl->offs[e] + mb * BM;
            const uint16_t* src[BM / 16];
#pragma unroll
            for (int i = 0; i < BM / 16; ++i) {
                const int rr = row0 + i * 16 + rsub;
                int v = rr < a_total ? (a_rows ? a_rows[rr] : rr) : 0;
                v = (unsigned)v < (unsigned)a_src_rows ? v : 0;
                src[i] = a_src + (size_t)v * H;
            }
            // the previous tile's gate/up MMAs are done with the x tile
            int go = 1;
            if (lane == 0) go = wait_bar(smem_u32(&ctl->x_empty), tpar ^ 1u, abort_flag, err);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            for (int kb = 0; kb < KBX; ++kb) {
                const uint32_t xs = x_addr + (uint32_t)kb * kTileBytes;
                const int col = kb * BK + chunk * 8;
                const bool in = col < H;  // H % 8 == 0: a chunk is wholly in or out
#pragma unroll
                for (int i = 0; i < BM / 16; ++i) {
                    const int rr = i * 16 + rsub;
                    cp_async_16(xs + rr * 128 + ((chunk ^ (rr & 7)) << 4), src[i] + (in ? col : 0),
                                in ? 16u : 0u);
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

bool fused_ffn_supported(int H) { return H > 0 && H <= kFusedMaxH && smem_plan(H).stages >= 2; }

moe_status launch_ffn_fused(const uint16_t* src, const int32_t* row_index, long long src_rows,
                            const GemmGroup& g, int H, int I, const uint16_t* wg,
                            const uint16_t* wu, const uint16_t* wd, uint16_t* y,
                            cudaStream_t st) {
    if (g.R == 0) return MOE_OK;
    if (!fused_ffn_supported(H)) return MOE_ERR_UNSUPPORTED;
    // long I: 128-column chunks keep the tensor pipe ahead of the MMA thread
    if (I >= kFusedWideMinI)
        return launch_ffn_fused_wide(src, row_index, src_rows, g, H, I, wg, wu, wd, y, st);
    const SmemPlan plan = smem_plan(H);
    const int NY = y_cols(H);
    CUtensorMap mg, mu, md, my, unused;
    bool ok_b;
    if (g.packed)
        ok_b = map_packed(&mg, &mu, wg, g.E, (I + 127) / 128, H, kChunk) &&
               map_packed(&md, &unused, wd, g.E, 1, I, (uint32_t)NY);
    else
        ok_b = map_3d(&mg, wg, g.E, I, H, kChunk) && map_3d(&mu, wu, g.E, I, H, kChunk) &&
               map_3d(&md, wd, g.E, H, I, (uint32_t)NY);
    if (!ok_b || !map_2d(&my, y, g.R, H, 32)) return MOE_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(fused_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)plan.bytes) != cudaSuccess)
        return MOE_ERR_CUDA;
    // tiles <= ceil(R / 128) + E (each expert adds at most one ragged m-block)
    const long long tiles = (g.R + BM - 1) / BM + g.E;
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    fused_ffn_kernel<<<grid, kThreads, plan.bytes, st>>>(
        mg, mu, md, my, g.offsets, g.counts, g.E, H, I, reinterpret_cast<__nv_bfloat16*>(y),
        g.err, row_index, (int)g.R, (int)src_rows, src, g.packed ? 1 : 0, plan.stages,
        plan.stage_bytes);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
