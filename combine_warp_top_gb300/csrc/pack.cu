// Expert weights in the packed layout the grouped GEMMs stream (moe_pack_weights).
//
// The gated MLP of FarSkip-Collective (arXiv 2511.11505) Sec. 2.1 reads each
// expert's weight matrices once per step; in nn.Linear layout one 64-deep
// k-slice of a 256-row weight tile is 256 pieces of 128 bytes, 2H or 2I bytes
// apart, and a layer that streams its weights from HBM reads them at the DRAM's
// strided rate.  Packed, each such slice is one contiguous 32 KB block, which
// the GEMMs load with a single TMA box of a [rows, 64] map.
//
// One thread per 16-byte chunk (8 bf16) of the output, in output order, so the
// writes are coalesced and eight consecutive threads read one 128-byte row
// piece of the source.  H and I are multiples of 8, so a chunk lies wholly
// inside or wholly outside the source matrix (outside: zeros).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;

// kGateUp: block row r < 128 comes from a (gate), r >= 128 from b (up), both
// [E, n_src, K] with 128-column n-blocks; otherwise a only, 256-row n-blocks.
template <bool kGateUp>
__global__ void __launch_bounds__(kThreads) pack_kernel(const uint4* __restrict__ a,
                                                        const uint4* __restrict__ b, int n_src,
                                                        int K, int NB, int KB, long long chunks,
                                                        uint4* __restrict__ out) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < chunks;
         i += (long long)gridDim.x * blockDim.x) {
        const int c8 = (int)(i & 7);
        const long long row = i >> 3;
        const int r = (int)(row % kPackRows);
        const long long blk = row / kPackRows;
        const int kb = (int)(blk % KB);
        const long long rest = blk / KB;
        const int nb = (int)(rest % NB);
        const long long e = rest / NB;
        const int n = kGateUp ? nb * 128 + (r & 127) : nb * kPackRows + r;
        const int col = kb * 64 + c8 * 8;
        const uint4* src = (kGateUp && r >= 128) ? b : a;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < n_src && col < K) v = src[((e * n_src + n) * K + col) >> 3];
        out[i] = v;
    }
}

template <bool kGateUp>
cudaError_t pack(const uint16_t* a, const uint16_t* b, int E, int n_src, int K, int NB,
                 uint16_t* out, cudaStream_t st) {
    const long long chunks = packed_rows(E, NB, K) * 8;
    if (chunks == 0) return cudaSuccess;
    long long blocks = (chunks + kThreads - 1) / kThreads;
    const long long cap = (long long)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    pack_kernel<kGateUp><<<(int)blocks, kThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(a), reinterpret_cast<const uint4*>(b), n_src, K, NB,
        (K + 63) / 64, chunks, reinterpret_cast<uint4*>(out));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pack(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                        const moe_shape& s, uint16_t* gate_up, uint16_t* down, cudaStream_t st) {
    if (gate_up) {
        const cudaError_t e = pack<true>(wg, wu, s.E, s.I, s.H, (s.I + 127) / 128, gate_up, st);
        if (e != cudaSuccess) return e;
    }
    if (down) return pack<false>(wd, nullptr, s.E, s.H, s.I, (s.H + 255) / 256, down, st);
    return cudaSuccess;
}

}  // namespace moe
