// Device-side twin of synth.c's normal_bf16 stream, used only to fill the
// large expert-weight tensors in device memory quickly.  Same counter-based
// SplitMix64 draws and Box-Muller transform as synth.c, evaluated in double
// precision with CUDA's own log/sqrt/sin/cos; a value can differ from the host
// generator only where the two libraries round the transcendental differently
// right at a bf16 rounding boundary.  Holds no arithmetic of the MoE method.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t mix64_h(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__device__ __forceinline__ double to_unit(uint64_t x) {
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// Each thread produces one Box-Muller pair (elements 2p and 2p+1).
__global__ void normal_bf16_kernel(uint64_t s0, uint64_t offset, int64_t n, double mean,
                                   double stdev, uint16_t* __restrict__ out) {
    const double two_pi = 6.283185307179586476925286766559;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // element range [first, first + n) of the stream; pairs p cover it
    const uint64_t first = offset;
    const uint64_t p0 = first >> 1;
    const uint64_t p1 = (first + (uint64_t)n + 1) >> 1;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; (uint64_t)i < p1 - p0;
         i += stride) {
        const uint64_t p = p0 + (uint64_t)i;
        const double u1 = to_unit(mix64(s0 + (2 * p + 1) * 0x9E3779B97F4A7C15ULL));
        const double u2 = to_unit(mix64(s0 + (2 * p + 2) * 0x9E3779B97F4A7C15ULL));
        const double r = sqrt(-2.0 * log(u1));
        double sn, cs;
        sincos(two_pi * u2, &sn, &cs);
        const uint64_t e0 = 2 * p, e1 = 2 * p + 1;
        if (e0 >= first && e0 < first + (uint64_t)n)
            out[e0 - first] = f32_to_bf16_rne((float)(mean + stdev * (r * cs)));
        if (e1 >= first && e1 < first + (uint64_t)n)
            out[e1 - first] = f32_to_bf16_rne((float)(mean + stdev * (r * sn)));
    }
}

}  // namespace

extern "C" int synth_normal_bf16_device(uint64_t seed, uint64_t stream, uint64_t offset,
                                        int64_t n, double mean, double stdev, uint16_t* out,
                                        void* cuda_stream) {
    if (n <= 0) return 0;
    const uint64_t s0 = mix64_h(mix64_h(seed) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
    const int threads = 256;
    const long long pairs = (n + 2) / 2;
    long long blocks = (pairs + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;
    normal_bf16_kernel<<<(int)blocks, threads, 0, (cudaStream_t)cuda_stream>>>(s0, offset, n, mean,
                                                                              stdev, out);
    return (int)cudaGetLastError();
}
