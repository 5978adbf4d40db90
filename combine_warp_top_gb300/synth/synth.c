/*
 * Seeded synthetic inputs for the MoE layer: counter-based SplitMix64 uniforms
 * and Box-Muller normals, rounded to fp32 or bf16.
 *
 * This file holds no arithmetic of the MoE method itself. It is shared by the
 * CPU oracle's tests and by the CUDA path's harness so that both see the very
 * same input bits.
 *
 * Generator definition (SplitMix64, Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *   GAMMA = 0x9E3779B97F4A7C15
 *   mix(z): z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *           z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *           return z ^ (z >> 31)
 *   stream start  s0 = mix(mix(seed) ^ (stream * 0xD1B54A32D192ED03 + 1))
 *   i-th draw     x_i = mix(s0 + (i + 1) * GAMMA)        (counter based)
 *   uniform       u_i = ((x_i >> 11) + 0.5) * 2^-53      in (0, 1)
 * Box-Muller (Box and Muller, 1958), element i of a normal stream uses the
 * pair p = i / 2:  r = sqrt(-2 ln u_{2p}),  a = 2 pi u_{2p+1},
 *                  n_i = r cos a (i even)  or  r sin a (i odd).
 * A value mean + std * n_i is formed in double, rounded to fp32 (round to
 * nearest even), and for bf16 rounded again from fp32 to bf16 (round to
 * nearest even on the bit pattern).
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_start(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed) ^ (stream * 0xD1B54A32D192ED03ULL + 1ULL));
}

static inline uint64_t draw(uint64_t s0, uint64_t i) {
    return mix64(s0 + (i + 1ULL) * GAMMA);
}

static inline double to_unit(uint64_t x) {
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t s0, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t p = i >> 1;
    double u1 = to_unit(draw(s0, 2 * p));
    double u2 = to_unit(draw(s0, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = two_pi * u2;
    return (i & 1ULL) ? r * sin(a) : r * cos(a);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t u = v.u;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
    uint64_t s0 = stream_start(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = draw(s0, offset + (uint64_t)i);
}

void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double* out) {
    uint64_t s0 = stream_start(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = to_unit(draw(s0, offset + (uint64_t)i));
}

void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean,
                      double stdev, double* out) {
    uint64_t s0 = stream_start(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = mean + stdev * normal_at(s0, offset + (uint64_t)i);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean,
                      double stdev, float* out) {
    uint64_t s0 = stream_start(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(mean + stdev * normal_at(s0, offset + (uint64_t)i));
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean,
                       double stdev, uint16_t* out) {
    uint64_t s0 = stream_start(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)(mean + stdev * normal_at(s0, offset + (uint64_t)i)));
}

int synth_threads(void) {
    int t = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        t = omp_get_num_threads();
    }
#endif
    return t;
}
