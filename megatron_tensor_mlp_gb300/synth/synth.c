/*
 * Seeded synthetic inputs for the tensor-parallel MLP (shared by the oracle
 * tests, the GPU parity tests and the benchmark).
 *
 * This file holds no arithmetic of the MLP itself: it only draws normal
 * variates and stores them in the storage type of the tensors (fp32 or bf16).
 *
 * Generator (counter based, so every element can be produced independently
 * and the result does not depend on the thread count):
 *   mix64(z)       = the SplitMix64 output function (Steele, Lea & Flood,
 *                    "Fast splittable pseudorandom number generators",
 *                    OOPSLA 2014; constants as in Vigna's public-domain
 *                    splitmix64.c)
 *   key(seed, s)   = mix64(seed * 2^8 + s)            (s = tensor stream id)
 *   word(c)        = mix64(key + (c + 1) * 0x9E3779B97F4A7C15)
 *   u1(i)          = ((word(2i) >> 11) + 1) * 2^-53    in (0, 1]
 *   u2(i)          = (word(2i+1) >> 11) * 2^-53        in [0, 1)
 *   n(i)           = sqrt(-2 ln u1) * cos(2 pi u2)     (Box-Muller, cosine branch)
 *   x(i)           = sigma * n(i)  in double, rounded to fp32 (round to nearest
 *                    even), and for bf16 tensors the fp32 value is rounded to
 *                    bf16 (round to nearest even on the upper 16 bits).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const uint64_t gamma = 0x9E3779B97F4A7C15ULL;
    uint64_t w1 = mix64(key + (2 * i + 1) * gamma);
    uint64_t w2 = mix64(key + (2 * i + 2) * gamma);
    double u1 = (double)((w1 >> 11) + 1) * 0x1.0p-53;
    double u2 = (double)(w2 >> 11) * 0x1.0p-53;
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    /* inputs are finite normals: no NaN/Inf handling needed */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * 256ULL + stream);
}

/* out[i] = fp32(sigma * n(offset + i)), i in [0, n) */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double sigma, float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(sigma * normal_at(key, offset + (uint64_t)i));
}

/* out[i] = bf16(fp32(sigma * n(offset + i))) as raw 16-bit patterns */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double sigma, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne((float)(sigma * normal_at(key, offset + (uint64_t)i)));
}

/* exact widening of bf16 patterns to fp64 (used to hand identical values to the oracle) */
void synth_bf16_to_f64(const uint16_t* in, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = (uint32_t)in[i] << 16;
        float f;
        memcpy(&f, &u, 4);
        out[i] = (double)f;
    }
}
