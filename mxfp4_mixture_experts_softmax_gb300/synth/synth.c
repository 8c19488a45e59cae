/*
 * Seeded synthetic inputs for the MXFP4 MoE layer.
 *
 * This file only draws random numbers: it holds none of the layer's
 * arithmetic (no routing, no MXFP4 decoding, no GEMM).  Both the GPU path and
 * the CPU oracle consume the bytes it writes, so the two always see identical
 * inputs.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used as a counter-based stream:
 *     base(seed, stream) = mix(seed * G + stream + 1)
 *     u64(seed, stream, i) = mix(base + (i + 1) * G),   G = 0x9E3779B97F4A7C15
 * where mix() is the SplitMix64 output function.  Element i of every stream
 * depends only on (seed, stream, i), so any slice can be regenerated alone and
 * the fill parallelises trivially.
 *
 * Normal variates use the Box-Muller transform on two 53-bit uniforms
 * (cosine branch only).  bf16 values are the fp32 normal rounded to nearest
 * even.
 */
#include <math.h>
#include <stdint.h>

#define SYNTH_G 0x9E3779B97F4A7C15ULL

static inline uint64_t synth_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t synth_base(uint64_t seed, uint64_t stream) {
    return synth_mix(seed * SYNTH_G + stream + 1ULL);
}

static inline uint64_t synth_at(uint64_t base, uint64_t i) {
    return synth_mix(base + (i + 1ULL) * SYNTH_G);
}

/* 53-bit uniform in [0, 1). */
static inline double synth_unit(uint64_t u) { return (double)(u >> 11) * 0x1.0p-53; }

static inline double synth_normal_at(uint64_t base, uint64_t i) {
    double u1 = 1.0 - synth_unit(synth_at(base, 2 * i)); /* (0, 1] */
    double u2 = synth_unit(synth_at(base, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs only). */
static inline uint16_t synth_to_bf16(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

void synth_u64(uint64_t seed, uint64_t stream, int64_t n, uint64_t* out) {
    uint64_t b = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = synth_at(b, (uint64_t)i);
}

/* Uniform bytes: byte j is byte (j mod 8) of u64(j / 8). */
void synth_bytes(uint64_t seed, uint64_t stream, int64_t n, uint8_t* out) {
    uint64_t b = synth_base(seed, stream);
    int64_t nw = n / 8;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nw; ++i) {
        uint64_t u = synth_at(b, (uint64_t)i);
        for (int k = 0; k < 8; ++k) out[8 * i + k] = (uint8_t)(u >> (8 * k));
    }
    if (nw * 8 < n) {
        uint64_t u = synth_at(b, (uint64_t)nw);
        for (int64_t j = nw * 8; j < n; ++j) out[j] = (uint8_t)(u >> (8 * (j - nw * 8)));
    }
}

/* Integers uniform in [lo, hi] (inclusive), one per u64, by multiply-shift. */
void synth_int_bytes(uint64_t seed, uint64_t stream, int64_t n, int lo, int hi, uint8_t* out) {
    uint64_t b = synth_base(seed, stream);
    uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t u = synth_at(b, (uint64_t)i) >> 32;
        out[i] = (uint8_t)(lo + (int)((u * span) >> 32));
    }
}

void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, float* out) {
    uint64_t b = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)synth_normal_at(b, (uint64_t)i);
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, uint16_t* out) {
    uint64_t b = synth_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = synth_to_bf16((float)synth_normal_at(b, (uint64_t)i));
}
