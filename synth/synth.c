/*
 * Seeded synthetic inputs shared by the CUDA path's tests/bench and by the
 * CPU oracle.  This file draws random numbers only: it holds none of the
 * quantisation, packing or model arithmetic.
 *
 * Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), the RNG the cpp20gemma README names for
 * its reproducible sampler.  It is used counter-style: draw i of stream s
 * under seed S is mix(base(S, s) + (i + 1) * GOLDEN), which is exactly the
 * i-th output of a splitmix64 whose state starts at base(S, s).  That makes
 * every array order-independent, so OpenMP may fill it in parallel.
 *
 * Normals: Box-Muller on consecutive draw pairs (2j, 2j+1); element 2j takes
 * the cosine branch and 2j+1 the sine branch.  Computed in double and
 * rounded once to the output type.
 *
 * Built with -ffp-contract=off.  libm's log/cos/sin may differ in the last
 * double bit between hosts; no stored expected value depends on them.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Start state of stream `stream` under `seed`. */
static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
    return mix64(seed * GOLDEN + 0x632BE59BD9B4E019ULL) ^ mix64(stream + 0x1234567ULL);
}

static inline uint64_t draw(uint64_t base, uint64_t i) {
    return mix64(base + (i + 1) * GOLDEN);
}

/* uniform in [0, 1) with 53 random bits */
static inline double u01(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* The plain splitmix64 sequence x_1, x_2, ... for initial state `seed`. */
void synth_splitmix64_seq(uint64_t seed, int64_t n, uint64_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = draw(seed, (uint64_t)i);
}

static inline double normal_at(uint64_t base, int64_t i) {
    uint64_t j = (uint64_t)(i >> 1);
    double u1 = ((double)(draw(base, 2 * j) >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0,1] */
    double u2 = u01(draw(base, 2 * j + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586 * u2;
    return (i & 1) ? r * sin(a) : r * cos(a);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, float *out) {
    uint64_t b = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (float)(mean + std * normal_at(b, i));
}

/* fp32 -> bf16 bits, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, double mean, double std, uint16_t *out) {
    uint64_t b = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = f32_to_bf16((float)(mean + std * normal_at(b, i)));
}

void synth_uniform_f32(uint64_t seed, uint64_t stream, int64_t n, double lo, double hi, float *out) {
    uint64_t b = stream_base(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (float)(lo + (hi - lo) * u01(draw(b, (uint64_t)i)));
}

/* iid trits: u < p_neg -> -1, u < p_neg + p_zero -> 0, else +1 */
void synth_trits(uint64_t seed, uint64_t stream, int64_t n, double p_neg, double p_zero, int8_t *out) {
    uint64_t b = stream_base(seed, stream);
    double t0 = p_neg, t1 = p_neg + p_zero;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) {
        double u = u01(draw(b, (uint64_t)i));
        out[i] = (int8_t)(u < t0 ? -1 : (u < t1 ? 0 : 1));
    }
}

/* uniform integers in [lo, hi] (inclusive), by 64-bit modulo (bias < 2^-40 for small ranges) */
void synth_int_range(uint64_t seed, uint64_t stream, int64_t n, int64_t lo, int64_t hi, int32_t *out) {
    uint64_t b = stream_base(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1u;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = (int32_t)(lo + (int64_t)(draw(b, (uint64_t)i) % span));
}
