/*
 * Seeded synthetic inputs for the attention workloads (host, plain C).
 *
 * This file computes no part of the attention method. It only draws the
 * inputs that both the CUDA path and the CPU oracle consume, so that the two
 * sides see the same bf16 bits:
 *
 *   counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
 *   pseudorandom number generators", OOPSLA 2014; the finaliser constants are
 *   the published ones) -> two 53-bit uniforms -> Box-Muller transform in
 *   double precision -> round-to-nearest-even to bfloat16.
 *
 * Element e of a stream (flat C-order index) is a pure function of
 * (seed, stream, e), so any subset of a tensor can be regenerated without the
 * rest: pair m = e/2 uses draws 2m and 2m+1; the even element takes the cosine
 * branch, the odd one the sine branch.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* Key of one stream: mixes the user seed and the stream id (tensor id). */
static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return sm64_mix(sm64_mix(seed + SM64_GAMMA) + stream * SM64_GAMMA);
}

/* Draw number c of a stream: the (c+1)-th output of SplitMix64 started at key. */
static inline uint64_t draw(uint64_t key, uint64_t c) {
    return sm64_mix(key + (c + 1) * SM64_GAMMA);
}

/* Round a finite double to the nearest bfloat16, ties to even, in one step. */
static inline uint16_t f64_to_bf16_rne(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    /* bf16 keeps 7 of the 52 fraction bits: round at bit 45. */
    uint64_t lsb = (b >> 45) & 1ULL;
    b += 0x1FFFFFFFFFFFULL + lsb;
    b &= ~0x1FFFFFFFFFFFULL;
    double r;
    memcpy(&r, &b, 8);
    float f = (float)r; /* exact: r is representable in bf16 */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static inline double normal_at(uint64_t key, uint64_t e) {
    uint64_t m = e >> 1;
    uint64_t x1 = draw(key, 2 * m);
    uint64_t x2 = draw(key, 2 * m + 1);
    double u1 = (double)((x1 >> 11) + 1) * 0x1.0p-53; /* (0, 1] */
    double u2 = (double)(x2 >> 11) * 0x1.0p-53;       /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (e & 1) ? r * sin(a) : r * cos(a);
}

/* out[k] = bf16 bits of N(0,1) element (offset + k) of stream (seed, stream). */
void wan_synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset,
                           uint64_t n, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long k = 0; k < nn; ++k)
        out[k] = f64_to_bf16_rne(normal_at(key, offset + (uint64_t)k));
}

/* Same values at arbitrary flat indices idx[0..n). */
void wan_synth_normal_bf16_at(uint64_t seed, uint64_t stream, const uint64_t* idx,
                              uint64_t n, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    long long nn = (long long)n;
#pragma omp parallel for schedule(static)
    for (long long k = 0; k < nn; ++k)
        out[k] = f64_to_bf16_rne(normal_at(key, idx[k]));
}

/* out[k] = lo + draw(k) mod (hi - lo + 1): integers uniform on [lo, hi]. */
void wan_synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t n, int64_t lo,
                           int64_t hi, int64_t* out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1ULL;
    for (uint64_t k = 0; k < n; ++k) out[k] = lo + (int64_t)(draw(key, k) % span);
}

/* Raw stream outputs, for checking the generator against published values. */
void wan_synth_raw(uint64_t key, uint64_t n, uint64_t* out) {
    for (uint64_t k = 0; k < n; ++k) out[k] = draw(key, k);
}
