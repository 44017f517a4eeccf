/*
 * Counter-based seeded generator for the synthetic drafter workloads.
 *
 * This file holds no arithmetic of the drafter: it only turns (seed, stream,
 * element index) into numbers.  Both the CPU oracle and the CUDA library are
 * fed from it, so that the two see the same bits.
 *
 * Definition (every value is a pure function of seed, stream and index, so the
 * draws can be made in any order and in parallel):
 *   mix(x)      = SplitMix64 output function (Steele, Lea, Flood 2014, "Fast
 *                 splittable pseudorandom number generators"): x += 0x9e3779b97f4a7c15,
 *                 then two xor-shift-multiply rounds and a final xor-shift.
 *   key(s, t)   = mix(mix(s) ^ (t * 0xd1b54a32d192ed03))
 *   word(s,t,i) = mix(key(s, t) + i)
 *   unit53(w)   = (w >> 11) * 2^-53                       in [0, 1)
 *   unit24(w)   = (w >> 40) * 2^-24                       in [0, 1), exact in float
 *   normal pair p (elements 2p and 2p+1), Box-Muller (Box & Muller 1958), one
 *   64-bit word per pair:
 *       u1 = 1 - unit24(word(p)) in (0, 1],  u2 = unit24(word(p) << 24)
 *       r  = sqrt(-2 ln u1), out[2p] = r cos(2 pi u2), out[2p+1] = r sin(2 pi u2)
 *     computed in float with the C library's logf/sinf/cosf, then scaled by std.
 *   bf16 values are the round-to-nearest-even bf16 of that float.
 *   uniform integer in [lo, hi]: lo + floor(unit53(word(i)) * (hi - lo + 1)).
 *
 * Portable C99 + OpenMP; no architecture flags, no fast-math (the draws must
 * not depend on the compiler's licence to reassociate).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

static inline uint64_t mix(uint64_t x) {
    x += 0x9e3779b97f4a7c15ULL;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ULL;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebULL;
    return x ^ (x >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix(mix(seed) ^ (stream * 0xd1b54a32d192ed03ULL));
}

static inline double unit53(uint64_t w) { return (double)(w >> 11) * (1.0 / 9007199254740992.0); }

static inline uint16_t f32_to_bf16_rne(float f) {
    union { float f; uint32_t u; } v;
    v.f = f;
    uint32_t u = v.u;
    if ((u & 0x7f800000u) == 0x7f800000u) { /* inf / nan: keep, quiet the nan */
        return (uint16_t)((u >> 16) | ((u & 0x007fffffu) ? 0x0040u : 0u));
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static inline float unit24(uint64_t w) { return (float)(w >> 40) * (1.0f / 16777216.0f); }

static void normal_pair(uint64_t key, int64_t p, float std, float* a, float* b) {
    uint64_t w = mix(key + (uint64_t)p);
    float u1 = 1.0f - unit24(w);
    float u2 = unit24(w << 24);
    float r = sqrtf(-2.0f * logf(u1));
    float th = 6.28318530717958647692f * u2;
    *a = r * cosf(th) * std;
    *b = r * sinf(th) * std;
}

void synth_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double std, float* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; ++p) {
        float a, b;
        normal_pair(key, p, (float)std, &a, &b);
        out[2 * p] = a;
        if (2 * p + 1 < n) out[2 * p + 1] = b;
    }
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, int64_t n, double std, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < npairs; ++p) {
        float a, b;
        normal_pair(key, p, (float)std, &a, &b);
        out[2 * p] = f32_to_bf16_rne(a);
        if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_rne(b);
    }
}

void synth_uniform_int(uint64_t seed, uint64_t stream, int64_t n, int64_t lo, int64_t hi, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
    double span = (double)(hi - lo + 1);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = (int64_t)floor(unit53(mix(key + (uint64_t)i)) * span);
        if (v > hi - lo) v = hi - lo;
        out[i] = (int32_t)(lo + v);
    }
}

void synth_words(uint64_t seed, uint64_t stream, int64_t n, uint64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = mix(key + (uint64_t)i);
}
