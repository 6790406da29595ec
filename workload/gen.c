/*
 * Seeded synthetic-input generators for the streamed-expert MoE layer.
 *
 * This module is shared by the CPU oracle, the tests and the benchmark. It
 * holds none of the layer's arithmetic: it only draws random numbers and
 * encodes them as bf16 / fp16 / 4-bit codes, the input formats the layer
 * consumes.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used counter-style: the i-th draw of a
 * stream with key K is mix64(K + (i + 1) * GAMMA), so any element can be
 * produced independently of the others. A stream key is derived from
 * (seed, tensor, layer, expert, matrix) by absorbing each field with the same
 * finaliser.
 *
 * Distributions (the synthetic workloads of the pages' model: Gemma-4-26B-A4B
 * style MoE with 4-bit experts):
 *   normal   : Box-Muller on two 53-bit uniforms, in double, rounded to fp32,
 *              then round-to-nearest-even to bf16;
 *   uniform  : lo + (hi - lo) * u in double, rounded to fp32, then
 *              round-to-nearest-even to fp16;
 *   codes    : 4-bit values taken from consecutive nibbles of the draws
 *              (16 codes per 64-bit draw).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define WL_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t wl_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t wl_key(uint64_t seed, uint64_t tensor, uint64_t layer, uint64_t expert, uint64_t matrix) {
    uint64_t h = seed;
    h = wl_mix64((h ^ tensor) + WL_GAMMA);
    h = wl_mix64((h ^ layer) + WL_GAMMA);
    h = wl_mix64((h ^ expert) + WL_GAMMA);
    h = wl_mix64((h ^ matrix) + WL_GAMMA);
    return h;
}

uint64_t wl_u64(uint64_t key, uint64_t i) { return wl_mix64(key + (i + 1) * WL_GAMMA); }

double wl_unif53(uint64_t key, uint64_t i) {
    return (double)(wl_u64(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* fp32 -> bf16, round to nearest even; NaN stays a quiet NaN. */
uint16_t wl_f32_to_bf16(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* fp32 -> fp16 (IEEE binary16), round to nearest even, with subnormals. */
uint16_t wl_f32_to_f16(float f) {
    uint32_t u = f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t ex = (u >> 23) & 0xFFu;
    uint32_t man = u & 0x007FFFFFu;
    if (ex == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x0200u : 0u));
    int32_t e = (int32_t)ex - 127 + 15;
    if (e >= 0x1F) return (uint16_t)(sign | 0x7C00u);
    if (e <= 0) {
        if (e < -10) return (uint16_t)sign;
        man |= 0x00800000u;
        uint32_t shift = (uint32_t)(14 - e);
        uint32_t half = man >> shift;
        uint32_t rem = man & ((1u << shift) - 1u);
        uint32_t mid = 1u << (shift - 1);
        if (rem > mid || (rem == mid && (half & 1u))) half++;
        return (uint16_t)(sign | half);
    }
    uint32_t half = sign | ((uint32_t)e << 10) | (man >> 13);
    uint32_t rem = man & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (half & 1u))) half++;
    return (uint16_t)half;
}

float wl_normal(uint64_t key, uint64_t i) {
    double u1 = wl_unif53(key, 2 * i);
    double u2 = wl_unif53(key, 2 * i + 1);
    double z = sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586476925 * u2);
    return (float)z;
}

void wl_normal_bf16(uint64_t key, uint64_t n, double sigma, uint16_t* out) {
    for (uint64_t i = 0; i < n; ++i) {
        double u1 = wl_unif53(key, 2 * i);
        double u2 = wl_unif53(key, 2 * i + 1);
        double z = sqrt(-2.0 * log(1.0 - u1)) * cos(6.283185307179586476925 * u2);
        out[i] = wl_f32_to_bf16((float)(sigma * z));
    }
}

void wl_normal_f32(uint64_t key, uint64_t n, double sigma, float* out) {
    for (uint64_t i = 0; i < n; ++i) out[i] = (float)(sigma * (double)wl_normal(key, i));
}

void wl_uniform_f16(uint64_t key, uint64_t n, double lo, double hi, uint16_t* out) {
    for (uint64_t i = 0; i < n; ++i)
        out[i] = wl_f32_to_f16((float)(lo + (hi - lo) * wl_unif53(key, i)));
}

void wl_codes(uint64_t key, uint64_t n, uint8_t* q) {
    for (uint64_t i = 0; i < n; ++i)
        q[i] = (uint8_t)((wl_u64(key, i >> 4) >> (4 * (i & 15))) & 15u);
}

/* Fisher-Yates shuffle of 0..n-1; step t draws j = u64 mod (i + 1). */
void wl_permutation(uint64_t key, int32_t n, int32_t* perm) {
    for (int32_t i = 0; i < n; ++i) perm[i] = i;
    for (int32_t i = n - 1, t = 0; i >= 1; --i, ++t) {
        int32_t j = (int32_t)(wl_u64(key, (uint64_t)t) % (uint64_t)(i + 1));
        int32_t tmp = perm[i]; perm[i] = perm[j]; perm[j] = tmp;
    }
}

/*
 * Zipf(s) expert popularity as an additive router-logit bias: rank r = 1..E
 * has p_r = r^-s / sum_j j^-s; a seeded permutation maps rank -> expert, and
 * bias[expert] = alpha * ln(p_rank).
 */
void wl_zipf_bias(uint64_t key, int32_t E, double s, double alpha, float* bias, int32_t* perm_out) {
    int32_t perm[4096];
    if (E > 4096) return;
    wl_permutation(key, E, perm);
    double z = 0.0;
    for (int32_t r = 1; r <= E; ++r) z += pow((double)r, -s);
    for (int32_t r = 1; r <= E; ++r) {
        double p = pow((double)r, -s) / z;
        bias[perm[r - 1]] = (float)(alpha * log(p));
    }
    if (perm_out) memcpy(perm_out, perm, sizeof(int32_t) * (size_t)E);
}
