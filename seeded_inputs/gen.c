/*
 * Seeded synthetic inputs for the routed-MoE layer.
 *
 * This file produces the INPUTS of the method (quantised weights in their
 * canonical storage format, router weights, router bias, activations). It
 * holds none of the method's arithmetic: no dequantisation, no dot product,
 * no routing, no activation function. Both the fp64 oracle and the GPU tests
 * draw from it, so each side sees the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; finaliser constants as in
 * Vigna's public-domain splitmix64.c). It is used in counter form: element i
 * of the stream with key K is mix64(K + (i + 1) * GOLDEN), which equals the
 * i-th output of a SplitMix64 generator whose state starts at K. Any element
 * is therefore a pure function of (key, i), and every fill below can run on
 * any number of threads and give identical bytes.
 *
 * Storage formats produced here (the canonical ones that cross the library's
 * C ABI):
 *   q4g64 matrix [N][K]:  codes uint8 [N][K/2], element k of a row sits in
 *                         byte k/2, low nibble for even k, high for odd k;
 *                         scale, bias: IEEE binary16 bit patterns [N][K/64].
 *   q8g64 matrix [N][K]:  codes uint8 [N][K], scale/bias binary16 [N][K/64].
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>

#define SI_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t si_at(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1ULL) * SI_GOLDEN);
}

/* Stream key from a seed and up to four small identifiers. */
uint64_t si_key(uint64_t seed, uint64_t tag, uint64_t a, uint64_t b, uint64_t c) {
    uint64_t k = mix64(seed + SI_GOLDEN);
    k = mix64(k ^ (tag * 0xD1B54A32D192ED03ULL + 1ULL));
    k = mix64(k ^ (a * 0xAEF17502108EF2D9ULL + 2ULL));
    k = mix64(k ^ (b * 0xDB4F0B9175AE2165ULL + 3ULL));
    k = mix64(k ^ (c * 0x9FB21C651E98DF25ULL + 4ULL));
    return k;
}

/* Raw stream elements [start, start + n). */
void si_fill_u64(uint64_t key, uint64_t start, uint64_t n, uint64_t* out) {
    #pragma omp parallel for schedule(static) if (n > (1u << 16))
    for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = si_at(key, start + (uint64_t)i);
}

/* Bytes of the stream, little-endian within each 64-bit element. Uniform
 * bytes give independent uniform nibbles 0..15 (4-bit codes) and uniform
 * bytes 0..255. */
void si_fill_bytes(uint64_t key, uint64_t nbytes, uint8_t* out) {
    uint64_t nw = nbytes / 8;
    #pragma omp parallel for schedule(static) if (nw > (1u << 16))
    for (int64_t i = 0; i < (int64_t)nw; ++i) {
        uint64_t r = si_at(key, (uint64_t)i);
        uint8_t b[8];
        for (int j = 0; j < 8; ++j) b[j] = (uint8_t)(r >> (8 * j));
        memcpy(out + 8 * i, b, 8);
    }
    if (nbytes % 8) {
        uint64_t r = si_at(key, nw);
        for (uint64_t j = 0; j < nbytes % 8; ++j) out[8 * nw + j] = (uint8_t)(r >> (8 * j));
    }
}

/* Uniform double in [0, 1) from the top 53 bits. */
static inline double si_u01(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }

/* IEEE binary16, round to nearest even, from a double. Handles normal,
 * subnormal, overflow (to inf) and NaN. */
uint16_t si_f64_to_f16(double v) {
    uint64_t u; memcpy(&u, &v, 8);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    int e = (int)((u >> 52) & 0x7FF);
    uint64_t m = u & 0xFFFFFFFFFFFFFULL;
    if (e == 0x7FF) return sign | 0x7C00u | (m ? 0x200u : 0u);
    if (e == 0 && m == 0) return sign;
    /* value = 1.m * 2^(e-1023) for normal doubles; doubles below 2^-1022
     * round to zero in binary16 anyway. */
    if (e == 0) return sign;
    int ue = e - 1023;                          /* unbiased exponent */
    uint64_t sig = m | (1ULL << 52);            /* 53-bit significand */
    int shift;                                  /* bits of sig to drop */
    uint16_t hexp;
    if (ue > 15) return sign | 0x7C00u;
    if (ue >= -14) { shift = 52 - 10; hexp = (uint16_t)(ue + 15); }
    else {                                      /* subnormal binary16 */
        shift = 52 - 10 + (-14 - ue);
        hexp = 0;
        if (shift > 63) return sign;
    }
    uint64_t keep = sig >> shift;
    uint64_t rem = sig & ((1ULL << shift) - 1ULL);
    uint64_t half = 1ULL << (shift - 1);
    if (rem > half || (rem == half && (keep & 1ULL))) keep += 1ULL;
    uint32_t out;
    if (hexp == 0) {
        out = (uint32_t)keep;                   /* may carry into the smallest normal */
    } else {
        /* keep holds the implicit bit at position 10 (or 11 after a carry) */
        if (keep >> 11) { keep >>= 1; hexp += 1; }
        if (hexp >= 31) return sign | 0x7C00u;
        out = ((uint32_t)hexp << 10) | (uint32_t)(keep & 0x3FFu);
    }
    return (uint16_t)(sign | out);
}

/* bfloat16, round to nearest even, from a float (NaN kept quiet). */
uint16_t si_f32_to_bf16(float f) {
    uint32_t u; memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* fp16 values drawn as fp16(lo + (hi - lo) * U[0,1)), rounded to nearest even. */
void si_fill_f16_uniform(uint64_t key, uint64_t n, double lo, double hi, uint16_t* out) {
    #pragma omp parallel for schedule(static) if (n > (1u << 16))
    for (int64_t i = 0; i < (int64_t)n; ++i)
        out[i] = si_f64_to_f16(lo + (hi - lo) * si_u01(si_at(key, (uint64_t)i)));
}

/* Normal(0, sd) via Box-Muller (cosine branch), element i from stream
 * elements 2i and 2i+1, rounded once to float. */
static inline double si_normal_at(uint64_t key, uint64_t i) {
    double u1 = ((double)(si_at(key, 2 * i) >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
    double u2 = si_u01(si_at(key, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

void si_fill_normal_f32(uint64_t key, uint64_t n, double sd, float* out) {
    #pragma omp parallel for schedule(static) if (n > (1u << 14))
    for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = (float)(sd * si_normal_at(key, (uint64_t)i));
}

/* Normal(0, sd) rounded to float, then to bfloat16 (round to nearest even). */
void si_fill_normal_bf16(uint64_t key, uint64_t n, double sd, uint16_t* out) {
    #pragma omp parallel for schedule(static) if (n > (1u << 14))
    for (int64_t i = 0; i < (int64_t)n; ++i)
        out[i] = si_f32_to_bf16((float)(sd * si_normal_at(key, (uint64_t)i)));
}

/* Heavy-tailed activations: Normal(0, 1) draws (stream `key`) in runs of
 * `group` elements; in every run, the one element at the position drawn from
 * stream `key_pos` (element r of that stream for run r) is multiplied by
 * `factor` (an outlier channel per run). Rounded once to float; to bfloat16
 * as well when out_bf16 is given. */
void si_fill_normal_outliers(uint64_t key, uint64_t key_pos, uint64_t n, uint64_t group, double factor,
                             float* out_f32, uint16_t* out_bf16) {
    for (int64_t i = 0; i < (int64_t)n; ++i) {
        const uint64_t run = (uint64_t)i / group, at = si_at(key_pos, run) % group;
        double v = si_normal_at(key, (uint64_t)i);
        if ((uint64_t)i - run * group == at) v *= factor;
        const float f = (float)v;
        if (out_f32) out_f32[i] = f;
        if (out_bf16) out_bf16[i] = si_f32_to_bf16(f);
    }
}

/* Fisher-Yates permutation of 0..n-1 driven by the stream; draw j uniformly in
 * [0, i] with Lemire's multiply-shift on a 64-bit element. */
void si_permutation(uint64_t key, int64_t n, int64_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        unsigned __int128 p = (unsigned __int128)si_at(key, (uint64_t)i) * (unsigned __int128)(uint64_t)(i + 1);
        int64_t j = (int64_t)(uint64_t)(p >> 64);
        int64_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}

/* Affine group-64 8-bit encoding of a float matrix [N][K] (K % 64 == 0):
 * per group, scale = fp16((max - min) / 255), bias = fp16(min), and
 * code = clamp(rne((w - bias) / scale), 0, 255) with the rounded fp16
 * scale and bias. A constant group stores scale 0 and codes 0.
 * This is how the synthetic 8-bit router weights are made; the method
 * itself only ever reads the codes back. */
static double si_f16_to_f64(uint16_t h) {
    int e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v = (e == 0) ? ldexp((double)m, -24) : ldexp((double)(m | 0x400), e - 25);
    return (h & 0x8000) ? -v : v;
}

void si_encode_q8g64(const float* w, int64_t N, int64_t K, uint8_t* codes, uint16_t* scale, uint16_t* bias) {
    int64_t G = K / 64;
    #pragma omp parallel for schedule(static) if (N * K > (1 << 16))
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float* p = w + n * K + g * 64;
            double mn = p[0], mx = p[0];
            for (int i = 1; i < 64; ++i) { if (p[i] < mn) mn = p[i]; if (p[i] > mx) mx = p[i]; }
            uint16_t sh = si_f64_to_f16((mx - mn) / 255.0);
            uint16_t bh = si_f64_to_f16(mn);
            double s = si_f16_to_f64(sh), b = si_f16_to_f64(bh);
            scale[n * G + g] = sh; bias[n * G + g] = bh;
            for (int i = 0; i < 64; ++i) {
                double c = (s > 0.0) ? nearbyint(((double)p[i] - b) / s) : 0.0; /* default mode: ties to even */
                if (c < 0.0) c = 0.0;
                if (c > 255.0) c = 255.0;
                codes[n * K + g * 64 + i] = (uint8_t)c;
            }
        }
    }
}
