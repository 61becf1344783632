/*
 * Seeded synthetic inputs for the int4-g128 weight-streaming GEMV (host side).
 *
 * This module holds no arithmetic of the method itself.  It only draws the
 * inputs the tests, the benchmark and the oracle share:
 *
 *   codes   uint32 [K/8][N]   8 uniform 4-bit codes per word (canonical order)
 *   scales  bf16   [K/128][N] U(0.002, 0.02), rounded to bf16
 *   mins    bf16   [K/128][N] -8 * scale_bf16 * (1 + U(-0.1, 0.1)), rounded to bf16
 *   x       bf16   [M][K]     N(0, 1) by Box-Muller, rounded to bf16
 *
 * The value distributions follow the Token Rush README's int4 format
 * (group-wise asymmetric int4, one bf16 scale and one bf16 minimum per 128
 * weights; "Quantization" section) with scale/min ranges of the usual
 * min = -8*scale centred code grid.
 *
 * Generator: counter-based SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; output mixing
 * constants as in S. Vigna's public-domain splitmix64).  Element i of a
 * stream with key `key` is mix64(key + (i + 1) * GAMMA), i.e. the i-th output
 * of a SplitMix64 sequence seeded with `key`.  Every element is therefore
 * computable on its own, which lets the device fill kernels (synth_dev.cu)
 * reproduce exactly the same bits and lets the host sample single columns of
 * a matrix too large to hold.
 *
 * Floating-point steps use only IEEE-754 double add/mul with round-to-nearest
 * (this file must be compiled with -ffp-contract=off), and the rounding to
 * bf16 is done with integer operations on the double's bits, so host and
 * device agree bit for bit.  Box-Muller (x only) uses libm and is host-only.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

enum { SYNTH_CODES = 0, SYNTH_SCALES = 1, SYNTH_MINS = 2, SYNTH_X = 3 };

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of one array (codes/scales/mins/x) of one matrix of one seeded workload. */
uint64_t synth_key(uint64_t seed, uint64_t matrix_id, uint32_t array_id) {
    return mix64(seed ^ mix64(matrix_id * SYNTH_GAMMA + (uint64_t)array_id + 1ULL));
}

uint64_t synth_draw(uint64_t key, uint64_t index) {
    return mix64(key + (index + 1ULL) * SYNTH_GAMMA);
}

/* Uniform double in [0, 1) with 53 random bits. */
static double u53(uint64_t v) { return (double)(v >> 11) * (1.0 / 9007199254740992.0); }

/* double -> bf16 bits, round to nearest, ties to even, integer-only. */
uint16_t synth_bf16_rn(double d) {
    uint64_t b;
    memcpy(&b, &d, 8);
    uint16_t sign = (uint16_t)((b >> 63) << 15);
    int e = (int)((b >> 52) & 0x7FF);
    uint64_t mant = b & ((1ULL << 52) - 1);
    if (e == 0x7FF) return (uint16_t)(sign | 0x7F80 | (mant ? 0x40 : 0));
    if (e == 0) return sign; /* zero or double-subnormal: far below bf16 range */
    int E = e - 1023;
    uint64_t m = (1ULL << 52) | mant; /* 53-bit significand */
    if (E >= -126) {
        uint64_t q = m >> 45, rem = m & ((1ULL << 45) - 1), half = 1ULL << 44;
        if (rem > half || (rem == half && (q & 1))) q++;
        if (q == 256) { q = 128; E++; }
        if (E > 127) return (uint16_t)(sign | 0x7F80);
        return (uint16_t)(sign | ((uint16_t)(E + 127) << 7) | (uint16_t)(q & 0x7F));
    }
    /* bf16 subnormal: value = q * 2^-133 */
    int s = -(E + 81);
    if (s >= 54) return sign;
    uint64_t q = m >> s, rem = m & ((1ULL << s) - 1), half = 1ULL << (s - 1);
    if (rem > half || (rem == half && (q & 1))) q++;
    return (uint16_t)(sign | (uint16_t)q); /* q == 128 encodes the smallest normal */
}

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

uint16_t synth_scale_at(uint64_t key_s, uint64_t idx) {
    double u = u53(synth_draw(key_s, idx));
    double t = 0.018 * u;
    return synth_bf16_rn(0.002 + t);
}

uint16_t synth_min_at(uint64_t key_s, uint64_t key_m, uint64_t idx) {
    double sb = bf16_to_double(synth_scale_at(key_s, idx));
    double v = u53(synth_draw(key_m, idx));
    double b = 2.0 * v - 1.0;      /* exact */
    double c = 0.1 * b;
    double f = 1.0 + c;
    double p = -8.0 * sb;          /* exact */
    return synth_bf16_rn(p * f);
}

/* codes[K/8][N]: word i = low 32 bits of draw i. */
void synth_codes(uint64_t seed, uint64_t matrix_id, int64_t n_words, uint32_t* out) {
    uint64_t key = synth_key(seed, matrix_id, SYNTH_CODES);
    for (int64_t i = 0; i < n_words; i++) out[i] = (uint32_t)synth_draw(key, (uint64_t)i);
}

/* scales/mins [G][N]. */
void synth_meta(uint64_t seed, uint64_t matrix_id, int64_t n, uint16_t* scales, uint16_t* mins) {
    uint64_t ks = synth_key(seed, matrix_id, SYNTH_SCALES);
    uint64_t km = synth_key(seed, matrix_id, SYNTH_MINS);
    for (int64_t i = 0; i < n; i++) {
        scales[i] = synth_scale_at(ks, (uint64_t)i);
        mins[i] = synth_min_at(ks, km, (uint64_t)i);
    }
}

/* Selected columns of a [K][N] matrix: codes_out[K/8][ncols], meta_out[G][ncols]. */
void synth_columns(uint64_t seed, uint64_t matrix_id, int K, int N, const int* cols, int ncols,
                   uint32_t* codes_out, uint16_t* scales_out, uint16_t* mins_out) {
    uint64_t kc = synth_key(seed, matrix_id, SYNTH_CODES);
    uint64_t ks = synth_key(seed, matrix_id, SYNTH_SCALES);
    uint64_t km = synth_key(seed, matrix_id, SYNTH_MINS);
    int J = K / 8, G = K / 128;
    for (int j = 0; j < J; j++)
        for (int c = 0; c < ncols; c++)
            codes_out[(int64_t)j * ncols + c] =
                (uint32_t)synth_draw(kc, (uint64_t)j * (uint64_t)N + (uint64_t)cols[c]);
    for (int g = 0; g < G; g++)
        for (int c = 0; c < ncols; c++) {
            uint64_t idx = (uint64_t)g * (uint64_t)N + (uint64_t)cols[c];
            scales_out[(int64_t)g * ncols + c] = synth_scale_at(ks, idx);
            mins_out[(int64_t)g * ncols + c] = synth_min_at(ks, km, idx);
        }
}

/* x[M][K] ~ N(0,1) by the Box-Muller transform (G. Box, M. Muller, 1958). */
void synth_x(uint64_t seed, uint64_t matrix_id, int64_t n, uint16_t* out) {
    uint64_t key = synth_key(seed, matrix_id, SYNTH_X);
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = 0; i < n; i++) {
        double u1 = 1.0 - u53(synth_draw(key, 2 * (uint64_t)i));     /* (0, 1] */
        double u2 = u53(synth_draw(key, 2 * (uint64_t)i + 1));
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[i] = synth_bf16_rn(z);
    }
}
