/*
 * Seeded synthetic inputs for the expert-streaming MoE layer.
 *
 * This file draws random numbers and converts them to storage formats. It holds
 * none of the layer's arithmetic (no dequantisation, no routing, no FFN): both
 * the CPU oracle and the CUDA library consume what it writes, so it must stay
 * independent of either.
 *
 * Counter-based generator. Every value is a pure function of
 *   (seed, tensor id, layer, expert-or-step, element index)
 * so any slice can be regenerated in isolation and in parallel. The mixing
 * function is the SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *   mix(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
 *           z *= 0x94D049BB133111EB; z ^= z >> 31.
 * Stream key  = mix(mix(seed) ^ (tensor << 56 | layer << 40 | sub)),
 * word j      = mix(key + (j + 1) * 0x9E3779B97F4A7C15).
 *
 * Storage conversions are round-to-nearest-even, written from the IEEE 754
 * binary16 definition and from the bfloat16 definition (top 16 bits of binary32).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ULL;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBULL;
    z ^= z >> 31;
    return z;
}

uint64_t synth_key(uint64_t seed, uint32_t tensor, uint32_t layer, uint64_t sub) {
    uint64_t tag = ((uint64_t)(tensor & 0xFF) << 56) | ((uint64_t)(layer & 0xFFFF) << 40) |
                   (sub & 0xFFFFFFFFFFULL);
    return mix64(mix64(seed) ^ tag);
}

static inline uint64_t word_at(uint64_t key, uint64_t j) { return mix64(key + (j + 1) * GOLDEN); }

/* 64-bit words of the stream, for tests of the generator itself. */
void synth_words(uint64_t key, uint64_t first, uint64_t n, uint64_t* out) {
    for (uint64_t j = 0; j < n; ++j) out[j] = word_at(key, first + j);
}

/* Uniform double in [0, 1) from the top 53 bits of a word. */
static inline double unit53(uint64_t w) { return (double)(w >> 11) * (1.0 / 9007199254740992.0); }

/* ---- storage conversions ------------------------------------------------ */

/* double -> IEEE binary16 bits, round to nearest, ties to even. Finite inputs
 * below the half range only (the generator never produces anything else);
 * values beyond 65504 saturate to infinity per IEEE rounding. */
uint16_t synth_f64_to_f16(double v) {
    uint16_t sign = 0;
    if (signbit(v)) { sign = 0x8000; v = -v; }
    if (v == 0.0) return sign;
    int e;
    double m = frexp(v, &e); /* v = m * 2^e, m in [0.5, 1) */
    int exp_unbiased = e - 1; /* v = (2m) * 2^(e-1), 2m in [1, 2) */
    if (exp_unbiased < -14) {
        /* subnormal: value = k * 2^-24 */
        double k = nearbyint(ldexp(v, 24));
        if (k >= 1024.0) return (uint16_t)(sign | 0x0400); /* rounded up to the smallest normal */
        return (uint16_t)(sign | (uint16_t)k);
    }
    double k = nearbyint(ldexp(v, 10 - exp_unbiased)); /* in [1024, 2048] */
    if (k >= 2048.0) { k = 1024.0; exp_unbiased += 1; }
    if (exp_unbiased > 15) return (uint16_t)(sign | 0x7C00);
    return (uint16_t)(sign | (uint16_t)((exp_unbiased + 15) << 10) | (uint16_t)((int)k - 1024));
}

/* binary32 -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
uint16_t synth_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---- tensors ------------------------------------------------------------ */

/* n unsigned 4-bit codes, uniform on 0..15, packed two per byte: element 2j in
 * the low nibble of byte j, element 2j+1 in the high nibble. Code i is nibble
 * (i % 16) of word i / 16. n must be even. */
void synth_codes_u4(uint64_t key, uint64_t n, uint8_t* out) {
    /* nibble c of a word sits at bits 4c..4c+3, so byte b of the packed pair
     * stream is bits 8b..8b+7 of the word (low nibble = even element). */
    uint64_t nbytes = n / 2;
    uint64_t words = (nbytes + 7) / 8;
    for (uint64_t w = 0; w < words; ++w) {
        uint64_t v = word_at(key, w);
        uint64_t base = w * 8;
        if (base + 8 <= nbytes) {
            for (int b = 0; b < 8; ++b) out[base + b] = (uint8_t)(v >> (8 * b));
        } else {
            for (int b = 0; base + b < nbytes; ++b) out[base + b] = (uint8_t)(v >> (8 * b));
        }
    }
}

/* n unsigned 8-bit codes, uniform on 0..255: code i is byte (i % 8) of word i / 8. */
void synth_codes_u8(uint64_t key, uint64_t n, uint8_t* out) {
    uint64_t words = (n + 7) / 8;
    for (uint64_t w = 0; w < words; ++w) {
        uint64_t v = word_at(key, w);
        for (int c = 0; c < 8 && w * 8 + c < n; ++c) out[w * 8 + c] = (uint8_t)((v >> (8 * c)) & 0xFFu);
    }
}

/* n group scales s ~ U(lo, hi) / div rounded to binary16, and biases
 * b = bias_mult * s (computed from the rounded s, then rounded to binary16;
 * exact when bias_mult is a power of two). */
void synth_scale_bias_f16(uint64_t key, uint64_t n, double lo, double hi, double div, double bias_mult,
                          uint16_t* scale, uint16_t* bias) {
    for (uint64_t i = 0; i < n; ++i) {
        double s = (lo + (hi - lo) * unit53(word_at(key, i))) / div;
        uint16_t sh = synth_f64_to_f16(s);
        scale[i] = sh;
        /* decode sh exactly to form the bias from the stored scale */
        int ex = (sh >> 10) & 0x1F, mant = sh & 0x3FF;
        double sv = ex ? ldexp(1024.0 + mant, ex - 25) : ldexp((double)mant, -24);
        bias[i] = synth_f64_to_f16(bias_mult * sv);
    }
}

/* rows x cols standard normals (Box-Muller on word pairs 2p, 2p+1), optionally
 * scaled per row to unit root-mean-square, stored as bfloat16. */
void synth_normal_bf16(uint64_t key, int rows, int cols, int rms_normalise, uint16_t* out, double* scratch) {
    for (int r = 0; r < rows; ++r) {
        uint64_t base = (uint64_t)r * (uint64_t)cols;
        for (int c = 0; c < cols; c += 2) {
            uint64_t p = (base + (uint64_t)c) / 2; /* cols is even */
            double u1 = ((double)((word_at(key, 2 * p) >> 11) + 1)) * (1.0 / 9007199254740992.0);
            double u2 = unit53(word_at(key, 2 * p + 1));
            double rad = sqrt(-2.0 * log(u1));
            scratch[c] = rad * cos(6.283185307179586 * u2);
            if (c + 1 < cols) scratch[c + 1] = rad * sin(6.283185307179586 * u2);
        }
        double scale = 1.0;
        if (rms_normalise) {
            double ss = 0.0;
            for (int c = 0; c < cols; ++c) ss += scratch[c] * scratch[c];
            scale = 1.0 / sqrt(ss / (double)cols);
        }
        for (int c = 0; c < cols; ++c) out[base + (uint64_t)c] = synth_f32_to_bf16((float)(scratch[c] * scale));
    }
}

/* A seeded permutation of 0..n-1 (Fisher-Yates, j = word(i) mod (i+1)). */
void synth_permutation(uint64_t key, int n, int32_t* perm) {
    for (int i = 0; i < n; ++i) perm[i] = i;
    for (int i = n - 1; i > 0; --i) {
        int j = (int)(word_at(key, (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}
