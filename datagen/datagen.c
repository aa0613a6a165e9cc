/*
 * datagen.c - seeded, counter-based synthetic inputs.
 *
 * This file only draws random numbers in the distributions the workloads
 * name (uniform bytes, uniform small integers, normals, |normal| + offset,
 * a seeded choice of k out of n). It holds none of the quantized-GEMV
 * arithmetic. Both the fp64 oracle driver and the GPU tests/benchmarks take
 * their inputs from here, so the two sides see identical bytes.
 *
 * Generator: every value is a pure function of (seed, stream, index):
 *     key      = mix(mix(seed + G) ^ (stream * C))
 *     bits(i)  = mix(key + (i + 1) * G)
 * where mix() is the SplitMix64 output finaliser (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) and G is
 * the 64-bit golden-ratio increment. Being counter-based, any sub-range of a
 * tensor can be regenerated alone and the result does not depend on the
 * thread count.
 *
 * Normals use the Box-Muller transform in double precision: element i uses
 * the uniform pair (2*(i/2), 2*(i/2)+1) and takes the cosine branch for even
 * i and the sine branch for odd i. Values are rounded once to the output type.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define DG_GOLDEN 0x9E3779B97F4A7C15ull
#define DG_STREAM 0xD1B54A32D192ED03ull

static inline uint64_t dg_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t dg_key(uint64_t seed, uint64_t stream) {
    return dg_mix(dg_mix(seed + DG_GOLDEN) ^ (stream * DG_STREAM));
}

static inline uint64_t dg_at(uint64_t key, uint64_t i) {
    return dg_mix(key + (i + 1) * DG_GOLDEN);
}

/* Uniform double strictly inside (0, 1): 53 random bits plus a half step. */
static inline double dg_unit(uint64_t b) {
    return ((double)(b >> 11) + 0.5) * 0x1.0p-53;
}

static inline double dg_normal_at(uint64_t key, uint64_t i) {
    uint64_t p = i >> 1;
    double u1 = dg_unit(dg_at(key, 2 * p));
    double u2 = dg_unit(dg_at(key, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1));
    double a = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(a) : r * cos(a);
}

/* Raw 64-bit draws (exposed so tests can check the generator itself). */
void dg_bits(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
             uint64_t *out) {
    uint64_t key = dg_key(seed, stream);
    for (uint64_t j = 0; j < n; ++j) out[j] = dg_at(key, start + j);
}

/* Uniform bytes 0..255; byte j of the tensor is byte (j % 8) of draw j / 8. */
void dg_u8(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
           uint8_t *out) {
    uint64_t key = dg_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j) {
        uint64_t g = start + (uint64_t)j;
        out[j] = (uint8_t)(dg_at(key, g >> 3) >> (8 * (g & 7)));
    }
}

/* Uniform integers in [-lim, lim]. */
void dg_int8_sym(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                 int lim, int8_t *out) {
    uint64_t key = dg_key(seed, stream);
    uint64_t span = (uint64_t)(2 * lim + 1);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j)
        out[j] = (int8_t)((int64_t)(dg_at(key, start + (uint64_t)j) % span) - lim);
}

/* mean + std * N(0,1), rounded once to fp32. */
void dg_normal_f32(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                   double mean, double std, float *out) {
    uint64_t key = dg_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j)
        out[j] = (float)(mean + std * dg_normal_at(key, start + (uint64_t)j));
}

/* |std * N(0,1)| + add, rounded once to fp32. */
void dg_absnormal_f32(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                      double std, double add, float *out) {
    uint64_t key = dg_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j)
        out[j] = (float)(fabs(std * dg_normal_at(key, start + (uint64_t)j)) + add);
}

/* std * N(0,1) rounded to bfloat16 (round to nearest even through fp32). */
void dg_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n,
                    double std, uint16_t *out) {
    uint64_t key = dg_key(seed, stream);
    int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < nn; ++j) {
        float f = (float)(std * dg_normal_at(key, start + (uint64_t)j));
        uint32_t u;
        memcpy(&u, &f, 4);
        uint32_t lsb = (u >> 16) & 1u;
        u += 0x7FFFu + lsb;
        out[j] = (uint16_t)(u >> 16);
    }
}

/* A seeded choice of n_pick distinct values out of 0..n_total-1, in the order
 * a partial Fisher-Yates shuffle draws them. Returns 0, or -1 on bad sizes. */
int dg_choose(uint64_t seed, uint64_t stream, int n_total, int n_pick,
              int32_t *out, int32_t *scratch /* n_total ints */) {
    if (n_total <= 0 || n_pick < 0 || n_pick > n_total) return -1;
    uint64_t key = dg_key(seed, stream);
    for (int i = 0; i < n_total; ++i) scratch[i] = i;
    for (int i = 0; i < n_pick; ++i) {
        uint64_t left = (uint64_t)(n_total - i);
        int j = i + (int)(dg_at(key, (uint64_t)i) % left);
        int32_t t = scratch[i];
        scratch[i] = scratch[j];
        scratch[j] = t;
        out[i] = scratch[i];
    }
    return 0;
}
