// qmv_device.cuh - device building blocks shared by the GB300 quantized GEMV kernels.
//
// The decode kernels stream packed weights once from HBM, turn them into exact
// fp16 values in registers, and let the warp-level tensor-core MMA
// (mma.sync m16n8k16, fp16 in, fp32 accumulate) do the multiply-adds:
//
//   * int4 offset-binary nibbles (value = nibble - 8, colibri PR #418 commit
//     "opt-in Vulkan int4/int8 quantized GEMV") and int8 values are small
//     integers, so their fp16 form is exact.
//   * Activations are split into two fp16 parts, v = hi + lo with
//     hi = fp16(v) and lo = fp16(v - hi), after a per-row power-of-two
//     rescale that puts max|v| in [2^13, 2^14). hi + lo carries ~22
//     significant bits, so the products keep fp32-level accuracy. hi and lo
//     occupy two MMA columns of the same token and are added after the MMA.
//   * The MMA accumulates one 64-wide K group at a time from zero; the group
//     partial is then scaled by that group's fp32 scale and added into an
//     fp32 register accumulator (colibri PR #418 commit "grouped scales in
//     the Vulkan kernels": the scale multiplies the group partial).
//
// The MMA K order inside a group is a fixed permutation of the 64 values,
// applied identically to weights and activations (a dot product does not
// depend on the order of its terms).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmv {

constexpr int kGroup = 64;  // K values per scale group

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;  // (a & b) | c
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt_u32(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Streaming loads of data read exactly once: skip L1, keep L2 for neighbours.
__device__ __forceinline__ uint2 ldg_stream_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream_u4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float ldg_stream_f32(const float *p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// d += A(16x16, row) * B(16x8, col), fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Output element i of a GEMV: fp32 into y, or, when ybf is set, the fp32
// result rounded to the nearest bf16 (ties to even) into ybf.
__device__ __forceinline__ void store_y(float *y, uint16_t *ybf, size_t i, float v) {
    if (ybf) ybf[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else y[i] = v;
}

// ------------------------------------------------------------------ dequant

// One 32-bit word of int4 weights holds elements e0..e7 (element i in bits
// 4i..4i+3). Returns four half2 with exact values (nibble - 8):
//   p[0] = (e0, e4), p[1] = (e1, e5), p[2] = (e2, e6), p[3] = (e3, e7)
// (first element in the low half). Exponent-bias technique: OR-ing a nibble
// into the mantissa of fp16 1024.0 (0x6400, unit spacing) gives 1024 + n;
// a nibble four bits higher gives 1024 + 16 n. Subtracting 1032, or scaling by
// 1/16 and subtracting 72, leaves n - 8 exactly.
__device__ __forceinline__ void dequant_int4_word(uint32_t w, uint32_t p[4]) {
    const uint32_t kBias = 0x64006400u;      // (1024, 1024)
    const uint32_t kMinus1032 = 0xE408E408u; // (-1032, -1032)
    const uint32_t kSixteenth = 0x2C002C00u; // (1/16, 1/16)
    const uint32_t kMinus72 = 0xD480D480u;   // (-72, -72)
    const uint32_t w8 = w >> 8;
    p[0] = hadd2_u32(lop3_and_or(w, 0x000F000Fu, kBias), kMinus1032);
    p[1] = hfma2_u32(lop3_and_or(w, 0x00F000F0u, kBias), kSixteenth, kMinus72);
    p[2] = hadd2_u32(lop3_and_or(w8, 0x000F000Fu, kBias), kMinus1032);
    p[3] = hfma2_u32(lop3_and_or(w8, 0x00F000F0u, kBias), kSixteenth, kMinus72);
}

// The tensor-map decode kernel's int4 form: no fp16 arithmetic at all. A
// nibble masked into the low bits of an fp16 word is the subnormal n * 2^-24,
// and a nibble four bits up is (16 n) * 2^-24, both exact:
//   p[0] = (e0, e4) * 2^-24, p[1] = (e1, e5) * 16 * 2^-24,
//   p[2] = (e2, e6) * 2^-24, p[3] = (e3, e7) * 16 * 2^-24.
// The activations that meet p[1] and p[3] are stored divided by 16 (exact,
// see make_unit_s), so the MMA sums 2^-24 * n * v, and the offset -8 enters
// as the accumulator's initial value -8 * 2^-24 * sum(v) of each token
// (tile_group_int4s). Five integer instructions for eight weights instead of
// nine with fp16 adds.
__device__ __forceinline__ void dequant_int4_word_s(uint32_t w, uint32_t p[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = w & 0x000F000Fu;
    p[1] = w & 0x00F000F0u;
    p[2] = w8 & 0x000F000Fu;
    p[3] = w8 & 0x00F000F0u;
}

// One 32-bit word of int8 weights (bytes b0..b3, signed). Returns exact half2
//   pa = (b0, b2), pb = (b1, b3).
// Flipping the sign bit maps b to b + 128 in 0..255; placing that byte under
// 0x64 gives fp16 1024 + b + 128; subtracting 1152 leaves b.
__device__ __forceinline__ void dequant_int8_word(uint32_t w, uint32_t &pa, uint32_t &pb) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t kHigh = 0x64646464u;
    const uint32_t kMinus1152 = 0xE480E480u;
    pa = hadd2_u32(prmt_u32(u, kHigh, 0x4240u), kMinus1152);
    pb = hadd2_u32(prmt_u32(u, kHigh, 0x4341u), kMinus1152);
}

// ------------------------------------------------------------------ activation fragments
//
// Activation fragment layout. For one row v[K] (a token's activations,
// already multiplied by the group's power-of-two factor) and one 64-wide
// group, the B operands of the four MMA steps m = 0..3 for quad lane q are
//   b0(m, q) = half2(v[k0], v[k1]),  b1(m, q) = half2(v[k2], v[k3])
// with the k's of the weight format's register order:
//   int4: kA = 16q + 8(m/2) + 2(m%2); (k0, k1, k2, k3) = (kA, kA+4, kA+1, kA+5)
//   int8: kA = 16q + 4m;              (k0, k1, k2, k3) = (kA, kA+2, kA+1, kA+3)
// Each value is split into hi = fp16(v) and lo = fp16(v - hi) ("part" 0 / 1).
// A group of one row is 16 units of 16 bytes (256 bytes):
//   unit (mh, q, part), index (mh*4 + q)*2 + part, holds
//   { b0(2mh, q), b1(2mh, q), b0(2mh+1, q), b1(2mh+1, q) } of that part,
// so a lane fetches the operands of two MMA steps with one 16-byte load, and
// the 32 lanes of a warp read 512 contiguous bytes (no bank conflicts).

template <bool kInt8>
__device__ __forceinline__ void frag_ks(int m, int q, int &k0, int &k1, int &k2, int &k3) {
    if (!kInt8) {
        const int kA = 16 * q + 8 * (m >> 1) + 2 * (m & 1);
        k0 = kA; k1 = kA + 4; k2 = kA + 1; k3 = kA + 5;
    } else {
        const int kA = 16 * q + 4 * m;
        k0 = kA; k1 = kA + 2; k2 = kA + 1; k3 = kA + 3;
    }
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

__device__ __forceinline__ __half split_part(float v, int part) {
    const __half h = __float2half_rn(v);
    return part ? __float2half_rn(v - __half2float(h)) : h;
}

// Unit u (0..15) of a group, from its 64 scaled values v[0..63].
template <bool kInt8>
__device__ __forceinline__ uint4 make_unit(const float *v, int u) {
    const int part = u & 1, q = (u >> 1) & 3, mh = u >> 3;
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        int k0, k1, k2, k3;
        frag_ks<kInt8>(2 * mh + i, q, k0, k1, k2, k3);
        r[2 * i] = pack_half2(split_part(v[k0], part), split_part(v[k1], part));
        r[2 * i + 1] = pack_half2(split_part(v[k2], part), split_part(v[k3], part));
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Unit u of a group in the tensor-map kernel's int4 form: as make_unit<false>
// with the values at k2, k3 (the ones multiplied by the high nibbles' 16 n)
// divided by 16 before the hi/lo split.
__device__ __forceinline__ uint4 make_unit_s(const float *v, int u) {
    const int part = u & 1, q = (u >> 1) & 3, mh = u >> 3;
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        int k0, k1, k2, k3;
        frag_ks<false>(2 * mh + i, q, k0, k1, k2, k3);
        r[2 * i] = pack_half2(split_part(v[k0], part), split_part(v[k1], part));
        r[2 * i + 1] = pack_half2(split_part(v[k2] * 0.0625f, part),
                                  split_part(v[k3] * 0.0625f, part));
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Initial accumulator of a group in that form: -8 * 2^-24 * sum of the
// group's 64 scaled values (the offset of nibble - 8, folded out of the
// weights). `sum` is the fp32 sum of the scaled values.
__device__ __forceinline__ float offset_init(float sum) { return sum * -0x1p-21f; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Power-of-two exponent that maps max|v| into [2^13, 2^14); 0 for an all-zero group.
__device__ __forceinline__ int split_exponent(float amax) {
    if (!(amax > 0.0f) || !isfinite(amax)) return 0;
    int e;
    frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
    int s = 14 - e;
    return s > 126 ? 126 : (s < -126 ? -126 : s);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// ------------------------------------------------------------------ tile compute
//
// One warp computes a 16-row tile for up to 4*NB tokens. Lane (gid = lane/4,
// q = lane%4) owns rows gid and gid+8; after the MMAs it holds, for token
// 4*nb + q, rows gid (d[0] + d[1]: hi + lo columns) and gid+8 (d[2] + d[3]).
// bu[nb][mh]: the lane's B unit for MMA steps 2mh, 2mh+1 of block nb (token
// 4*nb + gid/2, clamped to the last token, part gid & 1).

template <int NB>
__device__ __forceinline__ void tile_group_int4(uint2 w0, uint2 w8, const uint4 (&bu)[NB][2],
                                                float d[NB][4]) {
    uint32_t p0[4], p8[4], a[4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) d[nb][0] = d[nb][1] = d[nb][2] = d[nb][3] = 0.0f;
#pragma unroll
    for (int mh = 0; mh < 2; ++mh) {
        uint4 b[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) b[nb] = bu[nb][mh];
        dequant_int4_word(mh ? w0.y : w0.x, p0);
        dequant_int4_word(mh ? w8.y : w8.x, p8);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            a[0] = p0[2 * mm];
            a[1] = p8[2 * mm];
            a[2] = p0[2 * mm + 1];
            a[3] = p8[2 * mm + 1];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
                mma_16816(d[nb], a, mm ? b[nb].z : b[nb].x, mm ? b[nb].w : b[nb].y);
        }
    }
}

// The same tile in the tensor-map kernel's int4 form (dequant_int4_word_s):
// the token columns (hi) start from cinit[nb] (offset_init of the lane's
// token 4nb+q), so d[nb] ends as 2^-24 * sum (nibble - 8) * v.
template <int NB>
__device__ __forceinline__ void tile_group_int4s(uint2 w0, uint2 w8, const uint4 (&bu)[NB][2],
                                                 const float (&cinit)[NB], float d[NB][4]) {
    uint32_t p0[4], p8[4], a[4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        d[nb][0] = d[nb][2] = cinit[nb];
        d[nb][1] = d[nb][3] = 0.0f;
    }
#pragma unroll
    for (int mh = 0; mh < 2; ++mh) {
        uint4 b[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) b[nb] = bu[nb][mh];
        dequant_int4_word_s(mh ? w0.y : w0.x, p0);
        dequant_int4_word_s(mh ? w8.y : w8.x, p8);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            a[0] = p0[2 * mm];
            a[1] = p8[2 * mm];
            a[2] = p0[2 * mm + 1];
            a[3] = p8[2 * mm + 1];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
                mma_16816(d[nb], a, mm ? b[nb].z : b[nb].x, mm ? b[nb].w : b[nb].y);
        }
    }
}

// Two tiles of the same 16 rows' shape (A: w0, w8; B: v0, v8) against the
// same activation fragments, in the tensor-map kernel's int4 form: the two
// tiles' MMA chains interleave, and each B fragment serves both.
template <int NB>
__device__ __forceinline__ void tile2_group_int4s(uint2 w0, uint2 w8, uint2 v0, uint2 v8,
                                                  const uint4 (&bu)[NB][2],
                                                  const float (&cinit)[NB], float dA[NB][4],
                                                  float dB[NB][4]) {
    uint32_t p0[4], p8[4], q0[4], q8[4], a[4], b[4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        dA[nb][0] = dA[nb][2] = dB[nb][0] = dB[nb][2] = cinit[nb];
        dA[nb][1] = dA[nb][3] = dB[nb][1] = dB[nb][3] = 0.0f;
    }
#pragma unroll
    for (int mh = 0; mh < 2; ++mh) {
        uint4 bv[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) bv[nb] = bu[nb][mh];
        dequant_int4_word_s(mh ? w0.y : w0.x, p0);
        dequant_int4_word_s(mh ? w8.y : w8.x, p8);
        dequant_int4_word_s(mh ? v0.y : v0.x, q0);
        dequant_int4_word_s(mh ? v8.y : v8.x, q8);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            a[0] = p0[2 * mm]; a[1] = p8[2 * mm]; a[2] = p0[2 * mm + 1]; a[3] = p8[2 * mm + 1];
            b[0] = q0[2 * mm]; b[1] = q8[2 * mm]; b[2] = q0[2 * mm + 1]; b[3] = q8[2 * mm + 1];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                mma_16816(dA[nb], a, mm ? bv[nb].z : bv[nb].x, mm ? bv[nb].w : bv[nb].y);
                mma_16816(dB[nb], b, mm ? bv[nb].z : bv[nb].x, mm ? bv[nb].w : bv[nb].y);
            }
        }
    }
}

// int8: 16 bytes of row gid (w0) and of row gid+8 (w8); MMA step m uses word m.
template <int NB>
__device__ __forceinline__ void tile_group_int8(uint4 w0, uint4 w8, const uint4 (&bu)[NB][2],
                                                float d[NB][4]) {
    const uint32_t r0[4] = {w0.x, w0.y, w0.z, w0.w};
    const uint32_t r8[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) d[nb][0] = d[nb][1] = d[nb][2] = d[nb][3] = 0.0f;
#pragma unroll
    for (int mh = 0; mh < 2; ++mh) {
        uint4 b[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) b[nb] = bu[nb][mh];
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            const int m = 2 * mh + mm;
            uint32_t a[4];
            dequant_int8_word(r0[m], a[0], a[2]);
            dequant_int8_word(r8[m], a[1], a[3]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
                mma_16816(d[nb], a, mm ? b[nb].z : b[nb].x, mm ? b[nb].w : b[nb].y);
        }
    }
}

}  // namespace qmv
