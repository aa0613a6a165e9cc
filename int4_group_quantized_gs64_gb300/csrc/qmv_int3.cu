// qmv_int3.cu - dense GEMV over int3-g64 two-plane rows.
//
// Math (colibri PR #418, the fmt-5 commit: a 24-byte-per-64-group layout
// whose lanes stride the 16-value low-plane words, the high-plane word
// pre-shifted so that its bits start at bit 0, and each word's partial dot
// multiplied by its group scale): per 64-group, bytes 0..15 hold 2 low bits
// per element (element e at bits 2(e%4) of byte e/4, i.e. 16 elements to a
// little-endian 32-bit word), bytes 16..23 one high bit per element (bit e%8
// of byte 16 + e/8); code = low | high << 2, value = code - 4; one fp32 scale
// per group:
//     y[t][i] = sum_g s[i][g] * sum_{k in g} (code(i,k) - 4) * x[t][k]
//
// One warp per output row. Lane l of a warp takes, per step, group
// 8*step + l/4 and its low-plane word l%4 (16 elements) together with the
// matching 16 high bits; the 16 values are decoded once, as exact fp32, and
// used for every token. The partials of a group's four lanes are added with
// two shuffles, scaled once, and the lanes' sums are reduced at the end; all
// arithmetic is fp32 (products of a small integer and an fp32 x are exact).
#include <cuda_fp16.h>

#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace qmv {

namespace {

constexpr int kI3Warps = 8;
constexpr int kI3Tok = 4;    // tokens per pass over a row's weights
constexpr int kI3Steps = 8;  // steps (8 groups each) whose words are loaded at once

// Exact (code - 4) as fp32 for the 16 elements of a low-plane word `lo` and
// their high bits in bits 0..15 of `hi`, decoded in pairs (j, j + 8): their
// low bits sit 16 apart in `lo`, and a byte permute spreads the high bits the
// same way. OR-ing a pair's 3-bit codes into the mantissas of fp16 1024.0
// gives (1024 + code) exactly; subtracting 1028 leaves code - 4.
__device__ __forceinline__ void decode16(uint32_t lo, uint32_t hi, float (&v)[16]) {
    uint32_t hs;
    asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(hs) : "r"(hi));  // bytes (h0, 0, h1, 0)
    hs <<= 2;                                                 // element j's high bit at j + 2
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t t, r;
        asm("lop3.b32 %0, %1, 0x00030003, 0x64006400, 0xEA;" : "=r"(t) : "r"(lo >> (2 * j)));
        asm("lop3.b32 %0, %1, %2, 0x00040004, 0xF8;" : "=r"(r) : "r"(t), "r"(hs >> j));
        const __half2 p = __hadd2(*reinterpret_cast<const __half2 *>(&r),
                                  __halves2half2(__float2half(-1028.0f), __float2half(-1028.0f)));
        const float2 f = __half22float2(p);
        v[j] = f.x;
        v[j + 8] = f.y;
    }
}

__global__ void __launch_bounds__(32 * kI3Warps)
    k_int3_gemv(const uint8_t *__restrict__ wq, const float *__restrict__ scales, int N, int K,
                const float *__restrict__ x, float *__restrict__ y, int S) {
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * kI3Warps + (threadIdx.x >> 5);
    if (i >= N) return;
    const int G = K / 64, w = lane & 3;
    const uint8_t *row = wq + (size_t)i * G * 24;
    const float *srow = scales + (size_t)i * G;
    for (int t0 = 0; t0 < S; t0 += kI3Tok) {
        const int nt = min(kI3Tok, S - t0);
        float acc[kI3Tok] = {0.f, 0.f, 0.f, 0.f};
        for (int gb = 0; gb < G; gb += 8 * kI3Steps) {
            // the words of up to kI3Steps steps are requested before any is used
            uint32_t lo[kI3Steps], hw[kI3Steps];
#pragma unroll
            for (int st = 0; st < kI3Steps; ++st) {
                const int g = gb + 8 * st + (lane >> 2);
                lo[st] = hw[st] = 0u;
                if (g < G) {
                    const uint8_t *gp = row + (size_t)g * 24;
                    lo[st] = __ldg(reinterpret_cast<const uint32_t *>(gp) + w);
                    hw[st] = __ldg(reinterpret_cast<const uint32_t *>(gp + 16) + (w >> 1));
                }
            }
#pragma unroll
            for (int st = 0; st < kI3Steps; ++st) {
                const int g = gb + 8 * st + (lane >> 2);
                float part[kI3Tok] = {0.f, 0.f, 0.f, 0.f};
                if (g < G) {
                    float v[16];
                    decode16(lo[st], hw[st] >> (16 * (w & 1)), v);
                    const int k0 = g * 64 + 16 * w;
#pragma unroll
                    for (int t = 0; t < kI3Tok; ++t) {
                        if (t < nt) {
                            const float4 *xp =
                                reinterpret_cast<const float4 *>(x + (size_t)(t0 + t) * K + k0);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float4 xv = __ldg(xp + q);
                                part[t] = fmaf(v[4 * q + 0], xv.x, part[t]);
                                part[t] = fmaf(v[4 * q + 1], xv.y, part[t]);
                                part[t] = fmaf(v[4 * q + 2], xv.z, part[t]);
                                part[t] = fmaf(v[4 * q + 3], xv.w, part[t]);
                            }
                        }
                    }
                }
                const float sc = g < G ? __ldg(srow + g) : 0.f;
#pragma unroll
                for (int t = 0; t < kI3Tok; ++t) {
                    // the group's four word partials, then its scale (one lane adds it)
                    float p = part[t] + __shfl_xor_sync(0xffffffffu, part[t], 1);
                    p += __shfl_xor_sync(0xffffffffu, p, 2);
                    if (w == 0) acc[t] = fmaf(sc, p, acc[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kI3Tok; ++t) {
            float a = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0 && t < nt) y[(size_t)(t0 + t) * N + i] = a;
        }
    }
}

}  // namespace

cudaError_t launch_gemv_int3(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                             float *y, int S, cudaStream_t st) {
    return launch(k_int3_gemv, dim3((N + kI3Warps - 1) / kI3Warps), dim3(32 * kI3Warps), 0, st,
                  false, wq, scales, N, K, x, y, S);
}

}  // namespace qmv
