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
// Each warp walks output rows i, i + W, ... (W warps in the grid). Lane l
// takes, per step, group 8*step + l/4 and its low-plane word l%4 (16
// elements) with the matching 16 high bits; the 16 values are decoded once,
// as exact fp32, and used for every token of the pass. The words and scales
// of the warp's next block of 8 steps (the rest of this row or the start of
// its next row) are requested before the current block is computed, so a
// warp always has one row's loads in flight. Each lane multiplies its
// word's partial sum by the group scale and keeps its own sum; the lanes'
// sums are reduced when the row is done. All arithmetic is fp32 (products of
// a small integer and an fp32 x are exact). Tokens go in passes of
// NT = min(S, 4).
//
// A lane's 16 elements are x[16 l .. 16 l + 15] (relative to the step's 512),
// so each of its four 16-byte x reads has lanes 64 bytes apart: read from L1
// that is 16 cache lines per instruction. The CTA therefore first copies the
// pass's x rows into shared memory, transposed within each block of 128
// 16-byte chunks (one step): chunk 4 l + q of a block is stored at 32 q + l.
// A lane's four reads are then 512 bytes apart from one base, and the lanes
// of each read are consecutive (4 wavefronts, the minimum for 512 bytes).
// When one token's x does not fit the shared-memory budget (K > 24576) x is
// read from global memory instead.
#include <cuda_fp16.h>

#include <algorithm>

#include "qmv_internal.h"
#include "qmv_launch.cuh"

namespace qmv {

namespace {

constexpr int kI3Warps = 8;
constexpr int kI3Steps = 8;  // steps (8 groups each) whose words are requested at once
constexpr int kI3SmemX = 96 * 1024;  // shared-memory budget for the staged x rows

// Shared-memory slot of 16-byte x chunk c (see above), and the chunks a
// token takes there (a whole number of 128-chunk blocks).
__device__ __forceinline__ int i3_slot(int c) {
    return (c & ~127) | ((c & 3) << 5) | ((c & 127) >> 2);
}
__host__ __device__ __forceinline__ int i3_chunks(int K) { return ((K / 4 + 127) / 128) * 128; }

// A block of one row: kI3Steps steps of this lane's words and group scales.
struct I3Block {
    uint32_t lo[kI3Steps], hi[kI3Steps];
    float sc[kI3Steps];
};

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

// Requests row i's words and scales for groups gb .. gb + 8 kI3Steps - 1
// (zeros past the row's last group).
__device__ __forceinline__ void i3_load(const uint8_t *__restrict__ wq,
                                        const float *__restrict__ scales, int i, int G, int gb,
                                        I3Block &u) {
    const int lane = threadIdx.x & 31, w = lane & 3;
    const uint8_t *row = wq + (size_t)i * G * 24;
    const float *srow = scales + (size_t)i * G;
#pragma unroll
    for (int st = 0; st < kI3Steps; ++st) {
        const int g = gb + 8 * st + (lane >> 2);
        u.lo[st] = u.hi[st] = 0u;
        u.sc[st] = 0.f;
        if (g < G) {
            const uint8_t *gp = row + (size_t)g * 24;
            u.lo[st] = __ldg(reinterpret_cast<const uint32_t *>(gp) + w);
            u.hi[st] = __ldg(reinterpret_cast<const uint32_t *>(gp + 16) + (w >> 1));
            u.sc[st] = __ldg(srow + g);
        }
    }
}

// Adds the lane's scaled word partials of the block for tokens 0 .. nt - 1
// to acc.
// xt: the pass's x rows, in shared memory (i3_chunks(K) chunks a token, laid
// out as above) when STAGED, else in global memory (K floats a token).
template <int NT, bool STAGED>
__device__ __forceinline__ void i3_compute(const I3Block &u, int G, int gb,
                                           const float *__restrict__ xt, int K, int nt,
                                           float (&acc)[NT]) {
    const int lane = threadIdx.x & 31, w = lane & 3;
#pragma unroll
    for (int st = 0; st < kI3Steps; ++st) {
        const int g = gb + 8 * st + (lane >> 2);
        float part[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) part[t] = 0.f;
        if (g < G) {
            float v[16];
            decode16(u.lo[st], u.hi[st] >> (16 * (w & 1)), v);
            // the lane's first x chunk: 16 g + 4 w, global; 32 q + lane in the
            // step's shared block (gb is a multiple of 64, so block gb / 8 + st)
            const int c0 = STAGED ? (((gb >> 3) + st) << 7) + lane : 16 * g + 4 * w;
            const int ct = STAGED ? i3_chunks(K) : K / 4;  // chunks a token
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                if (t < nt) {
                    const float4 *xp = reinterpret_cast<const float4 *>(xt) + (size_t)t * ct + c0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 xv = STAGED ? xp[32 * q] : __ldg(xp + q);
                        part[t] = fmaf(v[4 * q + 0], xv.x, part[t]);
                        part[t] = fmaf(v[4 * q + 1], xv.y, part[t]);
                        part[t] = fmaf(v[4 * q + 2], xv.z, part[t]);
                        part[t] = fmaf(v[4 * q + 3], xv.w, part[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = fmaf(u.sc[st], part[t], acc[t]);
    }
}

template <int NT, bool STAGED>
__global__ void __launch_bounds__(32 * kI3Warps)
    k_int3_gemv(const uint8_t *__restrict__ wq, const float *__restrict__ scales, int N, int K,
                const float *__restrict__ x, float *__restrict__ y, int S) {
    extern __shared__ float4 xs4[];
    const int lane = threadIdx.x & 31;
    const int i0 = blockIdx.x * kI3Warps + (threadIdx.x >> 5), nw = gridDim.x * kI3Warps;
    const int G = K / 64, span = 8 * kI3Steps, nb = (G + span - 1) / span;  // blocks per row
    const int kc = K / 4, kcs = i3_chunks(K);  // x chunks a token: in x, staged
    for (int t0 = 0; t0 < S; t0 += NT) {
        const int nt = min(NT, S - t0);
        I3Block cur, nxt;
        if (i0 < N) i3_load(wq, scales, i0, G, 0, cur);  // requested before x is staged
        const float *xt = x + (size_t)t0 * K;
        if (STAGED) {
            __syncthreads();  // every warp is done with the previous pass's x
            const float4 *src = reinterpret_cast<const float4 *>(xt);
            for (int c = threadIdx.x; c < nt * kc; c += blockDim.x) {
                const int t = c / kc, cc = c - t * kc;
                xs4[t * kcs + i3_slot(cc)] = __ldg(src + c);
            }
            __syncthreads();
            xt = reinterpret_cast<const float *>(xs4);
        }
        if (i0 >= N) continue;
        float acc[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[t] = 0.f;
        int i = i0, b = 0;
        for (;;) {
            int ni = i, nbk = b + 1;
            if (nbk == nb) {
                ni = i + nw;
                nbk = 0;
            }
            const bool more = ni < N;
            if (more) i3_load(wq, scales, ni, G, nbk * span, nxt);
            i3_compute<NT, STAGED>(cur, G, b * span, xt, K, nt, acc);
            if (nbk == 0) {  // row i is done
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    float a = acc[t];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                    if (lane == 0 && t < nt) y[(size_t)(t0 + t) * N + i] = a;
                    acc[t] = 0.f;
                }
            }
            if (!more) break;
            cur = nxt;
            i = ni;
            b = nbk;
        }
    }
}

template <int NT, bool STAGED>
cudaError_t launch_int3_nt(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                           float *y, int S, cudaStream_t st) {
    const size_t smem = STAGED ? (size_t)NT * i3_chunks(K) * 16 : 0;
    cudaError_t e = set_smem(k_int3_gemv<NT, STAGED>, smem);
    if (e != cudaSuccess) return e;
    const int rows_blocks = (N + kI3Warps - 1) / kI3Warps;
    const int resident =
        sm_count() * max_ctas_per_sm(k_int3_gemv<NT, STAGED>, 32 * kI3Warps, smem);
    return launch(k_int3_gemv<NT, STAGED>, dim3(std::min(rows_blocks, resident)),
                  dim3(32 * kI3Warps), smem, st, false, wq, scales, N, K, x, y, S);
}

}  // namespace

cudaError_t launch_gemv_int3(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                             float *y, int S, cudaStream_t st) {
    if (int3_one_launch(wq, K, S))  // a few tokens: the warp-MMA single launch
        return launch_gemv_int3_mma(wq, scales, N, K, x, y, S, st);
    // tokens per pass: up to 4, as many as the staged x rows allow
    const int fit = kI3SmemX / (i3_chunks(K) * 16);
    if (fit < 1) {
        switch (std::min(S, 4)) {
            case 1: return launch_int3_nt<1, false>(wq, scales, N, K, x, y, S, st);
            case 2: return launch_int3_nt<2, false>(wq, scales, N, K, x, y, S, st);
            case 3: return launch_int3_nt<3, false>(wq, scales, N, K, x, y, S, st);
            default: return launch_int3_nt<4, false>(wq, scales, N, K, x, y, S, st);
        }
    }
    switch (std::min(std::min(S, 4), fit)) {
        case 1: return launch_int3_nt<1, true>(wq, scales, N, K, x, y, S, st);
        case 2: return launch_int3_nt<2, true>(wq, scales, N, K, x, y, S, st);
        case 3: return launch_int3_nt<3, true>(wq, scales, N, K, x, y, S, st);
        default: return launch_int3_nt<4, true>(wq, scales, N, K, x, y, S, st);
    }
}

}  // namespace qmv
