// qmv_gemv.cu - dense int4-gs64 and int8-row GEMV for decode (S tokens), and
// the activation split kernel shared with the MoE path.
//
// colibri PR #418 "Vulkan backend: expert tier + dense + MLA attention on any
// Vulkan 1.2 GPU", commits "opt-in Vulkan int4/int8 quantized GEMV" (int4 as
// nibble - 8, int8 with a per-row scale) and "grouped scales in the Vulkan
// kernels" (fmt 4: one scale per 64 inputs on the group partial).
//
// Two launches per call: k_split turns the S activation rows into fp16 hi/lo
// fragment cells with one power-of-two factor per 64-wide group; k_dense
// (launched with programmatic dependent launch) starts streaming its weight
// rows at once and waits for the cells only before its first MMA.
#include <mutex>

#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_rows.cuh"

namespace qmv {

namespace {

constexpr int kDenseWarps = 4;                 // 64-row items
constexpr int kDenseStages = 8;                // weight stages per warp ring
constexpr int kDenseRing = kDenseStages * kStageBytes;
constexpr int kDenseBudget = 32 * 1024;

// ------------------------------------------------------------------ split

// One CTA per activation row; warp w converts groups w, w + nwarps, ...:
// max |v| of the group -> exponent -> 16 fragment cells and the factor.
template <bool kInt8>
__global__ void __launch_bounds__(256)
    k_split(const float *__restrict__ v, int K, uint4 *__restrict__ cells,
            float *__restrict__ fac) {
    __shared__ float buf[8][64];
    pdl_trigger();  // the consumer may start streaming its weights at once
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const float *row = v + (size_t)r * K;
    for (int g = warp; g < G; g += blockDim.x >> 5) {
        const float a = row[g * kGroup + lane], b = row[g * kGroup + 32 + lane];
        const int e = split_exponent(warp_max(fmaxf(fabsf(a), fabsf(b))));
        const float mul = ldexpf(1.0f, e);
        buf[warp][lane] = a * mul;
        buf[warp][32 + lane] = b * mul;
        __syncwarp();
        if (lane < 16) cells[((size_t)r * G + g) * 16 + lane] = make_unit<kInt8>(buf[warp], lane);
        if (lane == 0) fac[(size_t)r * G + g] = ldexpf(1.0f, -e);
        __syncwarp();
    }
}

// ------------------------------------------------------------------ dense

template <int NB, bool kInt8, class WS>
__device__ __forceinline__ void dense_item(WS &ws, int item, int row0, int N, const float *scales,
                                           float *y, uint4 *cells, float *fac, int ntok, bool reuse,
                                           const StageCells &stage) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    float acc[NB][2];
    run_item<NB, kInt8>(ws, item, cells, fac, kDenseBudget, ntok, reuse, stage, acc);
    const int rA = row0 + gid, rB = row0 + gid + 8;
    float ra = 1.0f, rb = 1.0f;
    if constexpr (kInt8) {
        ra = rA < N ? scales[rA] : 0.0f;
        rb = rB < N ? scales[rB] : 0.0f;
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int t = 4 * nb + q;
        if (t < ntok) {
            if (rA < N) y[(size_t)t * N + rA] = acc[nb][0] * ra;
            if (rB < N) y[(size_t)t * N + rB] = acc[nb][1] * rb;
        }
    }
}

template <bool kInt8>
__global__ void __launch_bounds__(32 * kDenseWarps)
    k_dense(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
            const uint4 *__restrict__ xcells, const float *__restrict__ xfac,
            float *__restrict__ y, int ntok) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_rows[kMaxTok];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int ns = (G + Fmt<kInt8>::kGPS - 1) / Fmt<kInt8>::kGPS;
    const int nitems = (N + 16 * kDenseWarps - 1) / (16 * kDenseWarps);
    const int i0 = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);
    const size_t rowBytes = kInt8 ? (size_t)K : (size_t)K / 2;

    auto tile = [=](int item, int wp) {
        int row0 = (i0 + item) * 16 * kDenseWarps + 16 * wp;
        int nrows = N - row0;
        if (nrows <= 0) { row0 = N - 1; nrows = 1; }
        return TileSrc{w + (size_t)row0 * rowBytes, kInt8 ? nullptr : scales + (size_t)row0 * G,
                       rowBytes, nrows};
    };
    WarpStream<kInt8, kDenseStages, decltype(tile)> ws{smem + warp * kDenseRing, tile, G, ns, (i1 - i0) * ns,
                                         0, warp, lane};
    ws.prologue();  // weights are call inputs: safe to read before the wait

    pdl_wait();     // cells and factors come from k_split
    pdl_trigger();
    if (threadIdx.x < kMaxTok) s_rows[threadIdx.x] = threadIdx.x;
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kDenseWarps * kDenseRing);
    float *fac = reinterpret_cast<float *>(smem + kDenseWarps * kDenseRing + kDenseBudget);
    const StageCells stage{xcells, xfac, s_rows, ntok, G};

    for (int it = 0; it < i1 - i0; ++it) {
        const int row0 = (i0 + it) * 16 * kDenseWarps + 16 * warp;
        const bool reuse = it > 0;
        if (ntok <= 4)
            dense_item<1, kInt8>(ws, it, row0, N, scales, y, cells, fac, ntok, reuse, stage);
        else
            dense_item<2, kInt8>(ws, it, row0, N, scales, y, cells, fac, ntok, reuse, stage);
    }
    cp_async_wait<0>();
}

template <bool kInt8>
cudaError_t launch_dense(const uint8_t *w, const float *scales, int N, int K, const float *x,
                         float *y, int S, void *xcells, float *xfac, cudaStream_t st) {
    const size_t smem = engine_smem(kDenseWarps, kDenseStages, kDenseBudget, 0);
    cudaError_t e = set_smem(k_dense<kInt8>, smem);
    if (e != cudaSuccess) return e;
    const int nitems = (N + 16 * kDenseWarps - 1) / (16 * kDenseWarps);
    const int slots = sm_count() * max_ctas_per_sm(k_dense<kInt8>, 32 * kDenseWarps, smem);
    const int grid = nitems < slots ? nitems : slots;
    e = launch(k_split<kInt8>, dim3(S), dim3(256), 0, st, false, x, K,
               static_cast<uint4 *>(xcells), xfac);
    for (int s0 = 0; s0 < S && e == cudaSuccess; s0 += kMaxTok) {
        const int ntok = S - s0 < kMaxTok ? S - s0 : kMaxTok;
        e = launch(k_dense<kInt8>, dim3(grid), dim3(32 * kDenseWarps), smem, st, true, w, scales, N,
                   K, static_cast<const uint4 *>(xcells) + (size_t)s0 * (K / kGroup) * 16,
                   xfac + (size_t)s0 * (K / kGroup), y + (size_t)s0 * N, ntok);
    }
    return e;
}

}  // namespace

cudaError_t launch_split(const float *v, int R, int K, void *cells, float *fac, cudaStream_t st) {
    if (R == 0) return cudaSuccess;
    return launch(k_split<false>, dim3(R), dim3(256), 0, st, false, v, K,
                  static_cast<uint4 *>(cells), fac);
}

size_t dense_scratch_bytes(int K, int S) { return (size_t)S * K * 4 + (size_t)S * (K / kGroup) * 4; }

cudaError_t launch_dense_int4(const uint8_t *wq, const float *scales, int N, int K,
                              const float *x, float *y, int S, void *scratch, cudaStream_t st) {
    float *fac = reinterpret_cast<float *>(static_cast<char *>(scratch) + (size_t)S * K * 4);
    return launch_dense<false>(wq, scales, N, K, x, y, S, scratch, fac, st);
}

cudaError_t launch_dense_int8(const int8_t *w, const float *row_scale, int N, int K,
                              const float *x, float *y, int S, void *scratch, cudaStream_t st) {
    float *fac = reinterpret_cast<float *>(static_cast<char *>(scratch) + (size_t)S * K * 4);
    return launch_dense<true>(reinterpret_cast<const uint8_t *>(w), row_scale, N, K, x, y, S,
                              scratch, fac, st);
}

}  // namespace qmv
