// qmv_gemv.cu - dense int4-gs64 and int8-row GEMV for decode (S tokens).
//
// colibri PR #418 "Vulkan backend: expert tier + dense + MLA attention on any
// Vulkan 1.2 GPU", commits "opt-in Vulkan int4/int8 quantized GEMV" (int4 as
// nibble - 8, int8 with a per-row scale) and "grouped scales in the Vulkan
// kernels" (fmt 4: one scale per 64 inputs on the group partial).
//
// Grid: one CTA per 64 output rows (four 16-row warp tiles). Every CTA
// rescales its tokens by a power of two (max |x| into [2^13, 2^14)), splits
// them into fp16 hi/lo fragment cells in shared memory, and streams its rows
// through the register ring of qmv_rows.cuh. Any K that is a multiple of 64
// is handled: the activation cells are staged chunk by chunk.
#include "qmv_internal.h"
#include "qmv_rows.cuh"

namespace qmv {

namespace {

// Stages fragment cells straight from fp32 activation rows (dense GEMV).
template <bool kInt8>
struct StageFromFp32 {
    const float *x;        // [ntok][K]
    const float *mul;      // shared: 2^sigma per token
    int ntok, K;
    uint4 *cells;
    __device__ __forceinline__ void operator()(int gc, int ng) const {
        const int total = ng * 16 * ntok;
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int s = idx % ntok;
            const int r = idx / ntok;
            const int q = r & 3, m = (r >> 2) & 3, gl = r >> 4;
            int k0, k1, k2, k3;
            frag_ks<kInt8>(gc + gl, m, q, k0, k1, k2, k3);
            const float *xs = x + (size_t)s * K;
            const float f = mul[s];
            cells[idx] = make_cell(xs[k0] * f, xs[k1] * f, xs[k2] * f, xs[k3] * f);
        }
    }
};

template <int NB, bool kInt8>
__device__ __forceinline__ void dense_body(const uint8_t *w, const float *scales, int N, int K,
                                           const float *x, float *y, int ntok,
                                           WeightRing<kInt8> &ring, uint4 *cells, float *s_mul,
                                           float *s_fac) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int row0 = blockIdx.x * (16 * kWarps) + warp * 16;

    StageFromFp32<kInt8> stage{x, s_mul, ntok, K, cells};
    float acc[NB][2];
    rows_mainloop<NB, kInt8>(ring, cells, ntok, stage, acc);

    const int rA = row0 + gid, rB = row0 + gid + 8;
    float rsA = 1.0f, rsB = 1.0f;
    if constexpr (kInt8) {
        rsA = rA < N ? scales[rA] : 0.0f;
        rsB = rB < N ? scales[rB] : 0.0f;
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int t = 4 * nb + q;
        if (t < ntok) {
            const float f = s_fac[t];
            if (rA < N) y[(size_t)t * N + rA] = acc[nb][0] * f * rsA;
            if (rB < N) y[(size_t)t * N + rB] = acc[nb][1] * f * rsB;
        }
    }
}

template <bool kInt8>
__global__ void __launch_bounds__(kCtaThreads)
    k_dense(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
            const float *__restrict__ x, float *__restrict__ y, int ntok) {
    extern __shared__ uint4 cells[];
    __shared__ float s_mul[kMaxTok], s_fac[kMaxTok];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const int row0 = blockIdx.x * (16 * kWarps) + warp * 16;
    const int rA = min(row0 + gid, N - 1), rB = min(row0 + gid + 8, N - 1);
    const size_t rowBytes = kInt8 ? (size_t)K : (size_t)K / 2;

    // Start streaming weights before anything else.
    WeightRing<kInt8> ring;
    ring.init(w + (size_t)rA * rowBytes, w + (size_t)rB * rowBytes,
              kInt8 ? nullptr : scales + (size_t)rA * G, kInt8 ? nullptr : scales + (size_t)rB * G,
              G, q);
    ring.prologue();

    // Per-token power-of-two rescale from the row maximum.
    for (int s = warp; s < ntok; s += kWarps) {
        float m = 0.0f;
        for (int k = lane; k < K; k += 32) m = fmaxf(m, fabsf(x[(size_t)s * K + k]));
        m = warp_max(m);
        if (lane == 0) {
            const int e = split_exponent(m);
            s_mul[s] = ldexpf(1.0f, e);
            s_fac[s] = ldexpf(1.0f, -e);
        }
    }
    // (rows_mainloop begins with a barrier, which publishes s_mul / s_fac.)

    if (ntok <= 4)
        dense_body<1, kInt8>(w, scales, N, K, x, y, ntok, ring, cells, s_mul, s_fac);
    else if (ntok <= 8)
        dense_body<2, kInt8>(w, scales, N, K, x, y, ntok, ring, cells, s_mul, s_fac);
    else
        dense_body<4, kInt8>(w, scales, N, K, x, y, ntok, ring, cells, s_mul, s_fac);
}

template <bool kInt8>
cudaError_t launch_dense(const uint8_t *w, const float *scales, int N, int K, const float *x,
                         float *y, int S, cudaStream_t st) {
    const int grid = (N + 16 * kWarps - 1) / (16 * kWarps);
    for (int s0 = 0; s0 < S; s0 += kMaxTok) {
        const int ntok = S - s0 < kMaxTok ? S - s0 : kMaxTok;
        const size_t smem = (size_t)chunk_groups(ntok) * 256 * ntok;
        k_dense<kInt8><<<grid, kCtaThreads, smem, st>>>(w, scales, N, K, x + (size_t)s0 * K,
                                                        y + (size_t)s0 * N, ntok);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_dense_int4(const uint8_t *wq, const float *scales, int N, int K,
                              const float *x, float *y, int S, cudaStream_t st) {
    return launch_dense<false>(wq, scales, N, K, x, y, S, st);
}

cudaError_t launch_dense_int8(const int8_t *w, const float *row_scale, int N, int K,
                              const float *x, float *y, int S, cudaStream_t st) {
    return launch_dense<true>(reinterpret_cast<const uint8_t *>(w), row_scale, N, K, x, y, S, st);
}

}  // namespace qmv
