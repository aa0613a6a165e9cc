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

// Grid (rows, ceil(G / 8)): warp w of CTA (r, c) converts group 8c + w of
// activation row r (one group a warp, so the rows' groups convert in
// parallel): max |v| of the group -> exponent -> 16 fragment cells and the
// factor. kSub: the tensor-map kernel's int4 form (make_unit_s), with a
// record (factor, offset_init) per group, fac [rows][G][2]; else fac
// [rows][G]. CTA (0, 0) also clears zero[0 .. nzero) (the caller's status
// word and split counters), which the next kernel reads only after waiting
// for this one.
template <bool kInt8, bool kSub = false>
__global__ void __launch_bounds__(256)
    k_split(const float *__restrict__ v, int K, uint4 *__restrict__ cells,
            float *__restrict__ fac, int32_t *zero, int nzero) {
    __shared__ float buf[8][64];
    pdl_trigger();  // the consumer may start streaming its weights at once
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (zero && r == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
    const int G = K / kGroup;
    const float *row = v + (size_t)r * K;
    const int g = blockIdx.y * (blockDim.x >> 5) + warp;
    if (g < G) {
        const float a = row[g * kGroup + lane], b = row[g * kGroup + 32 + lane];
        const int e = split_exponent(warp_max(fmaxf(fabsf(a), fabsf(b))));
        const float mul = ldexpf(1.0f, e);
        buf[warp][lane] = a * mul;
        buf[warp][32 + lane] = b * mul;
        __syncwarp();
        if constexpr (kSub) {
            const float sum = warp_sum(a * mul + b * mul);
            if (lane < 16) cells[((size_t)r * G + g) * 16 + lane] = make_unit_s(buf[warp], lane);
            if (lane == 0)
                reinterpret_cast<float2 *>(fac)[(size_t)r * G + g] =
                    make_float2(ldexpf(1.0f, -e), offset_init(sum));
        } else {
            if (lane < 16)
                cells[((size_t)r * G + g) * 16 + lane] = make_unit<kInt8>(buf[warp], lane);
            if (lane == 0) fac[(size_t)r * G + g] = ldexpf(1.0f, -e);
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------------ dense

template <int NB, bool kInt8, class WS>
__device__ __forceinline__ void dense_item(WS &ws, int &cslot, int row0, int N, const float *scales,
                                           float *y, uint16_t *ybf, uint4 *cells, float *fac,
                                           int ntok, bool reuse, const StageCells &stage) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    float acc[NB][2];
    run_item<NB, kInt8>(ws, cslot, cells, fac, kDenseBudget, ntok, reuse, stage, acc);
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
            if (rA < N) store_y(y, ybf, (size_t)t * N + rA, acc[nb][0] * ra);
            if (rB < N) store_y(y, ybf, (size_t)t * N + rB, acc[nb][1] * rb);
        }
    }
}

// Rows of warp wp in item `item` of this CTA's range.
template <bool kInt8>
struct DenseTile {
    const uint8_t *w;
    const float *scales;
    size_t rowBytes;
    int N, G, i0;
    __device__ __forceinline__ TileSrc operator()(int item, int wp) const {
        int row0 = (i0 + item) * 16 * kDenseWarps + 16 * wp;
        int nrows = N - row0;
        if (nrows <= 0) { row0 = N - 1; nrows = 1; }
        return TileSrc{w + (size_t)row0 * rowBytes, kInt8 ? nullptr : scales + (size_t)row0 * G,
                       rowBytes, nrows, G};
    }
};

// K-split items: 16 rows per item, warp ks streams groups [ga, gb) of them.
template <bool kInt8>
struct DenseSplitTile {
    const uint8_t *w;
    const float *scales;
    size_t rowBytes;
    int N, G, i0, ga;
    __device__ __forceinline__ TileSrc operator()(int item, int) const {
        int row0 = (i0 + item) * 16;
        int nrows = N - row0;
        if (nrows <= 0) { row0 = N - 1; nrows = 1; }
        return TileSrc{w + (size_t)row0 * rowBytes + (size_t)ga * Fmt<kInt8>::kGroupBytes,
                       kInt8 ? nullptr : scales + (size_t)row0 * G + ga, rowBytes, nrows, G};
    }
};

// The items of k_dense_ks_x: 16-row tiles of the first matrix, then (for a
// pair sharing x) of the second; warp ks streams groups [ga, gb) of them.
template <bool kInt8>
struct PairSplitTile {
    const uint8_t *w0, *w1;
    const float *s0, *s1;
    size_t rowBytes;
    int N0, N1, items0, G, i0, ga;
    __device__ __forceinline__ TileSrc operator()(int item, int) const {
        const int gi = i0 + item;
        const bool sec = gi >= items0;
        const int N = sec ? N1 : N0;
        int row0 = (sec ? gi - items0 : gi) * 16;
        int nrows = N - row0;
        if (nrows <= 0) { row0 = N - 1; nrows = 1; }
        const uint8_t *w = sec ? w1 : w0;
        const float *sc = sec ? s1 : s0;
        return TileSrc{w + (size_t)row0 * rowBytes + (size_t)ga * Fmt<kInt8>::kGroupBytes,
                       kInt8 ? nullptr : sc + (size_t)row0 * G + ga, rowBytes, nrows, G};
    }
};

template <bool kInt8>
__global__ void __launch_bounds__(32 * kDenseWarps)
    k_dense(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
            const uint4 *__restrict__ xcells, const float *__restrict__ xfac,
            float *__restrict__ y, uint16_t *__restrict__ ybf, int ntok) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_rows[kMaxTok];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = K / kGroup;
    const int nitems = (N + 16 * kDenseWarps - 1) / (16 * kDenseWarps);
    const int i0 = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);
    const size_t rowBytes = kInt8 ? (size_t)K : (size_t)K / 2;

    DenseTile<kInt8> tile{w, scales, rowBytes, N, G, i0};
    WarpStream<kInt8, kDenseStages, DenseTile<kInt8>> ws;
    ws.init(smem + warp * kDenseRing, tile, G, i1 - i0, warp, lane);
    ws.prologue();  // weights are call inputs: safe to read before the wait
    int cslot = 0;

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
            dense_item<1, kInt8>(ws, cslot, row0, N, scales, y, ybf, cells, fac, ntok, reuse,
                                 stage);
        else
            dense_item<2, kInt8>(ws, cslot, row0, N, scales, y, ybf, cells, fac, ntok, reuse,
                                 stage);
    }
    cp_async_wait<0>();
}

// Dense GEMV for up to 4 tokens whose split activations fit in shared
// memory: every 16-row item is shared by the 8 warps of the CTA, warp ks
// taking an eighth of the K groups; partial sums meet in shared memory and
// are added in warp order (deterministic).
constexpr int kKsWarps = 8;
constexpr int kKsStages = 4;
constexpr int kKsRing = kKsStages * kStageBytes;

template <bool kInt8>
__global__ void __launch_bounds__(32 * kKsWarps)
    k_dense_ks(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
               const uint4 *__restrict__ xcells, const float *__restrict__ xfac,
               float *__restrict__ y, uint16_t *__restrict__ ybf, int ntok) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[kKsWarps][16][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const int gq = (G + kKsWarps - 1) / kKsWarps;
    const int ga = min(G, warp * gq), gb = min(G, ga + gq);
    const int nitems = (N + 15) / 16;
    const int i0 = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);
    const size_t rowBytes = kInt8 ? (size_t)K : (size_t)K / 2;

    DenseSplitTile<kInt8> tile{w, scales, rowBytes, N, G, i0, ga};
    WarpStream<kInt8, kKsStages, DenseSplitTile<kInt8>> ws;
    ws.init(smem + warp * kKsRing, tile, gb - ga, gb > ga ? i1 - i0 : 0, warp, lane);
    ws.prologue();  // weights are call inputs: safe to read before the wait
    int cslot = 0;

    pdl_wait();     // cells and factors come from k_split
    pdl_trigger();
    // token-major activation units: same layout as in global memory
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kKsWarps * kKsRing);
    float *fac = reinterpret_cast<float *>(smem + kKsWarps * kKsRing + kDenseBudget);
    for (int idx = threadIdx.x; idx < G * ntok * 16; idx += blockDim.x) cells[idx] = xcells[idx];
    for (int idx = threadIdx.x; idx < G * ntok; idx += blockDim.x) fac[idx] = xfac[idx];
    __syncthreads();
    const int sb = min(gid >> 1, ntok - 1), sd = min(q, ntok - 1);
    const uint4 *bp0 = cells + (sb * G + ga) * 16 + q * 2 + (gid & 1);
    const float *fp0 = fac + sd * G + ga;

    for (int it = 0; it < i1 - i0; ++it) {
        float acc[1][2] = {{0.f, 0.f}};
        if (gb > ga) run_staged<kInt8>(ws, cslot, bp0, fp0, acc);
        red[warp][gid][q] = acc[0][0];
        red[warp][gid + 8][q] = acc[0][1];
        __syncthreads();
        if (warp == 0 && q < ntok) {
            const int row0 = (i0 + it) * 16;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < kKsWarps; ++k) {
                a0 += red[k][gid][q];
                a1 += red[k][gid + 8][q];
            }
            const int rA = row0 + gid, rB = row0 + gid + 8;
            if constexpr (kInt8) {
                if (rA < N) a0 *= scales[rA];
                if (rB < N) a1 *= scales[rB];
            }
            if (rA < N) store_y(y, ybf, (size_t)q * N + rA, a0);
            if (rB < N) store_y(y, ybf, (size_t)q * N + rB, a1);
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

// Activation rows x[s][K] (s < ntok) -> the unit table cells[s][g][16] and
// factors fac[s][g] in shared memory, four threads per 64-group. Thread
// quarter q of a group holds values 16q .. 16q+15, which are exactly the
// values of the group's units (mh, q, part) (frag_ks: the quad's k's lie in
// [16q, 16q + 16)), so each thread builds its four units from its own values;
// the group's max |v| takes two shuffles between the four threads. Same
// arithmetic as k_split.
// The int3 decode's register order (dequant_int3_16: pairs (e_j, e_j+8) of a
// quad's 16 values, MMA step m taking pairs 2m and 2m + 1): the k's of the
// B operands of step m, relative to the quad's first value.
__device__ __forceinline__ void frag_ks_i3(int m, int &k0, int &k1, int &k2, int &k3) {
    k0 = 2 * m; k1 = 2 * m + 8; k2 = 2 * m + 1; k3 = 2 * m + 9;
}

template <bool kInt8, bool kI3 = false>
// Groups [ga, gb) of the ntok rows, split by the threads [t0, t0 + nthr) (a
// multiple of 4 threads: quad q of a group takes its values 16 q .. 16 q + 15).
// kI3: units in the int3 decode's order (frag_ks_i3) instead of int4's.
__device__ void split_rows_smem(const float *__restrict__ x, int K, int ntok, uint4 *cells,
                                float *fac, int ga, int gb, int t0, int nthr) {
    const int G = K / kGroup, ng = gb - ga, nq = ntok * ng * 4;
    const bool vec = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    for (int base = 0; base < nq; base += nthr) {  // uniform trip count: shuffles below
        const int idx = base + (int)threadIdx.x - t0;
        const bool valid = idx < nq;
        const int s = valid ? idx / (ng * 4) : 0, g = valid ? ga + (idx >> 2) % ng : 0, q = idx & 3;
        const float *src = x + (size_t)s * K + g * kGroup + 16 * q;
        float v[16];
        if (valid && vec) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 t = reinterpret_cast<const float4 *>(src)[i];
                v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = valid ? src[i] : 0.f;
        }
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
        const int e = split_exponent(am);
        const float mul = ldexpf(1.0f, e);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= mul;
        if (valid) {
            uint4 *dst = cells + ((size_t)s * G + g) * 16;
#pragma unroll
            for (int mh = 0; mh < 2; ++mh)
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    uint32_t r[4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        int k0, k1, k2, k3;
                        if constexpr (kI3)
                            frag_ks_i3(2 * mh + i, k0, k1, k2, k3);
                        else
                            frag_ks<kInt8>(2 * mh + i, 0, k0, k1, k2, k3);  // local to the quad
                        r[2 * i] = pack_half2(split_part(v[k0], part), split_part(v[k1], part));
                        r[2 * i + 1] = pack_half2(split_part(v[k2], part), split_part(v[k3], part));
                    }
                    dst[(mh * 4 + q) * 2 + part] = make_uint4(r[0], r[1], r[2], r[3]);
                }
            if (q == 0) fac[s * G + g] = ldexpf(1.0f, -e);
        }
    }
}

// k_dense_ks for activations given as fp32 rows: every CTA converts x into
// its shared-memory unit table itself (split_rows_smem) while its first
// weight stages are in flight, so the GEMV is one launch. With a second
// matrix (w2 != null: a pair sharing x) its row tiles follow the first's in
// the same item sequence. CTA 0 clears zero[0 .. nzero) (the caller's status
// word and counters).
// Weight stages per warp ring: with the 64 KB unit table, 2 stages keep the
// block under half the SM's shared memory, so two blocks stay resident.
constexpr int ks_x_stages(int budget) { return budget > 32 * 1024 ? 2 : 4; }

template <bool kInt8, int kBudget>
__global__ void __launch_bounds__(32 * kKsWarps)
    k_dense_ks_x(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
                 const float *__restrict__ x, float *__restrict__ y, uint16_t *__restrict__ ybf,
                 int ntok, int32_t *zero, int nzero, const uint8_t *__restrict__ w2,
                 const float *__restrict__ scales2, int N2, float *__restrict__ y2) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[kKsWarps][16][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    const int gq = (G + kKsWarps - 1) / kKsWarps;
    const int ga = min(G, warp * gq), gb = min(G, ga + gq);
    const int items0 = (N + 15) / 16;
    const int nitems = items0 + (w2 ? (N2 + 15) / 16 : 0);
    const int i0 = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);
    const size_t rowBytes = kInt8 ? (size_t)K : (size_t)K / 2;

    PairSplitTile<kInt8> tile{w, w2, scales, scales2, rowBytes, N, N2, items0, G, i0, ga};
    constexpr int kNS = ks_x_stages(kBudget), kRing = kNS * kStageBytes;
    WarpStream<kInt8, kNS, PairSplitTile<kInt8>> ws;
    ws.init(smem + warp * kRing, tile, gb - ga, gb > ga ? i1 - i0 : 0, warp, lane);
    ws.prologue();  // weights are call inputs: safe to read before the wait

    pdl_wait();     // x may come from the previous kernel
    pdl_trigger();
    if (zero && blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kKsWarps * kRing);
    float *fac = reinterpret_cast<float *>(smem + kKsWarps * kRing + kBudget);
    // each warp converts the groups of its own K share: no block barrier
    split_rows_smem<kInt8>(x, K, ntok, cells, fac, ga, gb, warp * 32, 32);
    __syncwarp();
    int cslot = 0;
    const int sb = min(gid >> 1, ntok - 1), sd = min(q, ntok - 1);
    const uint4 *bp0 = cells + (sb * G + ga) * 16 + q * 2 + (gid & 1);
    const float *fp0 = fac + sd * G + ga;

    for (int it = 0; it < i1 - i0; ++it) {
        float acc[1][2] = {{0.f, 0.f}};
        if (gb > ga) run_staged<kInt8>(ws, cslot, bp0, fp0, acc);
        red[warp][gid][q] = acc[0][0];
        red[warp][gid + 8][q] = acc[0][1];
        __syncthreads();
        if (warp == 0 && q < ntok) {
            const int gi = i0 + it;
            const bool sec = gi >= items0;
            const int Nm = sec ? N2 : N;
            const int row0 = (sec ? gi - items0 : gi) * 16;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < kKsWarps; ++k) {
                a0 += red[k][gid][q];
                a1 += red[k][gid + 8][q];
            }
            const int rA = row0 + gid, rB = row0 + gid + 8;
            if constexpr (kInt8) {
                const float *rs = sec ? scales2 : scales;
                if (rA < Nm) a0 *= rs[rA];
                if (rB < Nm) a1 *= rs[rB];
            }
            float *yo = sec ? y2 : y;
            uint16_t *ho = sec ? nullptr : ybf;
            if (rA < Nm) store_y(yo, ho, (size_t)q * Nm + rA, a0);
            if (rB < Nm) store_y(yo, ho, (size_t)q * Nm + rB, a1);
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

// Whether a GEMV of S tokens of length K runs as the single-launch
// k_dense_ks_x: up to 4 tokens whose units fit 64 KB of shared memory (the
// 32 KB form keeps two thread blocks per SM).
constexpr int kXBudgetSmall = 32 * 1024, kXBudgetLarge = 64 * 1024;
inline bool dense_one_launch(int K, int S) {
    return S <= 4 && (size_t)(K / kGroup) * S * 256 <= (size_t)kXBudgetLarge;
}

// The single-launch GEMV (k_dense_ks_x) of one matrix, or of a pair sharing x.
template <bool kInt8, int kBudget>
cudaError_t launch_ks_x_b(const uint8_t *w, const float *scales, int N, int K, const float *x,
                          float *y, uint16_t *ybf, int S, int32_t *zero, int nzero,
                          cudaStream_t st, const uint8_t *w2, const float *scales2, int N2,
                          float *y2) {
    const size_t smem_ks = (size_t)kKsWarps * ks_x_stages(kBudget) * kStageBytes + kBudget + kBudget / 64;
    cudaError_t e = set_smem(k_dense_ks_x<kInt8, kBudget>, smem_ks);
    if (e != cudaSuccess) return e;
    const int items = (N + 15) / 16 + (w2 ? (N2 + 15) / 16 : 0);
    const int slots =
        sm_count() * max_ctas_per_sm(k_dense_ks_x<kInt8, kBudget>, 32 * kKsWarps, smem_ks);
    return launch(k_dense_ks_x<kInt8, kBudget>, dim3(items < slots ? items : slots),
                  dim3(32 * kKsWarps), smem_ks, st, true, w, scales, N, K, x, y, ybf, S, zero,
                  nzero, w2, scales2, N2, y2);
}

template <bool kInt8>
cudaError_t launch_ks_x(const uint8_t *w, const float *scales, int N, int K, const float *x,
                        float *y, uint16_t *ybf, int S, int32_t *zero, int nzero, cudaStream_t st,
                        const uint8_t *w2 = nullptr, const float *scales2 = nullptr, int N2 = 0,
                        float *y2 = nullptr) {
    if ((size_t)(K / kGroup) * S * 256 <= (size_t)kXBudgetSmall)
        return launch_ks_x_b<kInt8, kXBudgetSmall>(w, scales, N, K, x, y, ybf, S, zero, nzero, st,
                                                   w2, scales2, N2, y2);
    return launch_ks_x_b<kInt8, kXBudgetLarge>(w, scales, N, K, x, y, ybf, S, zero, nzero, st, w2,
                                               scales2, N2, y2);
}

// ------------------------------------------------------------------ int3-g64 on the warp MMA
//
// The int3-g64 two-plane rows (24 bytes a group: a 16-byte low plane with
// element j of word w at bits 2j, then 8 bytes of high bits, element e at bit
// e % 8 of byte e / 8) through the same single-launch structure as
// k_dense_ks_x: 8 warps share each 16-row item, warp ks streams an eighth of
// its groups through a cp.async ring, every block splits x into its own unit
// table, and the 16 elements a lane quad takes of each group are decoded into
// exact fp16 (code - 4) as pairs (e_j, e_j+8), the order the activation units
// of this path are built in (frag_ks_i3); the MMA steps are int4's.

// A stage: 16 rows x 4 groups (96 bytes a row), rows 112 bytes apart so that
// a fragment load of the 8 row pairs (28 words apart) touches 8 distinct
// 4-bank windows; then the 16 x 4 group scales.
constexpr int kI3Row = 112;
constexpr int kI3StageW = 16 * kI3Row;
constexpr int kI3Stage = kI3StageW + 16 * 4 * 4;

// Exact (code - 4) of the 16 elements e_0 .. e_15 of one row that a lane
// quad takes from a group, as p[j] = (e_j, e_j+8), j = 0..7, first element in
// the low half (the units follow: frag_ks_i3). lo: their low-plane word (e_j
// at bits 2j); hs: their 16 high bits (e_j at bit j). Pair j's low bits sit
// at bits 2j' and 2j' + 16 of lo (j' = j) or of lo >> 8 (j' = j - 4), so
// OR-ing them into fp16 1024.0 gives t = 1024 + 4^j' low; its high bits,
// moved to j + 2 and j + 18, give u = 1024 + 2^(j+2) high. Then
//   t * 4^-j' - (4 + 1024 * 2^-j + 1024 * 4^-j') = low - 4 - 1024 * 2^-j
//   u * 2^-j + that                               = low + 4 high - 4
// are two fp16 fmas with exact results (small integers, and the intermediate
// within fp16's integer spacing at its magnitude).
__device__ __forceinline__ void dequant_int3_16(uint32_t lo, uint32_t hs, uint32_t p[8]) {
    const uint32_t kBias = 0x64006400u;
    const uint32_t x[2] = {lo, lo >> 8};
    const uint32_t h = prmt_u32(hs, 0u, 0x4140u) << 2;  // e_j at j + 2, e_j+8 at j + 18
    const uint32_t kLoScale[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};  // 4^-j'
    // -(4 + 1024 * 2^-j + 1024 * 4^-j'): -2052, -772, -324, -148, -1092, -292, -84, -28
    const uint32_t kLoAdd[8] = {0xE802E802u, 0xE208E208u, 0xDD10DD10u, 0xD8A0D8A0u,
                                0xE444E444u, 0xDC90DC90u, 0xD540D540u, 0xCF00CF00u};
    // 2^-j
    const uint32_t kHiScale[8] = {0x3C003C00u, 0x38003800u, 0x34003400u, 0x30003000u,
                                  0x2C002C00u, 0x28002800u, 0x24002400u, 0x20002000u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t t = lop3_and_or(x[j >> 2], 0x00030003u << (2 * (j & 3)), kBias);
        const uint32_t u = lop3_and_or(h, 0x00040004u << j, kBias);
        p[j] = hfma2_u32(u, kHiScale[j], hfma2_u32(t, kLoScale[j & 3], kLoAdd[j]));
    }
}

// One warp's 16-row tile of one group, up to 4 tokens (see tile_group_int4;
// MMA step m takes pairs 2m, 2m + 1): lo / hs of rows gid and gid + 8.
__device__ __forceinline__ void tile_group_int3(uint32_t lo0, uint32_t hs0, uint32_t lo8,
                                                uint32_t hs8, const uint4 (&bu)[2], float d[4]) {
    uint32_t p0[8], p8[8], a[4];
    dequant_int3_16(lo0, hs0, p0);
    dequant_int3_16(lo8, hs8, p8);
    d[0] = d[1] = d[2] = d[3] = 0.0f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        a[0] = p0[2 * m];
        a[1] = p8[2 * m];
        a[2] = p0[2 * m + 1];
        a[3] = p8[2 * m + 1];
        const uint4 &b = bu[m >> 1];
        mma_16816(d, a, (m & 1) ? b.z : b.x, (m & 1) ? b.w : b.y);
    }
}

// Per-warp cp.async stream of 4-group stages over the CTA's items (16-row
// tiles), groups [ga, ga + 4 nst) of each row. Lane l copies the 16-byte
// pieces l, l + 32, l + 64 of a stage's 96 (row = piece / 6) and two scales.
template <int NS>
struct I3Stream {
    uint32_t ring_s;
    const uint8_t *w;
    const float *sc;
    size_t rowBytes;
    int N, G, ga, nst, i0, nitems;
    int it_item, it_s, slot, lane;
    const uint8_t *wsrc[3];
    const float *ssrc[2];
    uint32_t wdst[3], sdst[2];

    __device__ __forceinline__ void init(uint8_t *ring, const uint8_t *w_, const float *sc_,
                                         int N_, int G_, int ga_, int nst_, int i0_, int nitems_,
                                         int lane_) {
        ring_s = smem_u32(ring);
        w = w_;
        sc = sc_;
        N = N_;
        G = G_;
        rowBytes = (size_t)G_ * 24;
        ga = ga_;
        nst = nst_;
        i0 = i0_;
        nitems = nst_ > 0 ? nitems_ : 0;
        it_item = it_s = slot = 0;
        lane = lane_;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int c = lane + 32 * k;
            wdst[k] = (c / 6) * kI3Row + (c % 6) * 16;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) sdst[k] = kI3StageW + (((lane >> 2) + 8 * k) * 4 + (lane & 3)) * 4;
        if (nitems > 0) set_item(0);
    }
    __device__ __forceinline__ void set_item(int item) {
        const int row0 = (i0 + item) * 16;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int c = lane + 32 * k;
            const int row = min(row0 + c / 6, N - 1);  // rows past N: read, never stored
            wsrc[k] = w + (size_t)row * rowBytes + (size_t)ga * 24 + (c % 6) * 16;
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int row = min(row0 + (lane >> 2) + 8 * k, N - 1);
            ssrc[k] = sc + (size_t)row * G + ga + (lane & 3);
        }
    }
    __device__ __forceinline__ void issue_next() {
        if (it_item < nitems) {
            const uint32_t base = ring_s + slot * kI3Stage;
#pragma unroll
            for (int k = 0; k < 3; ++k) cp_async16_s(base + wdst[k], wsrc[k] + it_s * 96);
#pragma unroll
            for (int k = 0; k < 2; ++k) cp_async4_s(base + sdst[k], ssrc[k] + 4 * it_s);
            if (++it_s == nst) {
                it_s = 0;
                if (++it_item < nitems) set_item(it_item);
            }
        }
        cp_async_commit();  // possibly empty: keeps the group count uniform
        slot = (slot + 1 == NS) ? 0 : slot + 1;
    }
    __device__ __forceinline__ void prologue() {
        for (int i = 0; i < NS - 1; ++i) issue_next();
    }
    __device__ __forceinline__ void acquire() {
        cp_async_wait<NS - 2>();
        __syncwarp();
        issue_next();
    }
};

// One stage of 4 groups: the lane's unit / factor pointers at the stage's
// first group; c2[i]: rows gid / gid + 8 of token q, groups of parity i.
__device__ __forceinline__ void compute_stage_int3(const uint8_t *slotp, const uint4 *bp,
                                                   const float *fp, float c2[2][2]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const float *ss = reinterpret_cast<const float *>(slotp + kI3StageW);
    const float4 SA = *reinterpret_cast<const float4 *>(ss + gid * 4);
    const float4 SB = *reinterpret_cast<const float4 *>(ss + (gid + 8) * 4);
    const float sa[4] = {SA.x, SA.y, SA.z, SA.w}, sb[4] = {SB.x, SB.y, SB.z, SB.w};
    const uint8_t *r0 = slotp + gid * kI3Row, *r8 = r0 + 8 * kI3Row;
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
        uint32_t lo0[2], lo8[2], hs0[2], hs8[2];
        uint4 bu[2][2];
        float f[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int gl = h + i;
            lo0[i] = *reinterpret_cast<const uint32_t *>(r0 + gl * 24 + 4 * q);
            lo8[i] = *reinterpret_cast<const uint32_t *>(r8 + gl * 24 + 4 * q);
            hs0[i] = *reinterpret_cast<const uint16_t *>(r0 + gl * 24 + 16 + 2 * q);
            hs8[i] = *reinterpret_cast<const uint16_t *>(r8 + gl * 24 + 16 + 2 * q);
            bu[i][0] = bp[gl * 16];
            bu[i][1] = bp[gl * 16 + 8];
            f[i] = fp[gl];
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int gl = h + i;
            float dd[4];
            tile_group_int3(lo0[i], hs0[i], lo8[i], hs8[i], bu[i], dd);
            c2[i][0] = fmaf(sa[gl] * f[i], dd[0] + dd[1], c2[i][0]);
            c2[i][1] = fmaf(sb[gl] * f[i], dd[2] + dd[3], c2[i][1]);
        }
    }
}

template <int kBudget>
__global__ void __launch_bounds__(32 * kKsWarps)
    k_int3_ks_x(const uint8_t *__restrict__ w, const float *__restrict__ scales, int N, int K,
                const float *__restrict__ x, float *__restrict__ y, int ntok) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ float red[kKsWarps][16][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = K / kGroup;
    // groups per warp: an eighth of G rounded up to whole 4-group stages
    const int gq = (G / 4 + kKsWarps - 1) / kKsWarps * 4;
    const int ga = min(G, warp * gq), gb = min(G, ga + gq);
    const int nitems = (N + 15) / 16;
    const int i0 = (int)((long long)blockIdx.x * nitems / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * nitems / gridDim.x);

    constexpr int kNS = ks_x_stages(kBudget), kRing = kNS * kI3Stage;
    I3Stream<kNS> ws;
    ws.init(smem + warp * kRing, w, scales, N, G, ga, (gb - ga) / 4, i0, i1 - i0, lane);
    ws.prologue();  // weights are call inputs: safe to read before the wait

    pdl_wait();     // x may come from the previous kernel
    pdl_trigger();
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kKsWarps * kRing);
    float *fac = reinterpret_cast<float *>(smem + kKsWarps * kRing + kBudget);
    // each warp converts the groups of its own K share: no block barrier
    split_rows_smem<false, true>(x, K, ntok, cells, fac, ga, gb, warp * 32, 32);
    __syncwarp();
    int cslot = 0;
    const int sb = min(gid >> 1, ntok - 1), sd = min(q, ntok - 1);
    const uint4 *bp0 = cells + (sb * G + ga) * 16 + q * 2 + (gid & 1);
    const float *fp0 = fac + sd * G + ga;

    for (int it = 0; it < i1 - i0; ++it) {
        float c2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        for (int s = 0; s < (gb - ga) / 4; ++s) {
            ws.acquire();
            compute_stage_int3(smem + warp * kRing + cslot * kI3Stage, bp0 + s * 64, fp0 + 4 * s, c2);
            cslot = (cslot + 1 == kNS) ? 0 : cslot + 1;
        }
        red[warp][gid][q] = c2[0][0] + c2[1][0];
        red[warp][gid + 8][q] = c2[0][1] + c2[1][1];
        __syncthreads();
        if (warp == 0 && q < ntok) {
            const int row0 = (i0 + it) * 16;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < kKsWarps; ++k) {
                a0 += red[k][gid][q];
                a1 += red[k][gid + 8][q];
            }
            const int rA = row0 + gid, rB = row0 + gid + 8;
            if (rA < N) y[(size_t)q * N + rA] = a0;
            if (rB < N) y[(size_t)q * N + rB] = a1;
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

template <int kBudget>
cudaError_t launch_i3_ks_b(const uint8_t *w, const float *scales, int N, int K, const float *x,
                           float *y, int S, cudaStream_t st) {
    const size_t smem = (size_t)kKsWarps * ks_x_stages(kBudget) * kI3Stage + kBudget + kBudget / 64;
    cudaError_t e = set_smem(k_int3_ks_x<kBudget>, smem);
    if (e != cudaSuccess) return e;
    const int items = (N + 15) / 16;
    const int slots = sm_count() * max_ctas_per_sm(k_int3_ks_x<kBudget>, 32 * kKsWarps, smem);
    return launch(k_int3_ks_x<kBudget>, dim3(items < slots ? items : slots), dim3(32 * kKsWarps),
                  smem, st, true, w, scales, N, K, x, y, S);
}

template <bool kInt8>
cudaError_t launch_dense(const uint8_t *w, const float *scales, int N, int K, const float *x,
                         float *y, int S, void *xcells, float *xfac, cudaStream_t st,
                         int32_t *zero = nullptr, int nzero = 0, uint16_t *ybf = nullptr) {
    const size_t smem = engine_smem(kDenseWarps, kDenseStages, kDenseBudget, 0);
    cudaError_t e = set_smem(k_dense<kInt8>, smem);
    if (e != cudaSuccess) return e;
    const int nitems = (N + 16 * kDenseWarps - 1) / (16 * kDenseWarps);
    const int slots = sm_count() * max_ctas_per_sm(k_dense<kInt8>, 32 * kDenseWarps, smem);
    const int grid = nitems < slots ? nitems : slots;
    if (dense_one_launch(K, S))  // one launch: every CTA splits x itself
        return launch_ks_x<kInt8>(w, scales, N, K, x, y, ybf, S, zero, nzero, st);
    e = launch(k_split<kInt8>, dim3(S, (K / kGroup + 7) / 8), dim3(256), 0, st, false, x, K,
               static_cast<uint4 *>(xcells), xfac, zero, nzero);
    for (int s0 = 0; s0 < S && e == cudaSuccess; s0 += kMaxTok) {
        const int ntok = S - s0 < kMaxTok ? S - s0 : kMaxTok;
        e = launch(k_dense<kInt8>, dim3(grid), dim3(32 * kDenseWarps), smem, st, true, w, scales, N,
                   K, static_cast<const uint4 *>(xcells) + (size_t)s0 * (K / kGroup) * 16,
                   xfac + (size_t)s0 * (K / kGroup), y ? y + (size_t)s0 * N : nullptr,
                   ybf ? ybf + (size_t)s0 * N : nullptr, ntok);
    }
    return e;
}

}  // namespace

cudaError_t launch_split(const float *v, int R, int K, void *cells, float *fac, cudaStream_t st,
                         bool sub) {
    if (R == 0) return cudaSuccess;
    if (sub)
        return launch(k_split<false, true>, dim3(R, (K / kGroup + 7) / 8), dim3(256), 0, st, false,
                      v, K, static_cast<uint4 *>(cells), fac, (int32_t *)nullptr, 0);
    return launch(k_split<false>, dim3(R, (K / kGroup + 7) / 8), dim3(256), 0, st, false, v, K,
                  static_cast<uint4 *>(cells), fac, (int32_t *)nullptr, 0);
}

bool int3_one_launch(const uint8_t *wq, int K, int S) {
    return S >= 1 && S <= 4 && K % 256 == 0 && (reinterpret_cast<uintptr_t>(wq) & 15) == 0 &&
           (size_t)(K / kGroup) * S * 256 <= (size_t)kXBudgetLarge;
}

cudaError_t launch_gemv_int3_mma(const uint8_t *wq, const float *scales, int N, int K,
                                 const float *x, float *y, int S, cudaStream_t st) {
    if ((size_t)(K / kGroup) * S * 256 <= (size_t)kXBudgetSmall)
        return launch_i3_ks_b<kXBudgetSmall>(wq, scales, N, K, x, y, S, st);
    return launch_i3_ks_b<kXBudgetLarge>(wq, scales, N, K, x, y, S, st);
}

// activation units (4 bytes a value) and a factor record of up to 8 bytes a group
size_t dense_scratch_bytes(int K, int S) { return (size_t)S * K * 4 + (size_t)S * (K / kGroup) * 8; }

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

// ------------------------------------------------------------------ workspace entry points
//
// Workspace of qmv_int4_gs / qmv_int8_row: the status word and the split
// counters (cleared by the split kernel), the activation units and factors,
// and the partial sums of row tiles split between CTAs.
namespace {
constexpr size_t kGemvHead = 1280;
static_assert(kGemvHead >= 4 * (1 + (size_t)kSkMaxCtas) && kGemvHead % 256 == 0, "head layout");

size_t gemv_part_offset(int K, int S) {
    return (kGemvHead + dense_scratch_bytes(K, S) + 255) & ~(size_t)255;
}
}  // namespace

size_t gemv_ws_bytes(int K, int S) {
    return gemv_part_offset(K, S) + (size_t)kSkMaxCtas * kSkPartFloats * 4;
}

cudaError_t launch_gemv_int4(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                             float *y, int S, void *ws, cudaStream_t st, uint16_t *ybf) {
    char *b = static_cast<char *>(ws);
    int32_t *head = reinterpret_cast<int32_t *>(b);
    void *cells = b + kGemvHead;
    float *fac = reinterpret_cast<float *>(b + kGemvHead + (size_t)S * K * 4);
    // one or a few tokens with x fitting shared memory: the single-launch
    // cp.async kernel (no activation split ahead of it) is faster than the
    // tensor-map kernel, whose split, pipeline fill and stream-K fix-up cost
    // more than a few stages of streaming
    if (!tma_dense_supported(wq, scales, N, K, S) || dense_one_launch(K, S))
        return launch_dense<false>(wq, scales, N, K, x, y, S, cells, fac, st, head,
                                   1 + kSkMaxCtas, ybf);
    float *part = reinterpret_cast<float *>(b + gemv_part_offset(K, S));
    cudaError_t e = launch(k_split<false, true>, dim3(S, (K / kGroup + 7) / 8), dim3(256), 0, st,
                           false, x, K, static_cast<uint4 *>(cells), fac, head, 1 + kSkMaxCtas);
    if (e != cudaSuccess) return e;
    return launch_dense_tma(wq, scales, N, K, S, cells, fac, y, head, head + 1, part, st, nullptr,
                            nullptr, 0, nullptr, ybf);
}

cudaError_t launch_gemv_int4_pair(const uint8_t *wq0, const float *s0, int N0, const uint8_t *wq1,
                                  const float *s1, int N1, int K, const float *x, float *y0,
                                  float *y1, int S, void *ws, cudaStream_t st) {
    if (dense_one_launch(K, S))  // both matrices' row tiles in one single-launch GEMV
        return launch_ks_x<false>(wq0, s0, N0, K, x, y0, nullptr, S,
                                  static_cast<int32_t *>(ws), 1 + kSkMaxCtas, st, wq1, s1, N1, y1);
    if (!tma_dense_supported(wq0, s0, N0, K, S) || !tma_dense_supported(wq1, s1, N1, K, S)) {
        cudaError_t e = launch_gemv_int4(wq0, s0, N0, K, x, y0, S, ws, st);
        return e == cudaSuccess ? launch_gemv_int4(wq1, s1, N1, K, x, y1, S, ws, st) : e;
    }
    char *b = static_cast<char *>(ws);
    int32_t *head = reinterpret_cast<int32_t *>(b);
    void *cells = b + kGemvHead;
    float *fac = reinterpret_cast<float *>(b + kGemvHead + (size_t)S * K * 4);
    float *part = reinterpret_cast<float *>(b + gemv_part_offset(K, S));
    cudaError_t e = launch(k_split<false, true>, dim3(S, (K / kGroup + 7) / 8), dim3(256), 0, st,
                           false, x, K, static_cast<uint4 *>(cells), fac, head, 1 + kSkMaxCtas);
    if (e != cudaSuccess) return e;
    return launch_dense_tma(wq0, s0, N0, K, S, cells, fac, y0, head, head + 1, part, st, wq1, s1,
                            N1, y1);
}

cudaError_t launch_gemv_int8(const int8_t *w, const float *row_scale, int N, int K,
                             const float *x, float *y, int S, void *ws, cudaStream_t st,
                             uint16_t *ybf) {
    char *b = static_cast<char *>(ws);
    float *fac = reinterpret_cast<float *>(b + kGemvHead + (size_t)S * K * 4);
    return launch_dense<true>(reinterpret_cast<const uint8_t *>(w), row_scale, N, K, x, y, S,
                              b + kGemvHead, fac, st, reinterpret_cast<int32_t *>(b),
                              1 + kSkMaxCtas, ybf);
}

}  // namespace qmv
