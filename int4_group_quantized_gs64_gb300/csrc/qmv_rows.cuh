// qmv_rows.cuh - the streaming row engine shared by the dense and MoE decode kernels.
//
// A CTA of kWarps warps owns kWarps 16-row tiles of one weight matrix (rows
// may come from different matrices, e.g. gate and up). Each warp streams its
// two rows per lane straight from HBM into a register ring kDepth groups deep
// (8 bytes of int4 or 16 bytes of int8 per row per group, plus the group
// scale), so every warp keeps kDepth * 512..1024 bytes in flight without
// waiting on shared memory. The activation fragments of the CTA's tokens are
// staged in shared memory one chunk of groups at a time; a chunk is a
// multiple of kDepth groups, so the ring continues across chunk boundaries.
#pragma once

#include <type_traits>

#include "qmv_device.cuh"

namespace qmv {

constexpr int kWarps = 4;                 // warps (16-row tiles) per CTA
constexpr int kCtaThreads = 32 * kWarps;
constexpr int kDepth = 8;                 // groups in flight per warp
constexpr int kMaxTok = 16;               // tokens per pass (4 MMA column blocks)
constexpr int kCellBudget = 32 * 1024;    // bytes of activation cells per chunk

// Groups per chunk for ntok tokens: 256 bytes of cells per token per group.
__host__ __device__ inline int chunk_groups(int ntok) {
    int c = kCellBudget / (256 * (ntok < 1 ? 1 : ntok));
    c = (c / kDepth) * kDepth;
    return c < kDepth ? kDepth : c;
}

template <bool kInt8>
struct WeightRing {
    using W = typename std::conditional<kInt8, uint4, uint2>::type;
    static constexpr int kGroupBytes = kInt8 ? 64 : 32;
    static constexpr int kLaneBytes = kInt8 ? 16 : 8;

    W ra[kDepth], rb[kDepth];
    float sa[kDepth], sb[kDepth];
    const uint8_t *pA, *pB;
    const float *sA, *sB;
    int G;

    // rowA / rowB: byte address of the two rows this lane streams; scaleA / B:
    // their group scales (ignored for int8).
    __device__ __forceinline__ void init(const uint8_t *rowA, const uint8_t *rowB,
                                         const float *scaleA, const float *scaleB, int groups,
                                         int q) {
        pA = rowA + kLaneBytes * q;
        pB = rowB + kLaneBytes * q;
        sA = scaleA;
        sB = scaleB;
        G = groups;
    }

    __device__ __forceinline__ void load(int slot_unused, int g, W &a, W &b, float &s0,
                                         float &s1) {
        (void)slot_unused;
        if constexpr (kInt8) {
            a = ldg_stream_u4(pA + (size_t)g * kGroupBytes);
            b = ldg_stream_u4(pB + (size_t)g * kGroupBytes);
            s0 = s1 = 1.0f;
        } else {
            a = ldg_stream_u2(pA + (size_t)g * kGroupBytes);
            b = ldg_stream_u2(pB + (size_t)g * kGroupBytes);
            s0 = ldg_stream_f32(sA + g);
            s1 = ldg_stream_f32(sB + g);
        }
    }

    __device__ __forceinline__ void prologue() {
#pragma unroll
        for (int d = 0; d < kDepth; ++d)
            if (d < G) load(d, d, ra[d], rb[d], sa[d], sb[d]);
    }
};

// Main loop over all groups. `stage(gc, ng)` must write the activation cells
// of groups [gc, gc + ng) into `cells` (all threads take part; no barriers
// inside). acc[nb][0 / 1]: rows gid / gid+8 for token 4*nb + q, sum of scaled
// group partials (before the per-token unscale).
template <int NB, bool kInt8, class Stage>
__device__ __forceinline__ void rows_mainloop(WeightRing<kInt8> &ring, uint4 *cells, int ntok,
                                              const Stage &stage, float acc[NB][2]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = ring.G;
    const int CG = chunk_groups(ntok);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = 0.0f;

    for (int gc = 0; gc < G; gc += CG) {
        const int ng = min(CG, G - gc);
        __syncthreads();  // all warps are done reading the previous chunk
        stage(gc, ng);
        __syncthreads();
        float c2[2][NB][2];  // two alternating accumulators halve the add depth
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) c2[h][nb][0] = c2[h][nb][1] = 0.0f;

        for (int g = gc; g < gc + ng; g += kDepth) {
#pragma unroll
            for (int d = 0; d < kDepth; ++d) {
                const int gg = g + d;
                if (gg < gc + ng) {
                    const auto a0 = ring.ra[d];
                    const auto a8 = ring.rb[d];
                    const float s0 = ring.sa[d], s8 = ring.sb[d];
                    if (gg + kDepth < G)
                        ring.load(d, gg + kDepth, ring.ra[d], ring.rb[d], ring.sa[d], ring.sb[d]);
                    float dd[NB][4];
                    if constexpr (kInt8)
                        tile_group_int8<NB>(a0, a8, cells, ntok, gg - gc, q, gid, dd);
                    else
                        tile_group_int4<NB>(a0, a8, cells, ntok, gg - gc, q, gid, dd);
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb) {
                        c2[d & 1][nb][0] = fmaf(s0, dd[nb][0] + dd[nb][1], c2[d & 1][nb][0]);
                        c2[d & 1][nb][1] = fmaf(s8, dd[nb][2] + dd[nb][3], c2[d & 1][nb][1]);
                    }
                }
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] += c2[0][nb][0] + c2[1][nb][0];
            acc[nb][1] += c2[0][nb][1] + c2[1][nb][1];
        }
    }
}

// Copies pre-split activation cells (layout [row][G][4][4] uint4, see
// qmv_device.cuh) of the CTA's token rows into the chunk buffer
// cells[(gl*4 + m)*4 + q][s].
struct StageFromCells {
    const uint4 *src;      // cells of all rows
    const int *rows;       // shared: cell row of each token slot
    int ntok, G;
    uint4 *cells;
    __device__ __forceinline__ void operator()(int gc, int ng) const {
        const int total = ng * 16 * ntok;
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int s = idx % ntok;
            const int r = idx / ntok;
            cells[idx] = src[(size_t)rows[s] * G * 16 + (size_t)gc * 16 + r];
        }
    }
};

}  // namespace qmv
