// qmv_rows.cuh - the streaming row engine shared by the dense and MoE decode kernels.
//
// Weights: every warp owns a 16-row tile and streams it from HBM through its
// own shared-memory ring of kStages stages with cp.async (16-byte copies that
// bypass L1). A stage holds 128 bytes of each of the 16 rows (4 int4 groups or
// 2 int8 groups) plus the 16 x 4 group scales. The 16-byte chunks of a row are
// XOR-swizzled by (row & 7) so the fragment reads below are bank-conflict free.
// NS - 1 stages are in flight while one is consumed, without holding any of
// it in registers.
//
// Work: a CTA walks a contiguous range of work items (an item is one row tile
// of every warp, e.g. 64 or 128 rows of one expert matrix); the warp rings run
// on across items, so they never drain inside a CTA.
//
// Activations: fragment cells (see qmv_device.cuh) plus one power-of-two
// factor per (row, group) are staged in shared memory one chunk of groups at a
// time; a chunk is a multiple of the stage size.
#pragma once

#include "qmv_device.cuh"

namespace qmv {

constexpr int kStageWBytes = 16 * 128;                 // weights of one stage
constexpr int kStageBytes = kStageWBytes + 16 * 4 * 4; // + 16 rows x 4 scales
constexpr int kMaxTok = 8;                             // tokens per pass (2 MMA blocks)

template <bool kInt8>
struct Fmt {
    static constexpr int kGPS = kInt8 ? 2 : 4;          // groups per stage
    static constexpr int kGroupBytes = kInt8 ? 64 : 32; // bytes of one row per group
};

// Groups per activation chunk for ntok tokens within `budget` bytes of cells
// (256 bytes per token per group); a multiple of 4 groups (both formats).
__host__ __device__ inline int chunk_groups(int ntok, int budget) {
    int c = budget / (256 * (ntok < 1 ? 1 : ntok));
    c &= ~3;
    return c < 4 ? 4 : c;
}

// ------------------------------------------------------------------ cp.async

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: wait for the previous kernel's results /
// let the next kernel's CTAs start. Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ tile source

// The 16 rows of one warp tile: row r at w + r * rowBytes (rows >= nrows are
// replaced by row nrows-1, which is read but never stored), its scales at
// s + r * G.
struct TileSrc {
    const uint8_t *w;
    const float *s;
    size_t rowBytes;
    int nrows;
};

template <bool kInt8>
__device__ __forceinline__ void issue_stage(uint8_t *slot, const TileSrc &t, int stage, int G,
                                            int lane) {
    const int g0 = stage * Fmt<kInt8>::kGPS;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = lane + 32 * j;
        const int r = i >> 3, c = i & 7;
        const int grp = g0 + (kInt8 ? (c >> 2) : (c >> 1));
        if (grp < G) {
            const int rr = r < t.nrows ? r : t.nrows - 1;
            const uint8_t *src =
                t.w + (size_t)rr * t.rowBytes + (size_t)g0 * Fmt<kInt8>::kGroupBytes + c * 16;
            cp_async16(slot + r * 128 + ((c ^ (r & 7)) << 4), src);
        }
    }
    if constexpr (!kInt8) {
        float *ss = reinterpret_cast<float *>(slot + kStageWBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j;
            const int r = i >> 2, gg = i & 3;
            if (g0 + gg < G) {
                const int rr = r < t.nrows ? r : t.nrows - 1;
                cp_async4(ss + r * 4 + gg, t.s + (size_t)rr * G + g0 + gg);
            }
        }
    }
}

// Consume one stage: groups [g0, g0 + GPS) of the chunk starting at group gc,
// stopping at gEnd. Activation units of the chunk are cells[gl][s][16] and
// factors fac[gl][s] (gl = g - gc, s < ntok). Accumulates
// scale * factor * (hi + lo) per row and token.
template <int NB, bool kInt8>
__device__ __forceinline__ void compute_stage(const uint8_t *slot, int g0, int gc, int gEnd,
                                              const uint4 *cells, const float *fac, int ntok,
                                              float c2[2][NB][2]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    float4 sA = make_float4(1.f, 1.f, 1.f, 1.f), sB = sA;
    if constexpr (!kInt8) {
        const float *ss = reinterpret_cast<const float *>(slot + kStageWBytes);
        sA = *reinterpret_cast<const float4 *>(ss + gid * 4);
        sB = *reinterpret_cast<const float4 *>(ss + (gid + 8) * 4);
    }
    const float sa[4] = {sA.x, sA.y, sA.z, sA.w}, sb[4] = {sB.x, sB.y, sB.z, sB.w};
    int sB_tok[NB], sD_tok[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        sB_tok[nb] = min(4 * nb + (gid >> 1), ntok - 1);  // token of this lane's B column
        sD_tok[nb] = min(4 * nb + q, ntok - 1);           // token of this lane's D columns
    }
#pragma unroll
    for (int gl = 0; gl < Fmt<kInt8>::kGPS; ++gl) {
        const int g = g0 + gl;
        if (g < gEnd) {
            const int glc = g - gc;
            const uint4 *bp[NB];
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
                bp[nb] = cells + (glc * ntok + sB_tok[nb]) * 16 + q * 2 + (gid & 1);
            float dd[NB][4];
            if constexpr (kInt8) {
                const int c = 4 * gl + q;
                const uint4 w0 = *reinterpret_cast<const uint4 *>(slot + gid * 128 + ((c ^ gid) << 4));
                const uint4 w8 =
                    *reinterpret_cast<const uint4 *>(slot + (gid + 8) * 128 + ((c ^ gid) << 4));
                tile_group_int8<NB>(w0, w8, bp, dd);
            } else {
                const int c = 2 * gl + (q >> 1);
                const int off = ((c ^ gid) << 4) + ((q & 1) << 3);
                const uint2 w0 = *reinterpret_cast<const uint2 *>(slot + gid * 128 + off);
                const uint2 w8 = *reinterpret_cast<const uint2 *>(slot + (gid + 8) * 128 + off);
                tile_group_int4<NB>(w0, w8, bp, dd);
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const float f = fac[glc * ntok + sD_tok[nb]];
                c2[gl & 1][nb][0] = fmaf(sa[gl] * f, dd[nb][0] + dd[nb][1], c2[gl & 1][nb][0]);
                c2[gl & 1][nb][1] = fmaf(sb[gl] * f, dd[nb][2] + dd[nb][3], c2[gl & 1][nb][1]);
            }
        }
    }
}

// Per-warp weight stream over the CTA's items, NS stages deep.
// TileFn(item, warp) -> TileSrc.
template <bool kInt8, int NS, class TileFn>
struct WarpStream {
    uint8_t *ring;  // this warp's NS * kStageBytes
    TileFn tile;
    int G, ns, total;  // groups per row, stages per item, stages of all items
    int next;          // next global stage to issue
    int warp, lane;

    __device__ __forceinline__ void issue_next() {
        if (next < total) {
            const int item = next / ns, s = next - item * ns;
            issue_stage<kInt8>(ring + (next % NS) * kStageBytes, tile(item, warp), s, G, lane);
        }
        cp_async_commit();  // possibly empty: keeps the group count uniform
        ++next;
    }
    __device__ __forceinline__ void prologue() {
        for (int i = 0; i < NS - 1; ++i) issue_next();
    }
    // Wait for stage j (global index), refill the slot freed by stage j-1.
    __device__ __forceinline__ const uint8_t *acquire(int j) {
        cp_async_wait<NS - 2>();
        __syncwarp();
        issue_next();
        return ring + (j % NS) * kStageBytes;
    }
};

// Runs one item for up to 4*NB tokens: chunks of activations are staged by
// `stage(gc, ng, cells, fac)` (all threads; no barriers inside) unless
// `reuse` says the previous item left the full K in shared memory.
// acc[nb][0 / 1]: rows gid / gid+8 of this warp, token 4*nb + q.
template <int NB, bool kInt8, int NS, class TileFn, class Stage>
__device__ __forceinline__ void run_item(WarpStream<kInt8, NS, TileFn> &ws, int item, uint4 *cells,
                                         float *fac, int budget, int ntok, bool reuse,
                                         const Stage &stage, float acc[NB][2]) {
    const int G = ws.G;
    const int CG = chunk_groups(ntok, budget);
    constexpr int GPS = Fmt<kInt8>::kGPS;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = 0.0f;
    int j = item * ws.ns;
    for (int gc = 0; gc < G; gc += CG) {
        const int ng = min(CG, G - gc);
        if (!(reuse && ng == G)) {
            __syncthreads();  // every warp is done with the previous chunk
            stage(gc, ng, cells, fac);
            __syncthreads();
        }
        float c2[2][NB][2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) c2[h][nb][0] = c2[h][nb][1] = 0.0f;
        for (int g0 = gc; g0 < gc + ng; g0 += GPS, ++j) {
            const uint8_t *slot = ws.acquire(j);
            compute_stage<NB, kInt8>(slot, g0, gc, gc + ng, cells, fac, ntok, c2);
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] += c2[0][nb][0] + c2[1][nb][0];
            acc[nb][1] += c2[0][nb][1] + c2[1][nb][1];
        }
    }
}

// Stages units + factors of `ntok` activation rows (rows `rows[s]` of the
// global layout [row][G][16 units] and [row][G] factors) for groups
// [gc, gc+ng) into cells[gl][s][16] and fac[gl][s].
struct StageCells {
    const uint4 *src;
    const float *fsrc;
    const int *rows;  // shared memory
    int ntok, G;
    __device__ __forceinline__ void operator()(int gc, int ng, uint4 *cells, float *fac) const {
        const int total = ng * ntok * 16;
        for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
            const int u = idx & 15, r = idx >> 4;
            const int s = r % ntok, gl = r / ntok;
            cells[idx] = src[((size_t)rows[s] * G + gc + gl) * 16 + u];
        }
        for (int idx = threadIdx.x; idx < ng * ntok; idx += blockDim.x) {
            const int s = idx % ntok, gl = idx / ntok;
            fac[idx] = fsrc[(size_t)rows[s] * G + gc + gl];
        }
    }
};

// Shared memory of a CTA: `warps` rings, `budget` bytes of cells, factors
// (ng * ntok <= budget / 256 floats), then `extra` bytes of epilogue scratch.
__host__ __device__ inline size_t engine_smem(int warps, int stages, int budget, int extra) {
    return (size_t)warps * stages * kStageBytes + budget + budget / 64 + extra;
}

}  // namespace qmv
