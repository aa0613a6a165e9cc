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

#include <type_traits>

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

// Whether expert e is served by the call: bit e % 32 of word e / 32 of the
// residency bitmap, or every expert when there is none.
__device__ __forceinline__ bool expert_served(const uint32_t *res, int e) {
    return res == nullptr || ((res[e >> 5] >> (e & 31)) & 1u) != 0;
}
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
    int sstride;  // floats between the scale rows (0: the stream's group count)
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async4_s(uint32_t dst, const void *gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(gmem) : "memory");
}

// Per-lane smem offsets of a stage slot, fixed for the whole kernel:
//   weights: lane copies chunk c = lane & 7 of rows lane/8 + 4j (j = 0..3);
//   scales (int4): lane copies scale lane & 3 of rows lane/4 + 8j (j = 0, 1);
//   fragments: row gid's 8 (int4) or 16 (int8) bytes of group gl of the stage.
template <bool kInt8>
struct LaneMap {
    uint32_t wdst[4], sdst[2];
    uint32_t frag[Fmt<kInt8>::kGPS];
    __device__ __forceinline__ void init(int lane) {
        const int c = lane & 7, gid = lane >> 2, q = lane & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = (lane >> 3) + 4 * j;
            wdst[j] = r * 128 + ((c ^ (r & 7)) << 4);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) sdst[j] = kStageWBytes + (((lane >> 2) + 8 * j) * 4 + (lane & 3)) * 4;
#pragma unroll
        for (int gl = 0; gl < Fmt<kInt8>::kGPS; ++gl) {
            if constexpr (kInt8)
                frag[gl] = gid * 128 + (((4 * gl + q) ^ gid) << 4);
            else
                frag[gl] = gid * 128 + (((2 * gl + (q >> 1)) ^ gid) << 4) + ((q & 1) << 3);
        }
    }
};

// Consume one stage: `ng` (<= GPS) groups of the stage. Activation units of
// the chunk are token-major, cells[s][gl][16], factors fac[s][gl]; bp0 / fp0
// point at this lane's unit / factor for the stage's first group, so the
// group offsets below are compile-time. Loads of two groups are issued before
// their math. Accumulates scale * factor * (hi + lo) per row and token.
template <int NB, bool kInt8>
__device__ __forceinline__ void compute_stage(const uint8_t *slotp, const LaneMap<kInt8> &lm,
                                              int ng, const uint4 *const bp0[NB],
                                              const float *const fp0[NB], float c2[2][NB][2]) {
    using W = typename std::conditional<kInt8, uint4, uint2>::type;
    constexpr int GPS = Fmt<kInt8>::kGPS;
    const int gid = (threadIdx.x & 31) >> 2;
    float sa[4] = {1.f, 1.f, 1.f, 1.f}, sb[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (!kInt8) {
        const float *ss = reinterpret_cast<const float *>(slotp + kStageWBytes);
        const float4 A = *reinterpret_cast<const float4 *>(ss + gid * 4);
        const float4 B = *reinterpret_cast<const float4 *>(ss + (gid + 8) * 4);
        sa[0] = A.x; sa[1] = A.y; sa[2] = A.z; sa[3] = A.w;
        sb[0] = B.x; sb[1] = B.y; sb[2] = B.z; sb[3] = B.w;
    }
#pragma unroll
    for (int h = 0; h < GPS; h += 2) {
        W w0[2], w8[2];
        uint4 bu[2][NB][2];
        float f[2][NB];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int gl = h + i;
            if (gl < ng) {
                w0[i] = *reinterpret_cast<const W *>(slotp + lm.frag[gl]);
                w8[i] = *reinterpret_cast<const W *>(slotp + lm.frag[gl] + 1024);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    bu[i][nb][0] = bp0[nb][gl * 16];
                    bu[i][nb][1] = bp0[nb][gl * 16 + 8];
                    f[i][nb] = fp0[nb][gl];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int gl = h + i;
            if (gl < ng) {
                float dd[NB][4];
                if constexpr (kInt8)
                    tile_group_int8<NB>(w0[i], w8[i], bu[i], dd);
                else
                    tile_group_int4<NB>(w0[i], w8[i], bu[i], dd);
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    c2[i][nb][0] = fmaf(sa[gl] * f[i][nb], dd[nb][0] + dd[nb][1], c2[i][nb][0]);
                    c2[i][nb][1] = fmaf(sb[gl] * f[i][nb], dd[nb][2] + dd[nb][3], c2[i][nb][1]);
                }
            }
        }
    }
}

// Per-warp weight stream over the CTA's items, NS stages deep.
// TileFn(item, warp) -> TileSrc (called once per item).
template <bool kInt8, int NS, class TileFn>
struct WarpStream {
    uint8_t *ring;     // this warp's NS * kStageBytes
    uint32_t ring_s;   // same, as a shared-window address
    TileFn tile;
    int G, ns, nitems;
    int it_item, it_s;  // next stage to issue
    const uint8_t *wsrc[4];
    const float *ssrc[2];
    int nfull;          // stages of an item that hold GPS whole groups
    int slot;           // slot of the next issue
    LaneMap<kInt8> lm;
    int warp, lane;

    __device__ __forceinline__ void init(uint8_t *ring_, TileFn tile_, int G_, int nitems_,
                                         int warp_, int lane_) {
        ring = ring_;
        ring_s = smem_u32(ring_);
        tile = tile_;
        G = G_;
        ns = (G_ + Fmt<kInt8>::kGPS - 1) / Fmt<kInt8>::kGPS;
        nfull = G_ / Fmt<kInt8>::kGPS;
        nitems = nitems_;
        it_item = 0;
        it_s = 0;
        slot = 0;
        warp = warp_;
        lane = lane_;
        lm.init(lane_);
        if (nitems > 0) set_item(0);
    }

    __device__ __forceinline__ void set_item(int item) {
        const TileSrc t = tile(item, warp);
        const int c = lane & 7;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = (lane >> 3) + 4 * j;
            const int rr = r < t.nrows ? r : t.nrows - 1;
            wsrc[j] = t.w + (size_t)rr * t.rowBytes + c * 16;
        }
        if constexpr (!kInt8) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int r = (lane >> 2) + 8 * j;
                const int rr = r < t.nrows ? r : t.nrows - 1;
                ssrc[j] = t.s + (size_t)rr * (t.sstride ? t.sstride : G) + (lane & 3);
            }
        }
    }

    __device__ __forceinline__ void issue_next() {
        if (it_item < nitems) {
            const uint32_t base = ring_s + slot * kStageBytes;
            const size_t wofs = (size_t)it_s * 128;
            const int g0 = it_s * Fmt<kInt8>::kGPS;
            if (it_s < nfull) {
#pragma unroll
                for (int j = 0; j < 4; ++j) cp_async16_s(base + lm.wdst[j], wsrc[j] + wofs);
                if constexpr (!kInt8) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) cp_async4_s(base + lm.sdst[j], ssrc[j] + g0);
                }
            } else {
                const int c = lane & 7;
                const int grp = g0 + (kInt8 ? (c >> 2) : (c >> 1));
                if (grp < G) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) cp_async16_s(base + lm.wdst[j], wsrc[j] + wofs);
                }
                if constexpr (!kInt8) {
                    if (g0 + (lane & 3) < G) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) cp_async4_s(base + lm.sdst[j], ssrc[j] + g0);
                    }
                }
            }
            if (++it_s == ns) {
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
    // Wait for the oldest outstanding stage (slot `cslot`), then refill the
    // slot that the previous stage freed.
    __device__ __forceinline__ void acquire() {
        cp_async_wait<NS - 2>();
        __syncwarp();
        issue_next();
    }
};

// Runs one item for up to 4*NB tokens: chunks of activations are staged by
// `stage(gc, ng, cells, fac)` (all threads; no barriers inside) unless
// `reuse` says the previous item left the full K in shared memory.
// cslot: slot of the next stage to consume (advanced here).
// acc[nb][0 / 1]: rows gid / gid+8 of this warp, token 4*nb + q.
template <int NB, bool kInt8, int NS, class TileFn, class Stage>
__device__ __forceinline__ void run_item(WarpStream<kInt8, NS, TileFn> &ws, int &cslot,
                                         uint4 *cells, float *fac, int budget, int ntok,
                                         bool reuse, const Stage &stage, float acc[NB][2]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = ws.G;
    const int CG = chunk_groups(ntok, budget);
    constexpr int GPS = Fmt<kInt8>::kGPS;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = 0.0f;
    const uint4 *bl[NB];
    const float *fl[NB];
    int sbt[NB], sdt[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        sbt[nb] = min(4 * nb + (gid >> 1), ntok - 1);  // token of this lane's B column
        sdt[nb] = min(4 * nb + q, ntok - 1);           // token of this lane's D columns
    }
    for (int gc = 0; gc < G; gc += CG) {
        const int ng = min(CG, G - gc);
        if (!(reuse && ng == G)) {
            __syncthreads();  // every warp is done with the previous chunk
            stage(gc, ng, cells, fac);
            __syncthreads();
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            bl[nb] = cells + (sbt[nb] * ng) * 16 + q * 2 + (gid & 1);
            fl[nb] = fac + sdt[nb] * ng;
        }
        float c2[2][NB][2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) c2[h][nb][0] = c2[h][nb][1] = 0.0f;
        for (int glc = 0; glc < ng; glc += GPS) {
            ws.acquire();
            const uint8_t *slotp = ws.ring + cslot * kStageBytes;
            compute_stage<NB, kInt8>(slotp, ws.lm, min(GPS, ng - glc), bl, fl, c2);
            cslot = (cslot + 1 == NS) ? 0 : cslot + 1;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                bl[nb] += GPS * 16;
                fl[nb] += GPS;
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] += c2[0][nb][0] + c2[1][nb][0];
            acc[nb][1] += c2[0][nb][1] + c2[1][nb][1];
        }
    }
}

// Runs the whole group range of one item against activation units that are
// already in shared memory (bp0 / fp0: this lane's units and factors at the
// first group of the range), NB = 1 token block. Used by the K-split dense
// kernel; acc: rows gid / gid+8, token q.
template <bool kInt8, int NS, class TileFn>
__device__ __forceinline__ void run_staged(WarpStream<kInt8, NS, TileFn> &ws, int &cslot,
                                           const uint4 *bp0, const float *fp0, float acc[1][2]) {
    constexpr int GPS = Fmt<kInt8>::kGPS;
    float c2[2][1][2] = {{{0.f, 0.f}}, {{0.f, 0.f}}};
    const uint4 *bp[1] = {bp0};
    const float *fp[1] = {fp0};
    for (int glc = 0; glc < ws.G; glc += GPS) {
        ws.acquire();
        const uint8_t *slotp = ws.ring + cslot * kStageBytes;
        compute_stage<1, kInt8>(slotp, ws.lm, min(GPS, ws.G - glc), bp, fp, c2);
        cslot = (cslot + 1 == NS) ? 0 : cslot + 1;
        bp[0] += GPS * 16;
        fp[0] += GPS;
    }
    acc[0][0] = c2[0][0][0] + c2[1][0][0];
    acc[0][1] = c2[0][0][1] + c2[1][0][1];
}

// Stages units + factors of `ntok` activation rows (rows `rows[s]` of the
// global layout [row][G][16 units] and [row][G] factors) for groups
// [gc, gc+ng) into the token-major chunk cells[s][gl][16] and fac[s][gl].
struct StageCells {
    const uint4 *src;
    const float *fsrc;
    const int *rows;  // shared memory
    int ntok, G;
    __device__ __forceinline__ void operator()(int gc, int ng, uint4 *cells, float *fac) const {
        const int per = ng * 16;
        for (int idx = threadIdx.x; idx < ntok * per; idx += blockDim.x) {
            const int s = idx / per, rem = idx - s * per;
            cells[idx] = src[((size_t)rows[s] * G + gc) * 16 + rem];
        }
        for (int idx = threadIdx.x; idx < ng * ntok; idx += blockDim.x) {
            const int s = idx / ng, gl = idx - s * ng;
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
