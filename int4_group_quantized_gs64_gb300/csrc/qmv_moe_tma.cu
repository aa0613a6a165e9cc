// qmv_moe_tma.cu - MoE decode gate+up and down kernels fed by the Tensor
// Memory Accelerator.
//
// Same arithmetic as k_gate_up / k_down (qmv_moe.cu): exact fp16 weights in
// registers, fp16 hi/lo activations, warp MMA per 64-group, group scale in
// fp32 (colibri PR #418, "qmatmul_gate_up.comp + coli_vk_gate_up",
// "coli_vk_expert_group", "grouped scales in the Vulkan kernels"). What
// changes is how the weights arrive: one producer warp issues 3-D tensor-map
// loads (cp.async.bulk.tensor, 128-byte swizzle) of 256 rows x 128 bytes plus
// their scales per stage into a 4-stage ring guarded by mbarriers, so the 16
// consumer warps spend no instructions on copies. Consumer warp w owns stage
// rows 16w..16w+15: for gate+up warps 0-7 hold gate rows and warps 8-15 the
// up rows of the same 128 hidden units; for down, 256 consecutive rows.
//
// Every mbarrier wait is bounded. A consumer warp whose wait runs out stops
// waiting but keeps computing (on whatever the slot holds) and keeps every
// barrier, so all warps finish; the producer gives up when the consumers stop
// releasing slots and drains its loads before exiting; bit 1 of the status
// word records the failure (the outputs are then not valid).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_rows.cuh"
#include "tc05.cuh"

namespace qmv {

namespace {

constexpr int kTConsumers = 16;
constexpr int kTThreads = 32 * (kTConsumers + 1);
constexpr int kTStages = 4;
constexpr int kTRows = 256;                          // weight rows per stage
constexpr int kTStageW = kTRows * 128;               // 32 KB
constexpr int kTStageS = kTRows * 16;                // 4 KB
constexpr int kTStage = kTStageW + kTStageS;         // 36 KB
constexpr int kTBudget = 64 * 1024;
constexpr int kTGuJ = 128;                           // hidden units per gate+up item
constexpr int kTDnRows = 256;                        // output rows per down item
constexpr int kTEpi = (2 * kTGuJ * kMaxTok + kTConsumers * 64) * 4;
constexpr int kTSmem = kTStages * kTStage + kTBudget + kTBudget / 64 + kTEpi + 1024;
constexpr uint32_t kTWait = 1u << 24;

static_assert(kTStage % 1024 == 0, "stages must stay 1024-aligned for the 128B swizzle");

struct TmaArgs {
    CUtensorMap wmap;    // weights: uint8 [E][rows][K/2], box 128 B x 128 rows, 128B swizzle
    CUtensorMap smap;    // scales: f32 [E][rows][K/64], box 4 x 128 rows
    int mode;            // 0: gate+up, 1: down
    int G, I, H, k;
    const int32_t *offsets, *list, *uexp, *n_used, *pass_ofs;
    const uint4 *cells;  // activation units [row][G][16]
    const float *cfac;   // their factors [row][G]
    float *h;            // gate+up: h fp32 [P][I]
    uint4 *hcells;       // gate+up: units of h [P][I/64][16]
    float *hfac;         // gate+up: factors of h [P][I/64]
    float *y;            // down: y [P][H]
    int32_t *status;
};

__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                          int c2, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     tc05::smem_addr(mbar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc05::smem_addr(mbar))
                 : "memory");
}

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kTConsumers) : "memory");
}

struct TItem {
    int e, beg, ntok, tile;
};

__device__ __forceinline__ TItem t_item(const TmaArgs &a, int nu, int tiles, int item) {
    const int pi = item / tiles;
    TItem r;
    r.tile = item - pi * tiles;
    int lo = 0, hi = nu - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.pass_ofs[mid] <= pi) lo = mid; else hi = mid - 1;
    }
    r.e = a.uexp[lo];
    const int pass = pi - a.pass_ofs[lo];
    const int b = a.offsets[r.e], cnt = a.offsets[r.e + 1] - b;
    r.beg = b + pass * kMaxTok;
    r.ntok = min(kMaxTok, cnt - pass * kMaxTok);
    return r;
}

// Fragments of one group of this warp's 16-row tile (smem rows r0..r0+15).
template <int NB>
struct GroupFrag {
    uint2 w0, w8;
    uint4 bu[NB][2];
    float f[NB];
};

template <int NB, int GL>
__device__ __forceinline__ void group_load(const uint8_t *wa, int gid, int q,
                                           const uint4 *const bp0[NB], const float *const fp0[NB],
                                           GroupFrag<NB> &g) {
    const int off = (((2 * GL + (q >> 1)) ^ gid) << 4) + ((q & 1) << 3);
    g.w0 = *reinterpret_cast<const uint2 *>(wa + off);
    g.w8 = *reinterpret_cast<const uint2 *>(wa + 1024 + off);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        g.bu[nb][0] = bp0[nb][GL * 16];
        g.bu[nb][1] = bp0[nb][GL * 16 + 8];
        g.f[nb] = fp0[nb][GL];
    }
}

template <int NB, int GL>
__device__ __forceinline__ void group_math(const GroupFrag<NB> &g, float s0, float s8,
                                           float c[2][NB][2]) {
    float d[NB][4];
    tile_group_int4<NB>(g.w0, g.w8, g.bu, d);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        c[GL & 1][nb][0] = fmaf(s0 * g.f[nb], d[nb][0] + d[nb][1], c[GL & 1][nb][0]);
        c[GL & 1][nb][1] = fmaf(s8 * g.f[nb], d[nb][2] + d[nb][3], c[GL & 1][nb][1]);
    }
}

// One stage of this warp's tile: the fragments of two groups are loaded
// before their math, so shared-memory latency overlaps the previous math.
template <int NB>
__device__ __forceinline__ void compute_stage1(const uint8_t *slot, int r0, int ng,
                                               const uint4 *const bp0[NB],
                                               const float *const fp0[NB], float c[2][NB][2]) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const float *ss = reinterpret_cast<const float *>(slot + kTStageW);
    const float4 s0 = *reinterpret_cast<const float4 *>(ss + (r0 + gid) * 4);
    const float4 s8 = *reinterpret_cast<const float4 *>(ss + (r0 + gid + 8) * 4);
    const uint8_t *wa = slot + (r0 + gid) * 128;
    GroupFrag<NB> g0, g1;
    group_load<NB, 0>(wa, gid, q, bp0, fp0, g0);
    if (ng > 1) group_load<NB, 1>(wa, gid, q, bp0, fp0, g1);
    group_math<NB, 0>(g0, s0.x, s8.x, c);
    if (ng > 2) group_load<NB, 2>(wa, gid, q, bp0, fp0, g0);
    if (ng > 1) group_math<NB, 1>(g1, s0.y, s8.y, c);
    if (ng > 3) group_load<NB, 3>(wa, gid, q, bp0, fp0, g1);
    if (ng > 2) group_math<NB, 2>(g0, s0.z, s8.z, c);
    if (ng > 3) group_math<NB, 3>(g1, s0.w, s8.w, c);
}

struct TShared {
    uint64_t full[kTStages];
    uint64_t empty[kTStages];
    int rows[kMaxTok];
    int pairs[kMaxTok];
};

// Consumer side of one item. A wait that runs out sets `failed`; from then on
// the warp stops waiting but keeps the same sequence of barriers, so every
// warp reaches the end. acc: rows gid / gid+8 of this warp's tile, token 4nb+q.
// Warp w owns stage rows 16w..16w+15 (gate+up: warps 0-7 gate, 8-15 up).
template <int NB>
__device__ __forceinline__ void t_consume_item(const TmaArgs &a, TShared &sh, uint8_t *ring,
                                               uint4 *cells, float *fac, int ntok, bool reuse,
                                               int &j, bool &failed, float acc[NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int G = a.G;
    const int CG = chunk_groups(ntok, kTBudget);
    const int r0 = 16 * warp;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = 0.f;
    int sbt[NB], sdt[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        sbt[nb] = min(4 * nb + (gid >> 1), ntok - 1);
        sdt[nb] = min(4 * nb + q, ntok - 1);
    }
    for (int gc = 0; gc < G; gc += CG) {
        const int ng = min(CG, G - gc);
        if (!(reuse && ng == G)) {
            consumers_sync();
            const int per = ng * 16;
            for (int idx = threadIdx.x; idx < ntok * per; idx += 32 * kTConsumers) {
                const int s = idx / per, rem = idx - s * per;
                cells[idx] = a.cells[((size_t)sh.rows[s] * G + gc) * 16 + rem];
            }
            for (int idx = threadIdx.x; idx < ng * ntok; idx += 32 * kTConsumers) {
                const int s = idx / ng, gl = idx - s * ng;
                fac[idx] = a.cfac[(size_t)sh.rows[s] * G + gc + gl];
            }
            consumers_sync();
        }
        const uint4 *bp[NB];
        const float *fp[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            bp[nb] = cells + (sbt[nb] * ng) * 16 + q * 2 + (gid & 1);
            fp[nb] = fac + sdt[nb] * ng;
        }
        float c[2][NB][2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) c[h2][nb][0] = c[h2][nb][1] = 0.f;
        for (int glc = 0; glc < ng; glc += 4, ++j) {
            const int slot = j % kTStages;
            if (!failed &&
                !tc05::mbar_wait(&sh.full[slot], (uint32_t)((j / kTStages) & 1), kTWait))
                failed = true;
            compute_stage1<NB>(ring + slot * kTStage, r0, min(4, ng - glc), bp, fp, c);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[slot]);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                bp[nb] += 64;
                fp[nb] += 4;
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[nb][0] += c[0][nb][0] + c[1][nb][0];
            acc[nb][1] += c[0][nb][1] + c[1][nb][1];
        }
    }
}

template <int NB>
__device__ __forceinline__ void t_epilogue(const TmaArgs &a, const TShared &sh, float *epi,
                                           const TItem &it, const float acc[NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int ntok = it.ntok;
    if (a.mode == 1) {
        const int H = a.H;
        const int r0 = it.tile * kTDnRows + 16 * warp;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q;
            if (s < ntok) {
                float *yb = a.y + (size_t)sh.pairs[s] * H;
                if (r0 + gid < H) yb[r0 + gid] = acc[nb][0];
                if (r0 + gid + 8 < H) yb[r0 + gid + 8] = acc[nb][1];
            }
        }
        return;
    }
    // gate+up: warps 0-7 hold gate rows, warps 8-15 the up rows of the same units
    constexpr int half = kTConsumers / 2;
    const int I = a.I;
    float *gbuf = epi;
    float *hbuf = epi + kTGuJ * kMaxTok;
    float *wbuf = epi + 2 * kTGuJ * kMaxTok;
    const int j0 = it.tile * kTGuJ;
    if (warp < half) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q;
            if (s < ntok) {
                gbuf[(16 * warp + gid) * kMaxTok + s] = acc[nb][0];
                gbuf[(16 * warp + gid + 8) * kMaxTok + s] = acc[nb][1];
            }
        }
    }
    consumers_sync();
    if (warp >= half) {
        const int lr = 16 * (warp - half) + gid;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q;
            if (s < ntok) {
                const float g0 = gbuf[lr * kMaxTok + s], g1 = gbuf[(lr + 8) * kMaxTok + s];
                const float h0 = g0 / (1.0f + expf(-g0)) * acc[nb][0];
                const float h1 = g1 / (1.0f + expf(-g1)) * acc[nb][1];
                hbuf[lr * kMaxTok + s] = h0;
                hbuf[(lr + 8) * kMaxTok + s] = h1;
                float *hb = a.h + (size_t)sh.pairs[s] * I + j0;
                if (j0 + lr < I) hb[lr] = h0;
                if (j0 + lr + 8 < I) hb[lr + 8] = h1;
            }
        }
    }
    consumers_sync();
    const int Gd = I / kGroup;
    for (int idx = warp; idx < ntok * 2; idx += kTConsumers) {
        const int s = idx >> 1, gg = idx & 1;
        const int gd = it.tile * 2 + gg;
        if (gd < Gd) {
            const float v0 = hbuf[(gg * 64 + lane) * kMaxTok + s];
            const float v1 = hbuf[(gg * 64 + 32 + lane) * kMaxTok + s];
            const int e = split_exponent(warp_max(fmaxf(fabsf(v0), fabsf(v1))));
            const float mul = ldexpf(1.0f, e);
            wbuf[warp * 64 + lane] = v0 * mul;
            wbuf[warp * 64 + 32 + lane] = v1 * mul;
            __syncwarp();
            const size_t cb = (size_t)sh.pairs[s] * Gd + gd;
            if (lane < 16) a.hcells[cb * 16 + lane] = make_unit<false>(wbuf + warp * 64, lane);
            if (lane == 0) a.hfac[cb] = ldexpf(1.0f, -e);
            __syncwarp();
        }
    }
    consumers_sync();
}

__global__ void __maxnreg__(120) k_moe_tma(const __grid_constant__ TmaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TShared sh;
    // 1024-byte alignment by an offset on the shared array itself, so the
    // compiler keeps shared-window addressing (LDS) for every access.
    uint8_t *ring = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint4 *cells = reinterpret_cast<uint4 *>(ring + kTStages * kTStage);
    float *fac = reinterpret_cast<float *>(ring + kTStages * kTStage + kTBudget);
    float *epi = fac + kTBudget / 256;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTStages; ++s) {
            tc05::mbar_init(&sh.full[s], 1);
            tc05::mbar_init(&sh.empty[s], kTConsumers);
        }
        tc05::fence_mbar_init();
    }
    __syncthreads();

    // gate+up needs the grouping (previous kernel) before its first load; the
    // down kernel's grouping finished before the previous kernel started, so
    // only its consumers (which read h) wait.
    if (a.mode == 0 || warp < kTConsumers) pdl_wait();
    pdl_trigger();

    const int nu = *a.n_used;
    const int tiles = a.mode == 0 ? (a.I + kTGuJ - 1) / kTGuJ : (a.H + kTDnRows - 1) / kTDnRows;
    const int total_items = nu > 0 ? a.pass_ofs[nu] * tiles : 0;
    const int i0 = (int)((long long)blockIdx.x * total_items / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * total_items / gridDim.x);
    const int ns = (a.G + 3) / 4;

    if (warp == kTConsumers) {
        // ---------------- producer
        if (lane == 0) {
            const int total = (i1 - i0) * ns;
            int cur = -1;
            TItem it{};
            bool ok = true;
            int issued = 0;
            for (int j = 0; j < total; ++j) {
                const int slot = j % kTStages;
                if (j >= kTStages &&
                    !tc05::mbar_wait(&sh.empty[slot], (uint32_t)(((j / kTStages) - 1) & 1), kTWait)) {
                    ok = false;
                    break;
                }
                const int item = i0 + j / ns, kb = j % ns;
                if (item != cur) {
                    it = t_item(a, nu, tiles, item);
                    cur = item;
                }
                int rowA, rowB;
                if (a.mode == 0) {
                    rowA = it.tile * kTGuJ;
                    rowB = a.I + it.tile * kTGuJ;
                } else {
                    rowA = it.tile * kTDnRows;
                    rowB = it.tile * kTDnRows + 128;
                }
                const uint32_t base = tc05::smem_addr(ring + slot * kTStage);
                const uint32_t fb = tc05::smem_addr(&sh.full[slot]);
                mbar_expect_tx(&sh.full[slot], (uint32_t)kTStage);
                tma_load3(base, &a.wmap, kb * 128, rowA, it.e, fb);
                tma_load3(base + 128 * 128, &a.wmap, kb * 128, rowB, it.e, fb);
                tma_load3(base + kTStageW, &a.smap, kb * 4, rowA, it.e, fb);
                tma_load3(base + kTStageW + 128 * 16, &a.smap, kb * 4, rowB, it.e, fb);
                issued = j + 1;
            }
            if (!ok) atomicOr(a.status, 2);
            // Drain: every load issued must land before the CTA may exit.
            for (int j = (issued > kTStages ? issued - kTStages : 0); j < issued; ++j)
                tc05::mbar_wait(&sh.full[j % kTStages], (uint32_t)((j / kTStages) & 1), kTWait);
        }
    } else {
        // ---------------- consumers
        int j = 0, cur_pi = -1;
        bool failed = false;
        for (int item = i0; item < i1; ++item) {
            const TItem it = t_item(a, nu, tiles, item);
            const int pi = item / tiles;
            const bool reuse = pi == cur_pi;
            if (!reuse) {
                consumers_sync();  // previous epilogue is done with sh.rows / pairs
                if (threadIdx.x < it.ntok) {
                    const int p = a.list[it.beg + threadIdx.x];
                    sh.pairs[threadIdx.x] = p;
                    sh.rows[threadIdx.x] = a.mode == 0 ? p / a.k : p;
                }
                cur_pi = pi;
            }
            if (it.ntok <= 4) {
                float acc[1][2];
                t_consume_item<1>(a, sh, ring, cells, fac, it.ntok, reuse, j, failed, acc);
                t_epilogue<1>(a, sh, epi, it, acc);
            } else {
                float acc[2][2];
                t_consume_item<2>(a, sh, ring, cells, fac, it.ntok, reuse, j, failed, acc);
                t_epilogue<2>(a, sh, epi, it, acc);
            }
        }
        if (failed && (threadIdx.x & 31) == 0) atomicOr(a.status, 2);
    }
    __syncthreads();
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_maps(TmaArgs &a, const uint8_t *wq, const float *ws, int E, int rows, int K) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int G = K / kGroup;
    {
        cuuint64_t dims[3] = {(cuuint64_t)K / 2, (cuuint64_t)rows, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)K / 2, (cuuint64_t)rows * (K / 2)};
        cuuint32_t box[3] = {128, 128, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(wq), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)G, (cuuint64_t)rows, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)G * 4, (cuuint64_t)rows * G * 4};
        cuuint32_t box[3] = {4, 128, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&a.smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ws), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

}  // namespace

bool tma_moe_supported(const MoeDims &m) {
    // tensor maps need 16-byte aligned bases and 16-byte strides (scale rows of
    // K/64 floats: K/64 a multiple of 4)
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    return encode_fn() != nullptr && (m.H / kGroup) % 4 == 0 && (m.I / kGroup) % 4 == 0 &&
           a16(m.gu_q) && a16(m.gu_s) && a16(m.dn_q) && a16(m.dn_s);
}

cudaError_t launch_moe_tma(const MoeDims &m, int mode, const void *cells, const float *cfac, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hcells,
                           float *hfac, float *y, int32_t *status, cudaStream_t st) {
    TmaArgs a;
    memset(&a, 0, sizeof(a));
    a.mode = mode;
    a.I = m.I;
    a.H = m.H;
    a.k = k;
    a.offsets = offsets; a.list = list; a.uexp = uexp; a.n_used = n_used; a.pass_ofs = pass_ofs;
    a.cells = static_cast<const uint4 *>(cells);
    a.cfac = cfac;
    a.h = h;
    a.hcells = static_cast<uint4 *>(hcells);
    a.hfac = hfac;
    a.y = y;
    a.status = status;
    bool ok;
    if (mode == 0) {
        a.G = m.H / kGroup;
        ok = make_maps(a, m.gu_q, m.gu_s, m.E, 2 * m.I, m.H);
    } else {
        a.G = m.I / kGroup;
        ok = make_maps(a, m.dn_q, m.dn_s, m.E, m.H, m.I);
    }
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = set_smem(k_moe_tma, kTSmem);
    if (e != cudaSuccess) return e;
    const int grid = sm_count() * max_ctas_per_sm(k_moe_tma, kTThreads, kTSmem);
    return launch(k_moe_tma, dim3(grid), dim3(kTThreads), (size_t)kTSmem, st, true, a);
}

}  // namespace qmv
