// qmv_moe_tma.cu - MoE decode gate+up and down kernels fed by the Tensor
// Memory Accelerator.
//
// Same arithmetic as k_gate_up / k_down (qmv_moe.cu): exact fp16 weights in
// registers, fp16 hi/lo activations, warp MMA per 64-group, group scale in
// fp32 (colibri PR #418, "qmatmul_gate_up.comp + coli_vk_gate_up",
// "coli_vk_expert_group", "grouped scales in the Vulkan kernels"). What
// changes is how the operands arrive: one producer warp fills a 4-stage ring
// guarded by mbarriers. A stage holds 256 weight rows x 4 groups (tensor-map
// loads of 128 or 256 rows x 128 bytes, 128-byte swizzle), their scales, and
// the activation units and factors of the same 4 groups for every token of
// the pass (one bulk copy of the pass-packed block, or one per token), so
// the 8 consumer warps spend no instructions on copies and never wait on a
// block barrier inside an item. Consumer warp w owns two 16-row tiles, stage
// rows 16w..16w+15 and 128+16w..128+16w+15: for gate+up the gate rows and
// the up rows of the same 16 hidden units; for down and dense, two row tiles.
// The dense int4-gs64 GEMV (qmv_int4_gs) runs as a third mode: one matrix (or
// a pair sharing x), its S tokens in passes of 8, row tiles of 256.
//
// Work split: the stages of all items (item-major) are shared out over the
// CTAs, by the grouping kernel's cost-balanced plan when there is one, else
// evenly. An item whose stages fall to several CTAs is finished by the last
// of them to publish its partial sums (an acquire-release counter; nobody
// waits for anybody), which adds the partial sums in CTA order and writes
// the item. A tenth warp keeps that off the consumers' path: it publishes
// the item a CTA starts in while the consumers go on, and fetches the next
// CTA's partial sums of the item a CTA ends in while the range still runs.
//
// Every mbarrier wait is bounded. A consumer warp whose wait runs out stops
// waiting but keeps computing (on whatever the slot holds) and keeps every
// barrier, so all warps finish; the producer gives up when the consumers stop
// releasing slots and drains its loads before exiting; bit 1 of the status
// word records the failure (the outputs are then not valid).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_rows.cuh"
#include "tc05.cuh"

namespace qmv {

namespace {

constexpr int kTConsumers = 8;                       // consumer warps, two 16-row tiles each
constexpr int kTSync = kTConsumers + 1;              // warp of the split items' counters
constexpr int kTThreads = 32 * (kTConsumers + 2);    // consumers, producer, sync warp
// Registers: warps are spread round-robin over the 4 SM sub-partitions, so
// one holds 3 of the 10 warps; 3 x 32 x 168 fits its 16,384 registers.
constexpr int kTRegBound = 3 * 4 * 32;               // launch bound giving 168 registers
constexpr int kTStages = 4;
constexpr int kTRows = 256;                          // weight rows per stage
constexpr int kTStageW = kTRows * 128;               // 32 KB of packed weights
constexpr int kTStageS = kTRows * 16;                // 4 KB of scales
constexpr int kTActTok = 4 * 16 * 16;                // units of 4 groups, one token: 1 KB
constexpr int kTFacTok = 32;                         // (factor, offset_init) of 4 groups, one token
// records, then units: the order of a pass-packed block (one copy)
constexpr int kTOffF = kTStageW + kTStageS;
constexpr int kTOffA = kTOffF + kMaxTok * kTFacTok;
constexpr int kTStage = (kTOffA + kMaxTok * kTActTok + 1023) / 1024 * 1024;  // 45 KB
static_assert(kTOffA - kTOffF + kMaxTok * kTActTok == kPackedStage, "pass-packed block layout");
constexpr int kTGuJ = 128;                           // hidden units per gate+up item
constexpr int kTDnRows = 256;                        // output rows per down item
constexpr int kTEpi = (kTGuJ * kMaxTok + kTConsumers * 64) * 4;  // h of an item, split scratch
constexpr int kTTail = kTRows * kMaxTok * 4;        // the next CTA's partial sums of the last item
constexpr int kTSmem = kTStages * kTStage + kTEpi + kTTail + 1024;
constexpr uint32_t kTWait = 1u << 24;
constexpr uint32_t kTPoll = 1u << 16;                // sync warp: polls of a counter (~0.5 us apart)

static_assert(kTStage % 1024 == 0, "stages must stay 1024-aligned for the 128B swizzle");
static_assert(kSkPartFloats == 2 * kTRows * kMaxTok, "partial-sum slots must match the stage");

struct TmaArgs {
    CUtensorMap wmap;    // weights: uint8 [E][rows][K/2], box 128 B x 128 rows, 128B swizzle
    CUtensorMap smap;    // scales: f32 [E][rows][K/64], box 4 x 128 rows
    CUtensorMap wmap2;   // dense pair: the second matrix's maps (row tiles tiles0 ..)
    CUtensorMap smap2;
    int H2, tiles0;      // dense pair: rows of the second matrix, row tiles of the first
    float *y2;           // dense pair: its output [S][H2]
    int mode;            // 0: gate+up, 1: down, 2: dense GEMV (one matrix, tokens 0..S-1)
    int G, I, H, k;
    int S;               // dense: tokens
    int packed;          // activation units pass-packed (else per row)
    const int32_t *offsets, *list, *uexp, *n_used, *pass_ofs;
    const uint4 *cells;  // activation units (int4 form of make_unit_s): per row
                         // [row][G][16], or pass-packed blocks of kPackedStage
                         // bytes [pass][G/4]
    const float *cfac;   // their (factor, offset_init) records [row][G][2] (per-row
                         // layout only)
    float *h;            // gate+up: h fp32 [P][I]
    uint4 *hcells;       // gate+up: units of h [P][I/64][16], or pass-packed blocks
    float *hfac;         // gate+up: records of h [P][I/64][2] (per-row layout only)
    float *y;            // down: y [P][H]; dense: y [S][H]
    uint16_t *ybf;       // dense, first matrix: y rounded to bf16 [S][H] instead of y
    const int4 *ptab;    // the grouping kernel's pass table, or null (PlanArgs)
    const int4 *plan;    // this mode's CTA plan [g + 1] (PlanArgs), or null
    int32_t *status;
    int32_t *cnt;        // per CTA: contributors done on the split item that starts in it
    float *part;         // per CTA: partial sums [2][kTRows][kMaxTok] (head / tail item)
    int skew_ns;         // test hook: the consumers of odd CTAs start this much later
};

__device__ __forceinline__ void tma_load3(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                          int c2, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned ends, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
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

// Walks the passes of the grouped pairs in order. `lo` indexes the used
// experts (uexp); passes of used expert lo are pass_ofs[lo] .. pass_ofs[lo+1]-1.
struct PassCursor {
    int lo, pi, e, beg, ntok;

    __device__ __forceinline__ void seek(const TmaArgs &a, int nu, int p) {
        pi = -1;
        if (a.mode == 2 || a.ptab) {
            to(a, p);
            return;
        }
        int l = 0, hgh = nu - 1;
        while (l < hgh) {
            const int mid = (l + hgh + 1) >> 1;
            if (a.pass_ofs[mid] <= p) l = mid; else hgh = mid - 1;
        }
        lo = l;
        pi = -1;
        to(a, p);
    }
    // Moves forward to pass p (p >= the current pass).
    __device__ __forceinline__ void to(const TmaArgs &a, int p) {
        if (p == pi) return;
        if (a.mode == 2) {  // dense: pass p is tokens 8p .. 8p + 7 of the one matrix
            pi = p;
            e = 0;
            beg = p * kMaxTok;
            ntok = min(kMaxTok, a.S - beg);
            return;
        }
        if (a.ptab) {  // one load instead of a walk over pass_ofs, uexp and offsets
            const int4 t = a.ptab[p];
            pi = p;
            e = t.x;
            beg = t.y;
            ntok = t.z;
            return;
        }
        while (a.pass_ofs[lo + 1] <= p) ++lo;
        pi = p;
        e = a.uexp[lo];
        const int pass = p - a.pass_ofs[lo];
        const int b = a.offsets[e], cnt = a.offsets[e + 1] - b;
        beg = b + pass * kMaxTok;
        ntok = min(kMaxTok, cnt - pass * kMaxTok);
    }
};

// Places a cursor on pass p, the first pass of this CTA: from the plan's
// entry (no load) when there is a plan, else by seek.
__device__ __forceinline__ void start_cursor(PassCursor &c, const TmaArgs &a, int nu, int p,
                                             int4 pl0) {
    if (a.plan) {
        c.pi = p;
        c.e = pl0.y;
        c.beg = pl0.z;
        c.ntok = pl0.w;
    } else {
        c.seek(a, nu, p);
    }
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Shared-memory row (within a 16-row tile) that holds MMA row gid (and gid + 8
// at +8). With the 128-byte swizzle, rows {0,2,4,6} and {1,3,5,7} each spread
// one 16-byte chunk pair over all 32 banks, so the 64-bit weight loads of a
// half-warp are conflict-free.
__device__ __forceinline__ int tile_row(int gid) { return 2 * (gid & 3) + (gid >> 2); }

// Consumer warp w owns two 16-row tiles of a stage: A = stage rows
// 16w..16w+15 and B = rows 128+16w..128+16w+15. For gate+up that is the gate
// and the up rows of the same 16 hidden units (pairs of the fused SiLU live in
// one warp); for down and dense, two independent row tiles. Both tiles take
// the same activation fragments, loaded once.
constexpr int kTRowB = 128;

// Fragments of one group of this warp's two tiles.
template <int NB>
struct GroupFrag {
    uint2 a0, a8, b0, b8;
    uint4 bu[NB][2];
};

template <int NB, int GL>
__device__ __forceinline__ void group_load(const uint8_t *waA, const uint8_t *waB, int pr, int q,
                                           const uint4 *const bp0[NB], GroupFrag<NB> &g) {
    const int off = (((2 * GL + (q >> 1)) ^ pr) << 4) + ((q & 1) << 3);
    g.a0 = *reinterpret_cast<const uint2 *>(waA + off);
    g.a8 = *reinterpret_cast<const uint2 *>(waA + 1024 + off);
    g.b0 = *reinterpret_cast<const uint2 *>(waB + off);
    g.b8 = *reinterpret_cast<const uint2 *>(waB + 1024 + off);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        g.bu[nb][0] = bp0[nb][GL * 16];
        g.bu[nb][1] = bp0[nb][GL * 16 + 8];
    }
}

// d = 2^-24 * sum (nibble - 8) * v over the group (tile2_group_int4s); the
// exact 2^24 comes back before the group scale and the activation factor.
// fp[nb]: the (factor, offset_init) records of the four groups of token
// block nb. c[tile][GL & 1][nb][row gid, gid + 8].
template <int NB, int GL>
__device__ __forceinline__ void group_math(const GroupFrag<NB> &g, float sA0, float sA8, float sB0,
                                           float sB8, const float *const fp[NB],
                                           float c[2][2][NB][2]) {
    float dA[NB][4], dB[NB][4], ci[NB], f[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const float2 r = reinterpret_cast<const float2 *>(fp[nb])[GL];
        f[nb] = r.x;
        ci[nb] = r.y;
    }
    tile2_group_int4s<NB>(g.a0, g.a8, g.b0, g.b8, g.bu, ci, dA, dB);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        c[0][GL & 1][nb][0] = fmaf(sA0 * f[nb], (dA[nb][0] + dA[nb][1]) * 0x1p24f, c[0][GL & 1][nb][0]);
        c[0][GL & 1][nb][1] = fmaf(sA8 * f[nb], (dA[nb][2] + dA[nb][3]) * 0x1p24f, c[0][GL & 1][nb][1]);
        c[1][GL & 1][nb][0] = fmaf(sB0 * f[nb], (dB[nb][0] + dB[nb][1]) * 0x1p24f, c[1][GL & 1][nb][0]);
        c[1][GL & 1][nb][1] = fmaf(sB8 * f[nb], (dB[nb][2] + dB[nb][3]) * 0x1p24f, c[1][GL & 1][nb][1]);
    }
}

// One stage of this warp's two tiles: four groups, the next group's
// fragments loaded before the current one's arithmetic.
template <int NB>
__device__ __forceinline__ void compute_stage(const uint8_t *slot, int warp,
                                              const uint4 *const bp[NB],
                                              const float *const fp[NB], float c[2][2][NB][2]) {
    const int lane = threadIdx.x & 31, q = lane & 3, pr = tile_row(lane >> 2);
    const int rA = 16 * warp + pr, rB = kTRowB + 16 * warp + pr;
    // the four groups' scales of a row are a 16-byte vector
    const float4 *sv = reinterpret_cast<const float4 *>(slot + kTStageW);
    const float4 sA0 = sv[rA], sA8 = sv[rA + 8], sB0 = sv[rB], sB8 = sv[rB + 8];
    const uint8_t *waA = slot + rA * 128, *waB = slot + rB * 128;
    GroupFrag<NB> g0, g1;
    group_load<NB, 0>(waA, waB, pr, q, bp, g0);
    group_load<NB, 1>(waA, waB, pr, q, bp, g1);
    group_math<NB, 0>(g0, sA0.x, sA8.x, sB0.x, sB8.x, fp, c);
    group_load<NB, 2>(waA, waB, pr, q, bp, g0);
    group_math<NB, 1>(g1, sA0.y, sA8.y, sB0.y, sB8.y, fp, c);
    group_load<NB, 3>(waA, waB, pr, q, bp, g1);
    group_math<NB, 2>(g0, sA0.z, sA8.z, sB0.z, sB8.z, fp, c);
    group_math<NB, 3>(g1, sA0.w, sA8.w, sB0.w, sB8.w, fp, c);
}

struct TShared {
    uint64_t full[kTStages];
    uint64_t empty[kTStages];
    uint64_t hp;   // the head item's partial sums are stored (each consumer warp arrives)
    uint64_t hd;   // the sync warp has counted the head item (defer is valid)
    uint64_t tp;   // the sync warp's verdict on the last item (ready is valid)
    long long ub[kSkMaxCtas + 1];  // first stage of each CTA's range (consumers' copy)
    int pairs[kMaxTok];
    int last;
    int h_bf, h_n;        // the head item's first contributor and contributor count
    volatile int stop;    // consumers are at the last item's end: stop polling
    volatile int ready;   // the next CTA's partial sums of the last item are in shared memory
    volatile int defer;   // this CTA was the head item's last contributor: it writes the item
};

// Consumer side of stages [kb0, kb1) of one item. A wait that runs out sets
// `failed`; from then on the warp stops waiting but keeps the same sequence
// of barriers, so every warp reaches the end. acc[tile][nb]: rows
// tile_row(gid) and +8 of the warp's tile A / B, token 4nb+q.
template <int NB>
__device__ __forceinline__ void t_consume(TShared &sh, const uint8_t *ring, int ntok, int kb0,
                                          int kb1, int &j, bool &failed, float acc[2][NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    int ob[NB], of[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        ob[nb] = min(4 * nb + (gid >> 1), ntok - 1) * (kTActTok / 16) + q * 2 + (gid & 1);
        of[nb] = min(4 * nb + q, ntok - 1) * (kTFacTok / 4);
    }
    float c[2][2][NB][2];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) c[t][h2][nb][0] = c[t][h2][nb][1] = 0.f;
    for (int kb = kb0; kb < kb1; ++kb, ++j) {
        const int slot = j % kTStages;
        if (!failed &&
            !tc05::mbar_wait(&sh.full[slot], (uint32_t)((j / kTStages) & 1), kTWait))
            failed = true;
        const uint8_t *sp = ring + slot * kTStage;
        const uint4 *bp[NB];
        const float *fp[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            bp[nb] = reinterpret_cast<const uint4 *>(sp + kTOffA) + ob[nb];
            fp[nb] = reinterpret_cast<const float *>(sp + kTOffF) + of[nb];
        }
        compute_stage<NB>(sp, warp, bp, fp, c);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.empty[slot]);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            acc[t][nb][0] = c[t][0][nb][0] + c[t][1][nb][0];
            acc[t][nb][1] = c[t][0][nb][1] + c[t][1][nb][1];
        }
}

template <int NB>
__device__ __forceinline__ void t_epilogue(const TmaArgs &a, const TShared &sh, float *epi,
                                           int tile, int ntok, int pi, const float acc[2][NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3;
    const int pr = tile_row(lane >> 2);
    if (a.mode != 0) {
        const bool second = tile >= a.tiles0;  // dense pair: the second matrix
        const int H = second ? a.H2 : a.H;
        const int base = (second ? tile - a.tiles0 : tile) * kTDnRows + 16 * warp + pr;
        float *yb = second ? a.y2 : a.y;
        uint16_t *hb = second ? nullptr : a.ybf;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int r0 = base + t * kTRowB;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int s = 4 * nb + q;
                if (s < ntok) {
                    const size_t o = (size_t)sh.pairs[s] * H + r0;
                    if (r0 < H) store_y(yb, hb, o, acc[t][nb][0]);
                    if (r0 + 8 < H) store_y(yb, hb, o + 8, acc[t][nb][1]);
                }
            }
        }
        return;
    }
    // gate+up: tile A holds the gate rows, tile B the up rows of the same units
    const int I = a.I;
    float *hbuf = epi;
    float *wbuf = epi + kTGuJ * kMaxTok;
    const int j0 = tile * kTGuJ;
    const int lr = 16 * warp + pr;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int s = 4 * nb + q;
        if (s < ntok) {
            const float g0 = acc[0][nb][0], g1 = acc[0][nb][1];
            const float h0 = g0 / (1.0f + expf(-g0)) * acc[1][nb][0];
            const float h1 = g1 / (1.0f + expf(-g1)) * acc[1][nb][1];
            hbuf[lr * kMaxTok + s] = h0;
            hbuf[(lr + 8) * kMaxTok + s] = h1;
            float *hg = a.h + (size_t)sh.pairs[s] * I + j0;
            if (j0 + lr < I) hg[lr] = h0;
            if (j0 + lr + 8 < I) hg[lr + 8] = h1;
        }
    }
    consumers_sync();
    const int Gd = I / kGroup;
    for (int idx = warp; idx < ntok * 2; idx += kTConsumers) {
        const int s = idx >> 1, gg = idx & 1;
        const int gd = tile * 2 + gg;
        if (gd < Gd) {
            const float v0 = hbuf[(gg * 64 + lane) * kMaxTok + s];
            const float v1 = hbuf[(gg * 64 + 32 + lane) * kMaxTok + s];
            const int e = split_exponent(warp_max(fmaxf(fabsf(v0), fabsf(v1))));
            const float mul = ldexpf(1.0f, e);
            wbuf[warp * 64 + lane] = v0 * mul;
            wbuf[warp * 64 + 32 + lane] = v1 * mul;
            const float2 rec =
                make_float2(ldexpf(1.0f, -e), offset_init(warp_sum(v0 * mul + v1 * mul)));
            __syncwarp();
            if (a.packed) {
                // down's pass pi, slot s (down groups the pairs as gate+up does)
                uint8_t *blk = reinterpret_cast<uint8_t *>(a.hcells) +
                               ((size_t)pi * (Gd / 4) + gd / 4) * kPackedStage;
                if (lane < 16)
                    reinterpret_cast<uint4 *>(blk + kPackedHead + s * 1024 + (gd % 4) * 256)[lane] =
                        make_unit_s(wbuf + warp * 64, lane);
                if (lane == 0) reinterpret_cast<float2 *>(blk)[s * 4 + gd % 4] = rec;
            } else {
                const size_t cb = (size_t)sh.pairs[s] * Gd + gd;
                if (lane < 16) a.hcells[cb * 16 + lane] = make_unit_s(wbuf + warp * 64, lane);
                if (lane == 0) reinterpret_cast<float2 *>(a.hfac)[cb] = rec;
            }
            __syncwarp();
        }
    }
    consumers_sync();
}

// The CTA whose range holds stage u (ub: first stage of each CTA, g + 1 entries).
__device__ __forceinline__ int unit_owner(const long long *ub, int g, long long u) {
    int l = 0, hgh = g - 1;
    while (l < hgh) {
        const int mid = (l + hgh + 1) >> 1;
        if (ub[mid] <= u) l = mid; else hgh = mid - 1;
    }
    return l;
}

// Split items. An item whose stages fall to several CTAs (contributors
// bf .. bl, those with non-empty ranges) is written by one of them with the
// sum of every contributor's partial sums, added in CTA order from zero (so
// the result does not depend on who writes it). Counter cnt[bf] counts the
// contributors that have published (stored their partial sums, then a
// release at gpu scope); a contributor that finds all the others published
// writes the item and clears the counter for the next launch. No CTA waits
// for another: whoever publishes last writes.
//
// The item a CTA starts in (begun by an earlier CTA) comes at the start of
// its range, where a block barrier and a counter round trip would stall the
// consumers while the ring is full; its publication goes to the sync warp
// (the consumers store and move on; should the count show this CTA last,
// it writes the item after its range). The item a CTA ends in comes at the
// end of its range: when exactly one later CTA holds the rest of it, the
// sync warp watches that CTA's publication during the range and copies its
// partial sums into shared memory, so the item ends without a round trip to
// L2; if they are not there by the end, the CTA publishes instead.

// This CTA's partial sums of an item: slot 0 if the item is the first of its
// range, else slot 1.
template <int NB>
__device__ __forceinline__ void t_store_part(const TmaArgs &a, int ntok, bool head,
                                             const float acc[2][NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3;
    const int r = 16 * warp + tile_row(lane >> 2);
    float *mine = a.part + ((size_t)blockIdx.x * 2 + (head ? 0 : 1)) * (kTRows * kMaxTok);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q, rt = r + t * kTRowB;
            if (s < ntok) {
                mine[rt * kMaxTok + s] = acc[t][nb][0];
                mine[(rt + 8) * kMaxTok + s] = acc[t][nb][1];
            }
        }
}

// Contributors of the item whose stages begin at `first`: the first one and
// how many (CTAs of [bf, bl] with a non-empty range all hold its stages).
__device__ __forceinline__ void t_contributors(const long long *ub, int g, long long first,
                                               int ns, int &bf, int &n) {
    bf = unit_owner(ub, g, first);
    const int bl = unit_owner(ub, g, first + ns - 1);
    n = 0;
    for (int c = bf; c <= bl; ++c) n += ub[c + 1] > ub[c];
}

// Publishes (acquire-release at gpu scope: this CTA's partials, then the
// others'); true if every other contributor had published before.
__device__ __forceinline__ bool t_publish(const TmaArgs &a, int bf, int n) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(&a.cnt[bf]) : "memory");
    return old == n - 1;
}

// Every contributor's partial sums of the item, added in CTA order from zero;
// clears the counter for the next launch.
template <int NB>
__device__ __forceinline__ void t_gather(const TmaArgs &a, const TShared &sh, int ntok, int item,
                                         int ns, float acc[2][NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3;
    const int g = gridDim.x;
    const int r = 16 * warp + tile_row(lane >> 2);
    const long long first = (long long)item * ns;
    const int bf = unit_owner(sh.ub, g, first), bl = unit_owner(sh.ub, g, first + ns - 1);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[t][nb][0] = acc[t][nb][1] = 0.f;
    for (int c = bf; c <= bl; ++c) {
        const long long c0 = sh.ub[c];
        if (sh.ub[c + 1] <= c0) continue;
        const float *pc =
            a.part + ((size_t)c * 2 + (c0 >= first ? 0 : 1)) * (kTRows * kMaxTok);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                const int s = 4 * nb + q, rt = r + t * kTRowB;
                if (s < ntok) {
                    acc[t][nb][0] += __ldcg(pc + rt * kMaxTok + s);
                    acc[t][nb][1] += __ldcg(pc + (rt + 8) * kMaxTok + s);
                }
            }
    }
    if (threadIdx.x == 0) a.cnt[bf] = 0;
}

// The item at hand, synchronously: store, publish (thread 0, between two
// barriers: the barrier orders every consumer's stores before the release;
// the acquire orders the others' partials before the readers' barrier),
// and gather if this CTA published last. True: the caller writes the item.
template <int NB>
__device__ __forceinline__ bool t_combine(const TmaArgs &a, TShared &sh, int ntok, int item,
                                          bool head, int ns, float acc[2][NB][2]) {
    t_store_part<NB>(a, ntok, head, acc);
    consumers_sync();
    if (threadIdx.x == 0) {
        int bf, n;
        t_contributors(sh.ub, gridDim.x, (long long)item * ns, ns, bf, n);
        sh.last = t_publish(a, bf, n);
    }
    consumers_sync();
    if (!sh.last) return false;
    t_gather<NB>(a, sh, ntok, item, ns, acc);
    return true;
}

// The last item, finished with the next CTA's partial sums that the sync
// warp copied into shared memory (tail: [kTRows][kMaxTok]): (0 + own) +
// next, the order t_gather adds them in.
template <int NB>
__device__ __forceinline__ void t_add_tail(const float *tail, int ntok, float acc[2][NB][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = lane & 3;
    const int r = 16 * warp + tile_row(lane >> 2);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q, rt = r + t * kTRowB;
            if (s < ntok) {
                acc[t][nb][0] = (0.f + acc[t][nb][0]) + tail[rt * kMaxTok + s];
                acc[t][nb][1] = (0.f + acc[t][nb][1]) + tail[(rt + 8) * kMaxTok + s];
            }
        }
}

// The split-item roles of a CTA's range [u0, u1) of stages (ns an item; u2:
// where the next CTA's range ends). head_async: its first item began in an
// earlier CTA and the range goes on past it (published by the sync warp).
// tail_next: its last item began inside the range and the next CTA holds all
// the rest of it (the sync warp fetches that CTA's partial sums).
struct TRoles {
    bool head_async, tail_next;
};
__device__ __forceinline__ TRoles t_roles(long long u0, long long u1, long long u2, int ns, int g) {
    TRoles r{false, false};
    if (u1 <= u0) return r;
    const long long hi = u0 / ns, ti = (u1 - 1) / ns;
    r.head_async = u0 % ns != 0 && ti != hi;
    r.tail_next = ti != hi && u1 % ns != 0 && (int)blockIdx.x + 1 < g && u2 >= (ti + 1) * ns;
    return r;
}

// Consumers, after the stages of an item: write it, or publish it and write
// it if this CTA is its last contributor (see t_store_part).
template <int NB>
__device__ __forceinline__ void t_finish(const TmaArgs &a, TShared &sh, float *epi, int tile,
                                         int ntok, int pi, int item, bool head, int ns, bool whole,
                                         bool head_pub, bool tail_fin, float acc[2][NB][2]) {
    bool write = whole;
    if (head_pub) {  // store and move on; the sync warp publishes
        t_store_part<NB>(a, ntok, true, acc);
        if (threadIdx.x == 0) {
            int bf, n;
            t_contributors(sh.ub, gridDim.x, (long long)item * ns, ns, bf, n);
            sh.h_bf = bf;
            sh.h_n = n;
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.hp);
    } else if (!whole) {
        bool fetched = false;
        if (tail_fin) {  // the next CTA's partial sums, if the sync warp has them
            if ((threadIdx.x & 31) == 0) sh.stop = 1;
            const bool ok = tc05::mbar_wait(&sh.tp, 0u, kTWait);
            if (!ok && (threadIdx.x & 31) == 0) atomicOr(a.status, 2);
            fetched = ok && sh.ready;
        }
        if (fetched) {
            t_add_tail<NB>(epi + kTEpi / 4, ntok, acc);
            if (threadIdx.x == 0) a.cnt[blockIdx.x] = 0;  // every other contributor is done
            write = true;
        } else {
            write = t_combine<NB>(a, sh, ntok, item, head, ns, acc);
        }
    }
    if (write) t_epilogue<NB>(a, sh, epi, tile, ntok, pi, acc);
}

// Consumers, after their range: the first item, which this CTA published
// last (rare: its first contributor finishes its part at the end of its own
// range). Out of line, so it costs the item loop no registers.
__device__ __noinline__ void t_write_deferred(const TmaArgs &a, TShared &sh, float *epi, int nu,
                                              int item, int tiles, int ns) {
    const int pi = item / tiles, tile = item - pi * tiles;
    PassCursor hc;
    hc.seek(a, nu, pi);
    consumers_sync();  // the last epilogue is done with sh.pairs
    if (threadIdx.x < hc.ntok)
        sh.pairs[threadIdx.x] = a.mode == 2 ? hc.beg + threadIdx.x : a.list[hc.beg + threadIdx.x];
    consumers_sync();
    if (hc.ntok <= 4) {
        float acc[2][1][2];
        t_gather<1>(a, sh, hc.ntok, item, ns, acc);
        t_epilogue<1>(a, sh, epi, tile, hc.ntok, pi, acc);
    } else {
        float acc[2][2][2];
        t_gather<2>(a, sh, hc.ntok, item, ns, acc);
        t_epilogue<2>(a, sh, epi, tile, hc.ntok, pi, acc);
    }
}

__global__ void __launch_bounds__(kTRegBound, 1) k_moe_tma(const __grid_constant__ TmaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TShared sh;
    // 1024-byte alignment by an offset on the shared array itself, so the
    // compiler keeps shared-window addressing (LDS) for every access.
    uint8_t *ring = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    float *epi = reinterpret_cast<float *>(ring + kTStages * kTStage);
    float *tail = reinterpret_cast<float *>(ring + kTStages * kTStage + kTEpi);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == kTConsumers && lane == 0) {  // the tensor-map descriptors, early
        prefetch_tmap(&a.wmap);
        prefetch_tmap(&a.smap);
        if (a.H2 > 0) {
            prefetch_tmap(&a.wmap2);
            prefetch_tmap(&a.smap2);
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTStages; ++s) {
            tc05::mbar_init(&sh.full[s], 1);
            tc05::mbar_init(&sh.empty[s], kTConsumers);
        }
        tc05::mbar_init(&sh.hp, kTConsumers);
        tc05::mbar_init(&sh.hd, 1);
        tc05::mbar_init(&sh.tp, 1);
        sh.stop = 0;
        sh.ready = 0;
        sh.defer = 0;
        tc05::fence_mbar_init();
    }
    __syncthreads();

    // gate+up needs the grouping (previous kernel) before its first load. The
    // down kernel's grouping finished before the previous kernel started, and
    // the dense GEMV has none, so their producers wait only before their first
    // copy of activation units (below).
    if (a.mode == 0 || warp != kTConsumers) pdl_wait();
    pdl_trigger();

    const int tiles = a.mode == 0 ? (a.I + kTGuJ - 1) / kTGuJ
                                  : a.tiles0 + (a.H2 + kTDnRows - 1) / kTDnRows;
    const int ns = a.G / 4;
    const int g = gridDim.x;
    // Stage-level split: CTA b takes stages [u0, u1) of the item-major sequence
    // (items pass-major): the grouping kernel's cost-balanced plan, or else an
    // even split [U*b/g, U*(b+1)/g).
    int nu = 1;
    long long U, u0, u1;
    int4 pl0 = make_int4(0, 0, 0, 0);  // the plan's first pass of this CTA
    if (a.plan) {
        pl0 = a.plan[blockIdx.x];
        U = a.plan[g].x;
        u0 = pl0.x;
        u1 = a.plan[blockIdx.x + 1].x;
    } else {
        nu = a.mode == 2 ? 1 : *a.n_used;
        const int passes =
            a.mode == 2 ? (a.S + kMaxTok - 1) / kMaxTok : (nu > 0 ? a.pass_ofs[nu] : 0);
        U = (long long)passes * tiles * ns;
        u0 = (long long)blockIdx.x * U / g;
        u1 = (long long)(blockIdx.x + 1) * U / g;
    }
    // first stage of CTA i's range
    auto ub_at = [&](int i) -> long long {
        return a.plan ? (long long)a.plan[i].x : (long long)i * U / g;
    };

    if (warp == kTConsumers) {
        // ---------------- producer (whole warp; lane 0 owns the barriers)
        // Down and dense: the weights of the first kTStages stages are requested
        // before the previous kernel (which writes the activation units) has
        // finished; their activation copies only after it has.
        const int total = (int)(u1 - u0);
        const int pre = a.mode != 0 ? min(total, kTStages) : 0;
        const int item0 = (int)(u0 / ns), kb_0 = (int)(u0 - (long long)item0 * ns);
        PassCursor pc;
        if (total > 0) start_cursor(pc, a, nu, item0 / tiles, pl0);
        auto weights = [&](int slot, int item, int kb, const PassCursor &c) {
            const int pi = item / tiles, tile = item - pi * tiles;
            const int rowA = a.mode == 0 ? tile * kTGuJ : tile * kTDnRows;
            const int rowB = a.mode == 0 ? a.I + tile * kTGuJ : tile * kTDnRows + 128;
            const uint32_t base = tc05::smem_addr(ring + slot * kTStage);
            const uint32_t fb = tc05::smem_addr(&sh.full[slot]);
            const uint32_t act = a.packed ? (uint32_t)(kMaxTok * kTFacTok + c.ntok * kTActTok)
                                          : (uint32_t)(c.ntok * (kTActTok + kTFacTok));
            mbar_expect_tx(&sh.full[slot], (uint32_t)(kTStageW + kTStageS) + act);
            if (a.mode == 0) {  // gate and up rows: two 128-row boxes each
                tma_load3(base, &a.wmap, kb * 128, rowA, c.e, fb);
                tma_load3(base + 128 * 128, &a.wmap, kb * 128, rowB, c.e, fb);
                tma_load3(base + kTStageW, &a.smap, kb * 4, rowA, c.e, fb);
                tma_load3(base + kTStageW + 128 * 16, &a.smap, kb * 4, rowB, c.e, fb);
            } else if (tile < a.tiles0) {  // 256 consecutive rows: one box each
                tma_load3(base, &a.wmap, kb * 128, rowA, c.e, fb);
                tma_load3(base + kTStageW, &a.smap, kb * 4, rowA, c.e, fb);
            } else {                       // the second matrix of a dense pair
                const int r2 = (tile - a.tiles0) * kTDnRows;
                tma_load3(base, &a.wmap2, kb * 128, r2, 0, fb);
                tma_load3(base + kTStageW, &a.smap2, kb * 4, r2, 0, fb);
            }
        };
        if (pre > 0) {
            int item = item0, kb = kb_0;
            PassCursor c = pc;
            for (int j = 0; j < pre; ++j) {
                c.to(a, item / tiles);
                if (lane == 0) weights(j, item, kb, c);
                if (++kb == ns) {
                    kb = 0;
                    ++item;
                }
            }
            pdl_wait();
        }
        int item = item0, kb = kb_0;
        int myrow = 0, cur_pi = -1;
        bool ok = true;
        int issued = 0;
        for (int j = 0; j < total; ++j) {
            const int slot = j % kTStages;
            if (j >= kTStages) {
                int done = 1;
                if (lane == 0)
                    done = tc05::mbar_wait(&sh.empty[slot], (uint32_t)(((j / kTStages) - 1) & 1),
                                           kTWait);
                if (!__shfl_sync(0xffffffffu, done, 0)) {
                    ok = false;
                    break;
                }
            }
            const int pi = item / tiles;
            if (pi != cur_pi) {
                pc.to(a, pi);
                cur_pi = pi;
                if (lane < pc.ntok) {
                    const int p = a.mode == 2 ? pc.beg + lane : a.list[pc.beg + lane];
                    myrow = a.mode == 0 ? p / a.k : p;
                }
            }
            if (j >= pre && lane == 0) weights(slot, item, kb, pc);
            __syncwarp();
            if (a.packed) {
                // the pass's factors and its token slots' units are one block
                if (lane == 0) {
                    const uint32_t base = tc05::smem_addr(ring + slot * kTStage);
                    const uint32_t fb = tc05::smem_addr(&sh.full[slot]);
                    const uint8_t *blk = reinterpret_cast<const uint8_t *>(a.cells) +
                                         ((size_t)pi * ns + kb) * kPackedStage;
                    bulk_load(base + kTOffF, blk,
                              (uint32_t)(kMaxTok * kTFacTok + pc.ntok * kTActTok), fb);
                }
            } else if (lane < pc.ntok) {
                const uint32_t base = tc05::smem_addr(ring + slot * kTStage);
                const uint32_t fb = tc05::smem_addr(&sh.full[slot]);
                const size_t cg = (size_t)myrow * a.G + 4 * kb;
                bulk_load(base + kTOffA + lane * kTActTok, a.cells + cg * 16, kTActTok, fb);
                bulk_load(base + kTOffF + lane * kTFacTok, a.cfac + 2 * cg, kTFacTok, fb);
            }
            issued = j + 1;
            if (++kb == ns) {
                kb = 0;
                ++item;
            }
        }
        if (lane == 0) {
            if (!ok) atomicOr(a.status, 2);
            // Drain: every copy issued must land before the CTA may exit.
            for (int j = (issued > kTStages ? issued - kTStages : 0); j < issued; ++j)
                tc05::mbar_wait(&sh.full[j % kTStages], (uint32_t)((j / kTStages) & 1), kTWait);
        }
    } else if (warp == kTSync) {
        // ---------------- split-item counters (lane 0) and the last item's fetch
        const TRoles ro = t_roles(u0, u1, (int)blockIdx.x + 1 < g ? ub_at(blockIdx.x + 2) : u1, ns, g);
        if (ro.head_async && lane == 0) {
            int d = 0;
            if (tc05::mbar_wait(&sh.hp, 0u, kTWait))
                d = t_publish(a, sh.h_bf, sh.h_n) ? 1 : 0;
            else
                atomicOr(a.status, 2);
            sh.defer = d;
            mbar_arrive(&sh.hd);
        }
        __syncwarp();
        if (ro.tail_next) {
            // this CTA is the item's first contributor: its counter reaches 1
            // when the next CTA has published
            const int32_t *c = a.cnt + blockIdx.x;
            bool got = false;
            for (uint32_t it = 0; it < kTPoll; ++it) {
                int v;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
                if (__all_sync(0xFFFFFFFFu, v == 1)) {
                    got = true;
                    break;
                }
                if (__any_sync(0xFFFFFFFFu, sh.stop != 0)) break;
                __nanosleep(256);
            }
            if (got) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.part + (size_t)(blockIdx.x + 1) * 2 * (kTRows * kMaxTok));
                float4 *dst = reinterpret_cast<float4 *>(tail);
                for (int i = lane; i < kTRows * kMaxTok / 4; i += 32) dst[i] = __ldcg(src + i);
            }
            __syncwarp();
            if (lane == 0) {
                sh.ready = got ? 1 : 0;
                mbar_arrive(&sh.tp);
            }
        }
    } else {
        // ---------------- consumers
        if (a.skew_ns > 0 && (blockIdx.x & 1)) {
            // test hook (qmv_test_split_skew): odd CTAs start late, so that
            // their neighbours finish first and the split items take the
            // fallback and deferred paths
            const unsigned long long t0 = globaltimer_ns();
            while (globaltimer_ns() - t0 < (unsigned long long)a.skew_ns) __nanosleep(1000);
        }
        for (int i = threadIdx.x; i <= g; i += 32 * kTConsumers) sh.ub[i] = ub_at(i);
        const TRoles ro = t_roles(u0, u1, (int)blockIdx.x + 1 < g ? ub_at(blockIdx.x + 2) : u1, ns, g);
        int j = 0, cur_pi = -1;
        bool failed = false;
        PassCursor pc;
        const int head_item = (int)(u0 / ns);
        int left = (int)(u1 - u0);
        int item = head_item, kb0 = (int)(u0 - (long long)head_item * ns);
        if (left > 0) start_cursor(pc, a, nu, head_item / tiles, pl0);
        for (; left > 0; ++item, kb0 = 0) {
            const int kb1 = min(ns, kb0 + left);
            left -= kb1 - kb0;
            const int pi = item / tiles, tile = item - pi * tiles;
            const bool fresh = pi != cur_pi;
            if (fresh) {
                pc.to(a, pi);
                consumers_sync();  // the previous epilogue is done with sh.pairs
                if (threadIdx.x < pc.ntok)
                    sh.pairs[threadIdx.x] =
                        a.mode == 2 ? pc.beg + threadIdx.x : a.list[pc.beg + threadIdx.x];
                cur_pi = pi;
            }
            const bool whole = kb0 == 0 && kb1 == ns;
            const bool head = item == head_item;
            if (pc.ntok <= 4) {
                float acc[2][1][2];
                t_consume<1>(sh, ring, pc.ntok, kb0, kb1, j, failed, acc);
                if (fresh) consumers_sync();  // sh.pairs written before the epilogue reads it
                t_finish<1>(a, sh, epi, tile, pc.ntok, pi, item, head, ns, whole,
                            ro.head_async && head, ro.tail_next && left == 0, acc);
            } else {
                float acc[2][2][2];
                t_consume<2>(sh, ring, pc.ntok, kb0, kb1, j, failed, acc);
                if (fresh) consumers_sync();
                t_finish<2>(a, sh, epi, tile, pc.ntok, pi, item, head, ns, whole,
                            ro.head_async && head, ro.tail_next && left == 0, acc);
            }
        }
        if (ro.head_async) {
            // the sync warp's count of the first item: if this CTA published
            // it last, it writes the item now
            const bool ok = tc05::mbar_wait(&sh.hd, 0u, kTWait);
            if (!ok) failed = true;
            if (ok && sh.defer) t_write_deferred(a, sh, epi, nu, head_item, tiles, ns);
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
    return encode_weight_maps(&a.wmap, &a.smap, wq, ws, E, rows, K, a.mode == 0 ? 128 : 256);
}

}  // namespace

bool encode_weight_maps(CUtensorMap *wmap, CUtensorMap *smap, const uint8_t *wq, const float *ws,
                        int E, int rows, int K, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    const int G = K / kGroup;
    {
        cuuint64_t dims[3] = {(cuuint64_t)K / 2, (cuuint64_t)rows, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)K / 2, (cuuint64_t)rows * (K / 2)};
        cuuint32_t box[3] = {128, (cuuint32_t)box_rows, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(wq), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        cuuint64_t dims[3] = {(cuuint64_t)G, (cuuint64_t)rows, (cuuint64_t)E};
        cuuint64_t strides[2] = {(cuuint64_t)G * 4, (cuuint64_t)rows * G * 4};
        cuuint32_t box[3] = {4, (cuuint32_t)box_rows, 1};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(smap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ws), dims, strides,
                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

bool encode_rows_swizzled(CUtensorMap *map, const uint8_t *base, long long rows, int row_bytes,
                          int box_rows) {
    auto enc = encode_fn();
    if (!enc || row_bytes % 128 || row_bytes / 128 > 256 || box_rows > 256) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128)};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};
    cuuint32_t box[3] = {128, (cuuint32_t)box_rows, (cuuint32_t)(row_bytes / 128)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(base), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_moe_supported(const MoeDims &m, long long P) {
    // tensor maps need 16-byte aligned bases and 16-byte strides (scale rows of
    // K/64 floats: K/64 a multiple of 4)
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!(encode_fn() != nullptr && (m.H / kGroup) % 4 == 0 && (m.I / kGroup) % 4 == 0 &&
          a16(m.gu_q) && a16(m.gu_s) && a16(m.dn_q) && a16(m.dn_s)))
        return false;
    // the kernel numbers items and stage boundaries with 32-bit ints: passes x
    // stages per pass must fit
    const long long passes = std::min(P, (P + kMaxTok - 1) / kMaxTok + std::min((long long)m.E, P));
    const long long s_gu = (long long)((m.I + kTGuJ - 1) / kTGuJ) * (m.H / 256);
    const long long s_dn = (long long)((m.H + kTDnRows - 1) / kTDnRows) * (m.I / 256);
    return passes * std::max(s_gu, s_dn) < (1LL << 31) - 1;
}

cudaError_t launch_moe_tma(const MoeDims &m, int mode, const void *cells, const float *cfac, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hcells,
                           float *hfac, float *y, int32_t *status, int32_t *cnt, float *part,
                           cudaStream_t st, bool packed, const int4 *ptab, const int4 *plan) {
    TmaArgs a;
    memset(&a, 0, sizeof(a));
    a.mode = mode;
    a.packed = packed ? 1 : 0;
    a.ptab = ptab;
    a.plan = plan;
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
    a.cnt = cnt;
    a.part = part;
    a.skew_ns = g_split_skew_ns;
    a.tiles0 = (m.H + kTDnRows - 1) / kTDnRows;  // down: every row tile is the first matrix's
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
    return launch(k_moe_tma, dim3(tma_grid()), dim3(kTThreads), (size_t)kTSmem, st, true, a);
}

int g_split_skew_ns = 0;

int tma_grid() {
    set_smem(k_moe_tma, kTSmem);
    return std::min(kSkMaxCtas, sm_count() * max_ctas_per_sm(k_moe_tma, kTThreads, kTSmem));
}

bool tma_dense_supported(const uint8_t *wq, const float *scales, int N, int K, int S) {
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    // a partial last row tile reads zeros past row N and writes nothing there;
    // the kernel numbers its items with 32-bit ints
    const long long stages =
        (long long)((S + kMaxTok - 1) / kMaxTok) * ((N + kTDnRows - 1) / kTDnRows) * (K / 256);
    return encode_fn() != nullptr && N % 16 == 0 && (K / kGroup) % 4 == 0 && a16(wq) &&
           a16(scales) && stages < (1LL << 31) - 1;
}

// Dense mode over one matrix, or a pair sharing the activations (wq2 != null):
// the row tiles of both form one item sequence.
cudaError_t launch_dense_tma(const uint8_t *wq, const float *scales, int N, int K, int S,
                             const void *cells, const float *cfac, float *y, int32_t *status,
                             int32_t *cnt, float *part, cudaStream_t st, const uint8_t *wq2,
                             const float *scales2, int N2, float *y2, uint16_t *ybf) {
    TmaArgs a;
    memset(&a, 0, sizeof(a));
    a.mode = 2;
    a.H = N;
    a.S = S;
    a.G = K / kGroup;
    a.tiles0 = (N + kTDnRows - 1) / kTDnRows;
    a.cells = static_cast<const uint4 *>(cells);
    a.cfac = cfac;
    a.y = y;
    a.ybf = ybf;
    a.status = status;
    a.cnt = cnt;
    a.part = part;
    a.skew_ns = g_split_skew_ns;
    if (!make_maps(a, wq, scales, 1, N, K)) return cudaErrorInvalidValue;
    if (wq2) {
        a.H2 = N2;
        a.y2 = y2;
        if (!encode_weight_maps(&a.wmap2, &a.smap2, wq2, scales2, 1, N2, K, 256))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem(k_moe_tma, kTSmem);
    if (e != cudaSuccess) return e;
    const int grid = std::min(kSkMaxCtas, sm_count() * max_ctas_per_sm(k_moe_tma, kTThreads, kTSmem));
    return launch(k_moe_tma, dim3(grid), dim3(kTThreads), (size_t)kTSmem, st, true, a);
}

}  // namespace qmv
