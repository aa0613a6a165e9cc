// qmv_moe_tc.cu - MoE decode gate+up and down on the 5th-generation tensor
// cores, fed by the Tensor Memory Accelerator.
//
// Math (colibri PR #418, "qmatmul_gate_up.comp + coli_vk_gate_up",
// "coli_vk_expert_group", "grouped scales in the Vulkan kernels"): per 64-group
// the exact products (nibble - 8) * x are summed and the group scale is applied
// in fp32 to that partial sum; gate+up gives h = SiLU(gate x) * up x for every
// served (token, expert) pair, down gives y = down h per pair. Activations
// enter as fp16 hi + lo with one power-of-two factor per (row, group), so the
// fp32-accumulated result keeps fp32 accuracy.
//
// One CTA per SM, 18 warps, a 4-slot ring of stages. A stage is 256 weight
// rows x 4 groups of one (pass, row tile) item:
//   * producer warp: two 3-D tensor-map loads of the packed weights (128 rows
//     x 128 bytes each, 128-byte swizzle) and two of their scales, plus the B
//     tile: hi / lo rows of the pass's up to 8 tokens for the 4 groups,
//     gathered with 16-byte loads into the canonical K-major, 128-byte
//     swizzled layout (16 rows: hi of token slots 0-7, then lo), and the
//     8 x 4 activation factors;
//   * 16 dequant warps, one weight row per thread (= tensor-memory lane):
//     each turns its row of two of the stage's groups into exact fp16
//     (nibble - 8) and stores it to tensor memory (tcgen05.st); one stage
//     later it reads that stage's per-group products back (tcgen05.ld) and
//     adds scale * factor * (hi + lo) to fp32 accumulators;
//   * MMA warp: one thread issues per stage 4 groups x 2 row halves x 4 MMAs
//     (M 128, N 16, K 16, A from tensor memory, B from shared memory) into a
//     double-buffered accumulator per group and commits them to an mbarrier.
// Tensor memory: A 256 columns (4 groups x 2 halves x 32), D 2 x 128.
// Within each group the K order is that of the dequantizer (tc_elem): the
// activation rows are stored in the same order, so A and B agree.
//
// Work split: the stages of all items (item-major) are shared out evenly over
// the CTAs. An item whose stages fall to several CTAs is finished by the last
// of them to arrive (an atomic counter; no CTA waits for another), which adds
// the partial sums in CTA order and writes the item.
//
// Every wait is bounded. A wait that runs out raises a CTA-wide abort flag,
// after which no role waits any more; copies and MMAs still in flight are
// waited for (bounded) before the tensor memory is released, and bit 1 of the
// status word is set (the outputs are then not valid).
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

constexpr int kCWarps = 16;                          // dequant / accumulate warps
constexpr int kCThreads = 32 * kCWarps;
constexpr int kProdWarp = kCWarps;
constexpr int kMmaWarp = kCWarps + 1;
constexpr int kCtaThreads = 32 * (kCWarps + 2);
constexpr int kStages = 4;
constexpr int kRows = 256;                           // weight rows per stage
constexpr int kOffS = kRows * 128;                   // scales [256][4] f32
constexpr int kOffB = kOffS + kRows * 16;            // B: 4 groups x 16 rows x 128 B
constexpr int kBGroup = 16 * 128;
constexpr int kOffF = kOffB + 4 * kBGroup;           // factors [4 groups][8 slots] f32
constexpr int kStage = (kOffF + 4 * kMaxTok * 4 + 1023) / 1024 * 1024;
constexpr uint32_t kTmaBytes = kRows * 128 + kRows * 16;
constexpr int kGuJ = 128;                            // hidden units per gate+up item
constexpr int kDnRows = 256;                         // output rows per down item
constexpr int kEpiFloats = kRows * kMaxTok + kMaxTok * kGuJ;
constexpr int kSmem = kStages * kStage + kEpiFloats * 4 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemD = 256;                     // first D column
constexpr uint32_t kWaitIters = 1u << 24;
constexpr uint32_t kIdesc = tc05::idesc_f16_f32(128, 16);

static_assert(kMaxTok == 8, "a B tile holds 8 token slots (hi and lo: N = 16)");
static_assert(kStage % 1024 == 0, "stages must stay 1024-aligned for the 128B swizzle");
static_assert(kSkPartFloats == 2 * kRows * kMaxTok, "partial-sum slots must match the stage");

struct TcArgs {
    CUtensorMap wmap;    // weights: uint8 [E][rows][K/2], box 128 B x 128 rows, 128B swizzle
    CUtensorMap smap;    // scales: f32 [E][rows][K/64], box 4 x 128 rows
    int mode;            // 0: gate+up, 1: down
    int G, I, H, k;
    const int32_t *offsets, *list, *uexp, *n_used, *pass_ofs;
    const uint4 *act;    // activation rows [row][G][2][64] fp16 (tc_elem order), as 16-byte chunks
    const float *afac;   // their factors [row][G]
    float *h;            // gate+up: h fp32 [P][I]
    uint32_t *hrows;     // gate+up: h as activation rows [P][I/64][2][32 words]
    float *hfac;         // gate+up: their factors [P][I/64]
    float *y;            // down: y [P][H]
    int32_t *status;
    int32_t *cnt;        // per CTA: contributors done on the split item that starts in it
    float *part;         // per CTA: partial sums [2][kRows][kMaxTok] (head / tail item)
};

struct TcShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t afull;
    uint64_t dfull[2];
    uint64_t dfree[2];
    long long ub[kSkMaxCtas + 1];  // first stage of each CTA's range
    uint32_t tmem;
    int abort;
    int pairs[kMaxTok];
    int last;
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

__device__ __forceinline__ bool mbar_try(uint64_t *mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(tc05::smem_addr(mbar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait that gives up at once when another role has aborted; running
// out of polls raises the abort flag.
__device__ __forceinline__ bool wait_ab(TcShared &sh, uint64_t *mbar, uint32_t parity) {
    volatile int *ab = &sh.abort;
    for (uint32_t i = 0; i < kWaitIters; ++i) {
        if (mbar_try(mbar, parity)) return true;
        if ((i & 15u) == 15u && *ab) return false;
    }
    *ab = 1;
    return false;
}

// Bounded wait that ignores the abort flag (draining work in flight).
__device__ __forceinline__ void wait_drain(uint64_t *mbar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitIters; ++i)
        if (mbar_try(mbar, parity)) return;
}

__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCThreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
    return *reinterpret_cast<const uint4 *>(p);
}

// Walks the passes of the grouped pairs in order. `lo` indexes the used
// experts (uexp); passes of used expert lo are pass_ofs[lo] .. pass_ofs[lo+1]-1.
struct PassCursor {
    int lo, pi, e, beg, ntok;

    __device__ __forceinline__ void seek(const TcArgs &a, int nu, int p) {
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
    __device__ __forceinline__ void to(const TcArgs &a, int p) {
        if (p == pi) return;
        while (a.pass_ofs[lo + 1] <= p) ++lo;
        pi = p;
        e = a.uexp[lo];
        const int pass = p - a.pass_ofs[lo];
        const int b = a.offsets[e], cnt = a.offsets[e + 1] - b;
        beg = b + pass * kMaxTok;
        ntok = min(kMaxTok, cnt - pass * kMaxTok);
    }
};

// The CTA whose range holds stage u (ub: first stage of each CTA, g + 1 entries).
__device__ __forceinline__ int unit_owner(const long long *ub, int g, long long u) {
    int l = 0, hgh = g - 1;
    while (l < hgh) {
        const int mid = (l + hgh + 1) >> 1;
        if (ub[mid] <= u) l = mid; else hgh = mid - 1;
    }
    return l;
}

// 32 packed bytes (one row, one group) -> 32 half2 columns of exact
// (nibble - 8): column 4i + m holds elements (8i + m, 8i + m + 4).
__device__ __forceinline__ void dequant_row_group(const uint4 &w0, const uint4 &w1,
                                                  uint32_t (&r)[32]) {
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t p[4];
        dequant_int4_word(w[i], p);
        r[4 * i + 0] = p[0];
        r[4 * i + 1] = p[1];
        r[4 * i + 2] = p[2];
        r[4 * i + 3] = p[3];
    }
}

// One stage's products of this thread's row, groups g0 and g0 + 1, into acc:
// acc[s] += scale_g * factor_g[s] * (hi + lo), D columns s (hi) and 8 + s (lo).
__device__ __forceinline__ void accumulate_stage(uint32_t d_addr0, uint32_t d_addr1,
                                                 const float *fs, float sc0, float sc1,
                                                 float (&acc)[kMaxTok]) {
    uint32_t d0[16], d1[16];
    tc05::tmem_ld16(d_addr0, d0);
    tc05::tmem_ld16(d_addr1, d1);
    tc05::tmem_wait_ld();
    const float4 fa = reinterpret_cast<const float4 *>(fs)[0];
    const float4 fb = reinterpret_cast<const float4 *>(fs)[1];
    const float4 fc = reinterpret_cast<const float4 *>(fs)[2];
    const float4 fd = reinterpret_cast<const float4 *>(fs)[3];
    const float f0[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
    const float f1[8] = {fc.x, fc.y, fc.z, fc.w, fd.x, fd.y, fd.z, fd.w};
#pragma unroll
    for (int s = 0; s < kMaxTok; ++s) {
        acc[s] = fmaf(sc0 * f0[s], __uint_as_float(d0[s]) + __uint_as_float(d0[8 + s]), acc[s]);
        acc[s] = fmaf(sc1 * f1[s], __uint_as_float(d1[s]) + __uint_as_float(d1[8 + s]), acc[s]);
    }
}

// An item whose stages are split between CTAs: this CTA stores its partial
// sums (slot 0 if the item is the first of its range, else slot 1), and the
// last contributor to arrive adds every contributor's partial in CTA order
// (so the sum does not depend on which CTA finishes last), clears the counter
// for the next launch and returns true: it then writes the item. Threads of
// rows r (own == true) hold the sums; every compute thread takes part.
__device__ __forceinline__ bool tc_combine(const TcArgs &a, TcShared &sh, int ntok, int item,
                                           bool head, int ns, bool own, int r,
                                           float (&acc)[kMaxTok]) {
    const int g = gridDim.x;
    if (own) {
        float *mine = a.part + ((size_t)blockIdx.x * 2 + (head ? 0 : 1)) * (kRows * kMaxTok);
#pragma unroll
        for (int s = 0; s < kMaxTok; ++s)
            if (s < ntok) mine[r * kMaxTok + s] = acc[s];
    }
    __threadfence();
    compute_sync();
    const long long first = (long long)item * ns;
    const int bf = unit_owner(sh.ub, g, first), bl = unit_owner(sh.ub, g, first + ns - 1);
    if (threadIdx.x == 0) {
        int n = 0;  // CTAs of [bf, bl] with a non-empty range all hold stages of this item
        for (int c = bf; c <= bl; ++c) n += sh.ub[c + 1] > sh.ub[c];
        sh.last = atomicAdd(&a.cnt[bf], 1) == n - 1;
    }
    compute_sync();
    if (!sh.last) return false;
    __threadfence();
    if (own) {
#pragma unroll
        for (int s = 0; s < kMaxTok; ++s) acc[s] = 0.f;
        for (int c = bf; c <= bl; ++c) {
            const long long c0 = sh.ub[c];
            if (sh.ub[c + 1] <= c0) continue;
            const float *pc =
                a.part + ((size_t)c * 2 + (c0 >= first ? 0 : 1)) * (kRows * kMaxTok) + r * kMaxTok;
#pragma unroll
            for (int s = 0; s < kMaxTok; ++s)
                if (s < ntok) acc[s] += __ldcg(pc + s);
        }
    }
    if (threadIdx.x == 0) a.cnt[bf] = 0;
    return true;
}

// Writes a finished item. Threads of set 0 (warps 0-7) hold row r's sums.
__device__ __forceinline__ void tc_epilogue(const TcArgs &a, const TcShared &sh, float *epi,
                                            int tile, int ntok, bool own, int r,
                                            const float (&acc)[kMaxTok]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.mode == 1) {
        if (own) {
            const int row = tile * kDnRows + r;
#pragma unroll
            for (int s = 0; s < kMaxTok; ++s)
                if (s < ntok) a.y[(size_t)sh.pairs[s] * a.H + row] = acc[s];
        }
        return;
    }
    // gate+up: rows 0-127 are gate rows, 128-255 the up rows of the same units
    float *ubuf = epi;                    // [128 units][8]
    float *hbuf = epi + kRows * kMaxTok;  // [8 slots][128 units]
    const int I = a.I, j0 = tile * kGuJ;
    if (own && r >= kGuJ) {
#pragma unroll
        for (int s = 0; s < kMaxTok; ++s) ubuf[(r - kGuJ) * kMaxTok + s] = acc[s];
    }
    compute_sync();
    if (own && r < kGuJ) {
#pragma unroll
        for (int s = 0; s < kMaxTok; ++s) {
            if (s < ntok) {
                const float gv = acc[s], uv = ubuf[r * kMaxTok + s];
                const float hv = gv / (1.0f + expf(-gv)) * uv;
                a.h[(size_t)sh.pairs[s] * I + j0 + r] = hv;
                hbuf[s * kGuJ + r] = hv;
            }
        }
    }
    compute_sync();
    // h of this item as activation rows of the down pass: 2 groups per slot
    const int Gd = I / kGroup;
    const int e0 = tc_elem(2 * lane);
    for (int idx = warp; idx < ntok * 2; idx += kCWarps) {
        const int s = idx >> 1, gg = idx & 1;
        const int gd = tile * 2 + gg;
        const float *v = hbuf + s * kGuJ + gg * kGroup;
        const size_t cb = (size_t)sh.pairs[s] * Gd + gd;
        uint32_t *dst = a.hrows + cb * 64;
        split_group_rows(v[e0], v[e0 + 4], dst, dst + 32, a.hfac + cb, lane);
    }
    compute_sync();
}

__global__ void __launch_bounds__(kCtaThreads, 1) k_moe_tc(const __grid_constant__ TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ TcShared sh;
    // 1024-byte alignment by an offset on the shared array itself, so the
    // compiler keeps shared-window addressing (LDS) for every access.
    uint8_t *ring = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    float *epi = reinterpret_cast<float *>(ring + kStages * kStage);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) tc05::tmem_alloc(&sh.tmem, kTmemCols);
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            tc05::mbar_init(&sh.full[s], 2);
            tc05::mbar_init(&sh.empty[s], kCWarps);
        }
        tc05::mbar_init(&sh.afull, kCWarps);
        for (int b = 0; b < 2; ++b) {
            tc05::mbar_init(&sh.dfull[b], 1);
            tc05::mbar_init(&sh.dfree[b], kCWarps);
        }
        sh.abort = 0;
        tc05::fence_mbar_init();
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = sh.tmem;

    // gate+up needs the grouping (previous kernel) before anything. The down
    // kernel's grouping finished before the previous kernel started, so its
    // producer requests the first weight stages before waiting (below).
    if (a.mode == 0 || warp != kProdWarp) pdl_wait();
    pdl_trigger();

    const int nu = *a.n_used;
    const int tiles = a.mode == 0 ? a.I / kGuJ : a.H / kDnRows;
    const int total_items = nu > 0 ? a.pass_ofs[nu] * tiles : 0;
    const int ns = a.G / 4;
    const long long U = (long long)total_items * ns;
    const int g = gridDim.x;
    const long long u0 = (long long)blockIdx.x * U / g;
    const long long u1 = (long long)(blockIdx.x + 1) * U / g;
    const int total = (int)(u1 - u0);
    const int item0 = (int)(u0 / ns), kb_0 = (int)(u0 - (long long)item0 * ns);

    if (warp == kProdWarp) {
        // ---------------- producer (whole warp; lane 0 owns the barriers)
        const int pre = a.mode == 1 ? min(total, kStages) : 0;
        PassCursor pc;
        if (total > 0) pc.seek(a, nu, item0 / tiles);
        auto weights = [&](int slot, int item, int kb, int e) {
            const int tile = item % tiles;
            const int rowA = a.mode == 0 ? tile * kGuJ : tile * kDnRows;
            const int rowB = a.mode == 0 ? a.I + tile * kGuJ : tile * kDnRows + 128;
            const uint32_t base = tc05::smem_addr(ring + slot * kStage);
            const uint32_t fb = tc05::smem_addr(&sh.full[slot]);
            mbar_expect_tx(&sh.full[slot], kTmaBytes);
            tma_load3(base, &a.wmap, kb * 128, rowA, e, fb);
            tma_load3(base + 128 * 128, &a.wmap, kb * 128, rowB, e, fb);
            tma_load3(base + kOffS, &a.smap, kb * 4, rowA, e, fb);
            tma_load3(base + kOffS + 128 * 16, &a.smap, kb * 4, rowB, e, fb);
        };
        if (pre > 0) {
            int item = item0, kb = kb_0;
            PassCursor c = pc;
            for (int j = 0; j < pre; ++j) {
                c.to(a, item / tiles);
                if (lane == 0) weights(j, item, kb, c.e);
                if (++kb == ns) {
                    kb = 0;
                    ++item;
                }
            }
            pdl_wait();  // h, its rows and factors come from the previous kernel
        }
        int item = item0, kb = kb_0;
        int myrow = 0, cur_pi = -1;
        int issued = 0;
        const int G = a.G;
        for (int j = 0; j < total; ++j) {
            const int slot = j % kStages;
            const int pi = item / tiles;
            if (pi != cur_pi) {
                pc.to(a, pi);
                cur_pi = pi;
                if (lane < pc.ntok) {
                    const int p = a.list[pc.beg + lane];
                    myrow = a.mode == 0 ? p / a.k : p;
                }
            }
            // B chunks of this stage: chunk c = lane + 32 i -> group i / 4,
            // tile row n = 4 (i % 4) + lane / 8 (slot n % 8, hi / lo n / 8),
            // 16-byte column lane % 8.
            uint4 bv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int n = 4 * (i & 3) + (lane >> 3);
                const int rs = __shfl_sync(0xffffffffu, myrow, min(n & 7, pc.ntok - 1));
                const size_t src = (((size_t)rs * G + 4 * kb + (i >> 2)) * 2 + (n >> 3)) * 8 + (lane & 7);
                bv[i] = __ldg(a.act + src);
            }
            const int rf = __shfl_sync(0xffffffffu, myrow, min(lane & 7, pc.ntok - 1));
            const float fv = __ldg(a.afac + (size_t)rf * G + 4 * kb + (lane >> 3));
            if (j >= kStages) {
                int done = 1;
                if (lane == 0)
                    done = wait_ab(sh, &sh.empty[slot], (uint32_t)(((j / kStages) - 1) & 1));
                if (!__shfl_sync(0xffffffffu, done, 0)) break;
            }
            if (j >= pre && lane == 0) weights(slot, item, kb, pc.e);
            uint8_t *sp = ring + slot * kStage;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int n = 4 * (i & 3) + (lane >> 3);
                *reinterpret_cast<uint4 *>(sp + kOffB + (i >> 2) * kBGroup + n * 128 +
                                           (((lane & 7) ^ (n & 7)) << 4)) = bv[i];
            }
            reinterpret_cast<float *>(sp + kOffF)[lane] = fv;
            tc05::fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.full[slot]);
            issued = j + 1;
            if (++kb == ns) {
                kb = 0;
                ++item;
            }
        }
        if (lane == 0) {
            // Drain: every copy issued must land before the CTA may exit.
            for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
                wait_drain(&sh.full[j % kStages], (uint32_t)((j / kStages) & 1));
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread)
        if (lane == 0) {
            int last = -1;
            for (int j = 0; j < total; ++j) {
                const int slot = j % kStages, b = j & 1;
                if (!wait_ab(sh, &sh.full[slot], (uint32_t)((j / kStages) & 1))) break;
                if (!wait_ab(sh, &sh.afull, (uint32_t)(j & 1))) break;
                if (j >= 2 && !wait_ab(sh, &sh.dfree[b], (uint32_t)(((j - 2) >> 1) & 1))) break;
                tc05::fence_after_sync();
                const uint32_t sB = tc05::smem_addr(ring + slot * kStage + kOffB);
                // K step outermost: the 8 accumulators are independent, so
                // consecutive MMAs never wait on each other's result.
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                    for (int gl = 0; gl < 4; ++gl) {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            tc05::mma_ts(tmem + kTmemD + b * 128 + gl * 32 + hf * 16,
                                         tmem + gl * 64 + hf * 32 + kk * 8,
                                         tc05::sdesc_sw128(sB + gl * kBGroup + kk * 32), kIdesc,
                                         kk > 0 ? 1u : 0u);
                        }
                    }
                }
                tc05::mma_commit(&sh.dfull[b]);
                last = j;
            }
            // MMAs still in flight must finish before the tensor memory is freed.
            if (last >= 0) wait_drain(&sh.dfull[last & 1], (uint32_t)((last >> 1) & 1));
        }
    } else {
        // ---------------- dequant / accumulate warps
        const int set = warp >> 3, half = (warp >> 2) & 1, quarter = warp & 3;
        const int r = half * 128 + quarter * 32 + lane;  // stage row = TMEM lane of its half
        const int g0 = 2 * set;                           // this thread's groups g0, g0 + 1
        const bool own = set == 0;
        const uint32_t lrow = (uint32_t)(quarter * 32) << 16;
        const uint32_t a_addr0 = tmem + lrow + g0 * 64 + half * 32;
        const uint32_t a_addr1 = a_addr0 + 64;
        for (int i = threadIdx.x; i <= g; i += kCThreads) sh.ub[i] = (long long)i * U / g;
        int j = 0, cur_pi = -1;
        PassCursor pc;
        if (total > 0) pc.seek(a, nu, item0 / tiles);
        int left = total;
        int item = item0, kb0 = kb_0;
        for (; left > 0; ++item, kb0 = 0) {
            const int kb1 = min(ns, kb0 + left);
            left -= kb1 - kb0;
            const int pi = item / tiles, tile = item - pi * tiles;
            if (pi != cur_pi) {
                pc.to(a, pi);
                compute_sync();  // the previous epilogue is done with sh.pairs
                if (threadIdx.x < pc.ntok) sh.pairs[threadIdx.x] = a.list[pc.beg + threadIdx.x];
                cur_pi = pi;
            }
            float acc[kMaxTok];
#pragma unroll
            for (int s = 0; s < kMaxTok; ++s) acc[s] = 0.f;
            int jp = -1;
            float sp0 = 0.f, sp1 = 0.f;
            for (int kb = kb0; kb < kb1; ++kb, ++j) {
                const int slot = j % kStages;
                wait_ab(sh, &sh.full[slot], (uint32_t)((j / kStages) & 1));
                const uint8_t *sp = ring + slot * kStage;
                const uint8_t *wr = sp + r * 128;
                const int x7 = r & 7;
                const uint4 wa0 = lds128(wr + (((2 * g0) ^ x7) << 4));
                const uint4 wa1 = lds128(wr + (((2 * g0 + 1) ^ x7) << 4));
                const uint4 wb0 = lds128(wr + (((2 * g0 + 2) ^ x7) << 4));
                const uint4 wb1 = lds128(wr + (((2 * g0 + 3) ^ x7) << 4));
                const float2 sc = *reinterpret_cast<const float2 *>(sp + kOffS + r * 16 + g0 * 4);
                uint32_t A[32];
                dequant_row_group(wa0, wa1, A);
                if (jp >= 0) {
                    // MMA(jp) done: A may be overwritten, D(jp) may be read
                    wait_ab(sh, &sh.dfull[jp & 1], (uint32_t)((jp >> 1) & 1));
                    tc05::fence_after_sync();
                }
                tc05::tmem_st32(a_addr0, A);
                dequant_row_group(wb0, wb1, A);
                tc05::tmem_st32(a_addr1, A);
                tc05::tmem_wait_st();
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.afull);
                if (jp >= 0) {
                    const int pslot = jp % kStages;
                    const uint32_t d0 = tmem + lrow + kTmemD + (jp & 1) * 128 + g0 * 32 + half * 16;
                    accumulate_stage(d0, d0 + 32,
                                     reinterpret_cast<const float *>(ring + pslot * kStage + kOffF) + g0 * 8,
                                     sp0, sp1, acc);
                    tc05::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.dfree[jp & 1]);
                        mbar_arrive(&sh.empty[pslot]);
                    }
                }
                jp = j;
                sp0 = sc.x;
                sp1 = sc.y;
            }
            // the item's last stage
            if (jp >= 0) {
                wait_ab(sh, &sh.dfull[jp & 1], (uint32_t)((jp >> 1) & 1));
                tc05::fence_after_sync();
                const int pslot = jp % kStages;
                const uint32_t d0 = tmem + lrow + kTmemD + (jp & 1) * 128 + g0 * 32 + half * 16;
                accumulate_stage(d0, d0 + 32,
                                 reinterpret_cast<const float *>(ring + pslot * kStage + kOffF) + g0 * 8,
                                 sp0, sp1, acc);
                tc05::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sh.dfree[jp & 1]);
                    mbar_arrive(&sh.empty[pslot]);
                }
            }
            // groups 2-3 (set 1) into the set-0 thread of the same row
            if (!own) {
#pragma unroll
                for (int s = 0; s < kMaxTok; ++s) epi[r * kMaxTok + s] = acc[s];
            }
            compute_sync();
            if (own) {
#pragma unroll
                for (int s = 0; s < kMaxTok; ++s) acc[s] += epi[r * kMaxTok + s];
            }
            compute_sync();
            const bool whole = kb0 == 0 && kb1 == ns;
            if (whole || tc_combine(a, sh, pc.ntok, item, item == item0, ns, own, r, acc))
                tc_epilogue(a, sh, epi, tile, pc.ntok, own, r, acc);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && sh.abort) atomicOr(a.status, 2);
    tc05::fence_after_sync();
    if (warp == 0) tc05::tmem_dealloc(tmem, kTmemCols);
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

bool make_maps(TcArgs &a, const uint8_t *wq, const float *ws, int E, int rows, int K) {
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

bool tc_moe_supported(const MoeDims &m) {
    // stages of 4 groups, gate+up items of 128 units, down items of 256 rows;
    // tensor maps need 16-byte aligned bases and 16-byte strides
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    return encode_fn() != nullptr && (m.H / kGroup) % 4 == 0 && (m.I / kGroup) % 4 == 0 &&
           a16(m.gu_q) && a16(m.gu_s) && a16(m.dn_q) && a16(m.dn_s);
}

cudaError_t launch_moe_tc(const MoeDims &m, int mode, const void *act, const float *afac, int k,
                          const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                          const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hrows,
                          float *hfac, float *y, int32_t *status, int32_t *cnt, float *part,
                          cudaStream_t st) {
    TcArgs a;
    memset(&a, 0, sizeof(a));
    a.mode = mode;
    a.I = m.I;
    a.H = m.H;
    a.k = k;
    a.offsets = offsets; a.list = list; a.uexp = uexp; a.n_used = n_used; a.pass_ofs = pass_ofs;
    a.act = static_cast<const uint4 *>(act);
    a.afac = afac;
    a.h = h;
    a.hrows = static_cast<uint32_t *>(hrows);
    a.hfac = hfac;
    a.y = y;
    a.status = status;
    a.cnt = cnt;
    a.part = part;
    bool ok;
    if (mode == 0) {
        a.G = m.H / kGroup;
        ok = make_maps(a, m.gu_q, m.gu_s, m.E, 2 * m.I, m.H);
    } else {
        a.G = m.I / kGroup;
        ok = make_maps(a, m.dn_q, m.dn_s, m.E, m.H, m.I);
    }
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = set_smem(k_moe_tc, kSmem);
    if (e != cudaSuccess) return e;
    const int grid = std::min(kSkMaxCtas, sm_count() * max_ctas_per_sm(k_moe_tc, kCtaThreads, kSmem));
    return launch(k_moe_tc, dim3(grid), dim3(kCtaThreads), (size_t)kSmem, st, true, a);
}

}  // namespace qmv
