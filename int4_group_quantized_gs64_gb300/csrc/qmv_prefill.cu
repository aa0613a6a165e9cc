// qmv_prefill.cu - batched MoE prefill on the 5th-generation tensor cores.
//
// With hundreds of tokens, each expert sees tens of tokens, so its gate+up and
// down products are real (skinny) matrix products: the int4-gs64 weights are
// streamed once per batch, dequantized to bf16 (group scale folded in) and
// multiplied on tcgen05 with fp32 accumulation in tensor memory.
//
// Sources: colibri PR #418 "Vulkan backend: expert tier + dense + MLA
// attention on any Vulkan 1.2 GPU" (int4 nibble - 8 with one scale per
// 64-group; fused gate+up with silu(gate) * up; gate+up then down per expert)
// and its PR summary (cooperative-matrix prefill kernels named as the next
// step for batched prompts); colibri PR #1338 (weighted accumulation of the
// expert outputs).
//
// Kernel shape (both projections): a CTA of 256 threads owns a 256-row tile
// (gate_up: 128 gate rows + the matching 128 up rows; down: 256 output rows)
// for one "pass" of up to 64 tokens of one expert, and walks a contiguous range
// of such items. Per 64-wide K group:
//   * every thread cp.async-copies its own row's 32 packed bytes and scale,
//     and a share of the B tile (the pass's token rows, bf16, 128-byte
//     swizzled K-major layout), kPrefetch groups ahead;
//   * every thread dequantizes its row to 64 bf16 values (nibble - 8) * scale
//     and stores them to tensor memory with tcgen05.st: thread = TMEM lane =
//     MMA row, so A never passes through shared memory;
//   * one thread issues 2 x 4 MMAs (M 128, N = tokens rounded up to 16,
//     K 16 each; A from TMEM, B from shared memory) and commits them to an
//     mbarrier that frees the A slot and the data slot two groups later.
// After the last group of an item the accumulators are read back with
// tcgen05.ld: gate_up writes h = SiLU(g) * u as bf16, down writes y as fp32.
// Every mbarrier wait is bounded; on timeout the kernel flags the status word
// and leaves its loop.
#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_rows.cuh"
#include "tc05.cuh"

#include <cuda_bf16.h>

#include <cstring>

namespace qmv {

namespace {

constexpr int kPfThreads = 256;
constexpr int kPfMaxN = 64;                         // tokens per pass
constexpr int kPfPrefetch = 6;                      // K groups in flight
constexpr int kPfSlots = kPfPrefetch + 2;
constexpr int kPfWBytes = 2 * 256 * 16;             // packed weights of 256 rows, one group
constexpr int kPfSBytes = 256 * 4;                  // their scales
constexpr int kPfBBytes = kPfMaxN * 128;            // B tile: 64 tokens x 64 bf16
constexpr int kPfSlotBytes = kPfWBytes + kPfSBytes + kPfBBytes;  // 17 KB, 1024-multiple
constexpr int kPfSmem = kPfSlots * kPfSlotBytes + 1024;           // + alignment slack
constexpr uint32_t kTmemCols = 256;                 // A: 2 slots x 2 tiles x 32; D: 2 x 64
constexpr uint32_t kWaitIters = 1u << 22;

static_assert(kPfSlotBytes % 1024 == 0, "slots must keep the B tiles 1024-aligned");

struct PfArgs {
    const uint8_t *wq;   // weight pool [E][rows][K/2]
    const float *ws;     // scale pool [E][rows][K/64]
    size_t eq, es;       // per-expert strides (bytes, floats)
    int rows;            // rows per expert matrix (2I or H)
    int K;               // reduction length (H or I)
    int tiles;           // 256-row tiles per pass
    const uint16_t *b;   // B rows, bf16: x [T][H] or h [P][I]
    int by_pair;         // 1: B row = pair id; 0: B row = pair / k
    int k;
    const int32_t *offsets, *list, *uexp, *n_used, *pass_ofs;
    uint16_t *h;         // gate_up output [P][I] bf16
    float *y;            // down output [P][H] fp32
    int I, H;
    int mode;            // 0: gate_up, 1: down
    int32_t *status;
};

struct PfItem {
    int e, beg, ntok, npad, tile;
};

__device__ __forceinline__ PfItem pf_item(const PfArgs &a, int nu, int item) {
    const int pi = item / a.tiles;
    const int tl = item - pi * a.tiles;
    int lo = 0, hi = nu - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.pass_ofs[mid] <= pi) lo = mid; else hi = mid - 1;
    }
    PfItem r;
    r.e = a.uexp[lo];
    const int pass = pi - a.pass_ofs[lo];
    const int b = a.offsets[r.e], cnt = a.offsets[r.e + 1] - b;
    r.beg = b + pass * kPfMaxN;
    r.ntok = min(kPfMaxN, cnt - pass * kPfMaxN);
    r.npad = (r.ntok + 15) & ~15;
    r.tile = tl;
    return r;
}

// Matrix row of thread t in tile `tl`.
__device__ __forceinline__ int pf_row(const PfArgs &a, int tl, int t) {
    const int tt = t >> 7, r = t & 127;
    int row;
    if (a.mode == 0) row = (tt == 0 ? 0 : a.I) + tl * 128 + r;
    else row = tl * 256 + tt * 128 + r;
    return row < a.rows ? row : a.rows - 1;
}

__device__ __forceinline__ int pf_brow(const PfArgs &a, int pair) {
    return a.by_pair ? pair : pair / a.k;
}

// Per-thread copy sources of the current item: its weight row, its scale row
// and up to two B-tile chunks (token row, 16-byte chunk), advanced per group.
struct PfCursor {
    const uint8_t *wrow;
    const float *srow;
    const uint16_t *bsrc[2];
    uint32_t bdst[2];
    int nb;  // B chunks this thread copies (0..2)

    __device__ __forceinline__ void set(const PfArgs &a, const PfItem &it, int t) {
        const int row = pf_row(a, it.tile, t);
        wrow = a.wq + it.e * a.eq + (size_t)row * (a.K / 2);
        srow = a.ws + it.e * a.es + (size_t)row * (a.K / 64);
        nb = 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = t + i * kPfThreads;
            const int n = c >> 3, ch = c & 7;
            const int nn = min(n, it.ntok - 1);
            const bool on = c < it.npad * 8;
            const int brow = on ? pf_brow(a, a.list[it.beg + nn]) : 0;
            bsrc[i] = a.b + (size_t)brow * a.K + ch * 8;
            bdst[i] = kPfWBytes + kPfSBytes + (n >> 3) * 1024 + (n & 7) * 128 + ((ch ^ (n & 7)) << 4);
            nb += on ? 1 : 0;
        }
    }
    // One K group of loads into the slot at shared address sW.
    __device__ __forceinline__ void issue(uint32_t sW, int kg, int t) const {
        const uint8_t *w = wrow + kg * 32;
        cp_async16_s(sW + t * 16, w);
        cp_async16_s(sW + 4096 + t * 16, w + 16);
        cp_async4_s(sW + kPfWBytes + t * 4, srow + kg);
        if (nb > 0) cp_async16_s(sW + bdst[0], bsrc[0] + kg * 64);
        if (nb > 1) cp_async16_s(sW + bdst[1], bsrc[1] + kg * 64);
    }
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
    return d;
}
__device__ __forceinline__ uint32_t lop3_andor_(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 32 packed bytes of one row (K values 0..63 of a group) -> 32 bf16x2 with
// (nibble - 8) * scale in natural K order: column c holds values (2c, 2c+1),
// the low and high nibble of byte c. A byte permute takes byte c of the word
// into the low half and byte c of (word >> 4) into the high half, so each
// half has its nibble in mantissa bits 0..3; OR-ing the bf16 bias 128 (unit
// spacing) gives 128 + n exactly, subtracting 136 gives n - 8 exactly, and
// one multiply applies the group scale (one bf16 rounding).
__device__ __forceinline__ void pf_dequant(const uint4 &w0, const uint4 &w1, float scale,
                                           uint32_t (&r)[32]) {
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t kBias = 0x43004300u;   // (128, 128) in bf16
    const uint32_t kSub = 0xC308C308u;    // (-136, -136)
    const __nv_bfloat162 s2 = __float2bfloat162_rn(scale);
    const uint32_t s = *reinterpret_cast<const uint32_t *>(&s2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t hs = words[i] >> 4;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            // result bytes: [w.b, w.b, hs.b, hs.b]
            const uint32_t sel = (uint32_t)b | ((uint32_t)b << 4) | ((uint32_t)(4 + b) << 8) |
                                 ((uint32_t)(4 + b) << 12);
            const uint32_t v = lop3_andor_(prmt(words[i], hs, sel), 0x000F000Fu, kBias);
            r[4 * i + b] = bmul2(badd2(v, kSub), s);
        }
    }
}

// The same values in the MMA K order of the tensor-map kernel's B tiles:
// column 4i + m holds the elements (8i + m, 8i + m + 4) of the group, which
// are nibbles m and m + 4 of word i. Masking the word, or the word shifted
// by 4, 8 or 12 bits, with 0x000F000F puts such a pair in the two halves'
// mantissa bits 0..3 directly, with no byte permute (15 instructions a word
// instead of 17). The B operands are stored in the same K order (kperm).
__device__ __forceinline__ void pf_dequant_perm(const uint4 &w0, const uint4 &w1, float scale,
                                                uint32_t (&r)[32]) {
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t kBias = 0x43004300u;   // (128, 128) in bf16
    const uint32_t kSub = 0xC308C308u;    // (-136, -136)
    const __nv_bfloat162 s2 = __float2bfloat162_rn(scale);
    const uint32_t s = *reinterpret_cast<const uint32_t *>(&s2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = words[i], w4 = w >> 4, w8 = w >> 8, w12 = w4 >> 8;
        r[4 * i + 0] = bmul2(badd2(lop3_andor_(w, 0x000F000Fu, kBias), kSub), s);
        r[4 * i + 1] = bmul2(badd2(lop3_andor_(w4, 0x000F000Fu, kBias), kSub), s);
        r[4 * i + 2] = bmul2(badd2(lop3_andor_(w8, 0x000F000Fu, kBias), kSub), s);
        r[4 * i + 3] = bmul2(badd2(lop3_andor_(w12, 0x000F000Fu, kBias), kSub), s);
    }
}

// Position of group element kq (0..63) in the MMA K order of pf_dequant_perm.
__host__ __device__ __forceinline__ int kperm_pos(int kq) {
    return 8 * (kq >> 3) + 2 * (kq & 3) + ((kq >> 2) & 1);
}

__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_splat(float v) {
    const __nv_bfloat162 b = __float2bfloat162_rn(v);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// The same values and K order as pf_dequant_perm in 11 instructions a word
// instead of 15. Each nibble is moved to bits 4..7 of its 16-bit half with
// nothing else set: as a bf16 bit pattern below 0x100 (exponent field 0 or 1,
// where consecutive patterns are 2^-133 apart) that reads exactly n * 2^-129.
// One fused multiply-add per pair, n * 2^-129 * (s * 2^129) - 8 s, is then
// (n - 8) * s with a single bf16 rounding: the product is exact and -8 s is
// exact in bf16, so the result is bit for bit the two-step form's. Valid
// while s * 2^129 and 8 s stay normal bf16 numbers: 2^-120 <= |s| < 2^-2
// (or s = 0); pf_dequant_fast checks that per warp.
__device__ __forceinline__ void pf_dequant_sub(const uint4 &w0, const uint4 &w1, float scale,
                                               uint32_t (&r)[32]) {
    const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t s = bf16x2_splat(scale * 0x1p64f * 0x1p65f);  // two exact steps
    const uint32_t c = bf16x2_splat(-8.0f * scale);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t w = words[i];
        r[4 * i + 0] = bfma2((w << 4) & 0x00F000F0u, s, c);  // nibbles 0 and 4
        r[4 * i + 1] = bfma2(w & 0x00F000F0u, s, c);         // 1 and 5
        r[4 * i + 2] = bfma2((w >> 4) & 0x00F000F0u, s, c);  // 2 and 6
        r[4 * i + 3] = bfma2((w >> 8) & 0x00F000F0u, s, c);  // 3 and 7
    }
}

// pf_dequant_sub when every lane's scale is in its range, else
// pf_dequant_perm (same bits either way). Whole warp.
__device__ __forceinline__ void pf_dequant_fast(const uint4 &w0, const uint4 &w1, float scale,
                                                uint32_t (&r)[32]) {
    const float m = fabsf(scale);
    if (__all_sync(0xffffffffu, (m < 0.25f && m >= 0x1p-120f) || scale == 0.0f))
        pf_dequant_sub(w0, w1, scale, r);
    else
        pf_dequant_perm(w0, w1, scale, r);
}

__global__ void __launch_bounds__(kPfThreads, 1) k_prefill(PfArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t mbar[2];
    __shared__ uint32_t tmem_base_s;
    // 1024-byte alignment by an offset on the shared array itself, so the
    // compiler keeps shared-window addressing (LDS) for every access.
    uint8_t *smem = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int t = threadIdx.x, warp = t >> 5;

    if (warp == 0) tc05::tmem_alloc(&tmem_base_s, kTmemCols);
    if (t == 0) {
        tc05::mbar_init(&mbar[0], 1);
        tc05::mbar_init(&mbar[1], 1);
        tc05::fence_mbar_init();
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = tmem_base_s;

    pdl_wait();  // grouping and B rows come from earlier kernels
    pdl_trigger();

    const int nu = *a.n_used;
    const int total_items = nu > 0 ? a.pass_ofs[nu] * a.tiles : 0;
    const int i0 = (int)((long long)blockIdx.x * total_items / gridDim.x);
    const int i1 = (int)((long long)(blockIdx.x + 1) * total_items / gridDim.x);
    const int G = a.K / 64;
    const int total = (i1 - i0) * G;  // K groups of this CTA

    // issue-side cursor
    int is_item = 0, is_kg = 0;
    PfCursor cur{};
    if (total > 0) cur.set(a, pf_item(a, nu, i0), t);
    const uint32_t smem_s = tc05::smem_addr(smem);
    auto issue_next = [&](int j) {
        if (j < total) {
            cur.issue(smem_s + (j % kPfSlots) * kPfSlotBytes, is_kg, t);
            if (++is_kg == G) {
                is_kg = 0;
                if (++is_item < i1 - i0) cur.set(a, pf_item(a, nu, i0 + is_item), t);
            }
        }
        cp_async_commit();
    };
    for (int j = 0; j < kPfPrefetch; ++j) issue_next(j);

    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int tt = t >> 7;
    bool ok = true;
    int c_item = 0, c_kg = 0;
    PfItem c_it{};
    if (total > 0) c_it = pf_item(a, nu, i0);

    for (int j = 0; j < total && ok; ++j) {
        // A slot j&1 and data slot (j-2) % kPfSlots are free once MMA(j-2) is done.
        if (j >= 2) ok = tc05::mbar_wait(&mbar[j & 1], ((j - 2) >> 1) & 1, kWaitIters);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        issue_next(j + kPfPrefetch);
        cp_async_wait<kPfPrefetch>();
        tc05::fence_proxy_async();

        // dequantize this thread's row of group c_kg into A slot j&1, tile tt
        const uint8_t *slot = smem + (j % kPfSlots) * kPfSlotBytes;
        const uint4 w0 = *reinterpret_cast<const uint4 *>(slot + t * 16);
        const uint4 w1 = *reinterpret_cast<const uint4 *>(slot + 4096 + t * 16);
        const float sc = *reinterpret_cast<const float *>(slot + kPfWBytes + t * 4);
        uint32_t r[32];
        pf_dequant(w0, w1, sc, r);
        tc05::tmem_st32(tmem + lane_base + (uint32_t)((j & 1) * 64 + tt * 32), r);
        tc05::tmem_wait_st();
        tc05::fence_before_sync();
        __syncthreads();

        if (t == 0) {
            tc05::fence_after_sync();
            const uint32_t idesc = tc05::idesc_bf16_f32(128, c_it.npad);
            const uint32_t sB = tc05::smem_addr(slot + kPfWBytes + kPfSBytes);
#pragma unroll
            for (int tile = 0; tile < 2; ++tile) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    tc05::mma_ts(tmem + 128 + tile * 64,
                                 tmem + (uint32_t)((j & 1) * 64 + tile * 32 + kk * 8),
                                 tc05::sdesc_sw128(sB + kk * 32), idesc,
                                 (c_kg > 0 || kk > 0) ? 1u : 0u);
                }
            }
            tc05::mma_commit(&mbar[j & 1]);
        }

        if (c_kg == G - 1) {
            // item done: wait for its last MMAs, then read the accumulators.
            ok = tc05::mbar_wait(&mbar[j & 1], (j >> 1) & 1, kWaitIters);
            ok = __syncthreads_and(ok);
            if (!ok) break;
            tc05::fence_after_sync();
            const int nblk = c_it.npad / 16;
            const int r128 = t & 127;
            if (a.mode == 0) {
                // gate_up: warpgroup tt takes column blocks tt, tt+2, ...
                for (int blk = tt; blk < nblk; blk += 2) {
                    uint32_t g[16], u[16];
                    tc05::tmem_ld16(tmem + lane_base + 128 + blk * 16, g);
                    tc05::tmem_ld16(tmem + lane_base + 192 + blk * 16, u);
                    tc05::tmem_wait_ld();
                    const int j0 = c_it.tile * 128 + r128;
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int n = blk * 16 + c;
                        if (n < c_it.ntok) {
                            const float gv = __uint_as_float(g[c]), uv = __uint_as_float(u[c]);
                            const float hv = gv / (1.0f + expf(-gv)) * uv;
                            const int p = a.list[c_it.beg + n];
                            const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                            a.h[(size_t)p * a.I + j0] = *reinterpret_cast<const uint16_t *>(&hb);
                        }
                    }
                }
            } else {
                const int row = c_it.tile * 256 + tt * 128 + r128;
                for (int blk = 0; blk < nblk; ++blk) {
                    uint32_t d[16];
                    tc05::tmem_ld16(tmem + lane_base + 128 + tt * 64 + blk * 16, d);
                    tc05::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int n = blk * 16 + c;
                        if (n < c_it.ntok && row < a.H) {
                            const int p = a.list[c_it.beg + n];
                            a.y[(size_t)p * a.H + row] = __uint_as_float(d[c]);
                        }
                    }
                }
            }
            tc05::fence_before_sync();
        }
        if (++c_kg == G) {
            c_kg = 0;
            if (++c_item < i1 - i0) c_it = pf_item(a, nu, i0 + c_item);
        }
    }
    if (!ok && t == 0) atomicOr(a.status, 2);
    cp_async_wait<0>();
    // Drain the MMAs still in flight before the tensor memory is released.
    if (ok && total > 0) {
        const int jl = total - 1;
        ok = tc05::mbar_wait(&mbar[jl & 1], (jl >> 1) & 1, kWaitIters);
        if (total > 1) ok = tc05::mbar_wait(&mbar[(jl - 1) & 1], ((jl - 1) >> 1) & 1, kWaitIters) && ok;
        if (!ok && t == 0) atomicOr(a.status, 2);
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    if (warp == 0) tc05::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ pipelined variant
//
// Shapes with H/64 and I/64 multiples of 4 and 16-byte aligned pools run a
// warp-specialized version of the same computation. One CTA per SM, 26 warps,
// two rings of stages in shared memory; a stage is 256 weight rows x 4 groups
// of one item:
//   * weight producer warp: two 3-D tensor-map loads of the packed weights
//     (128 rows x 128 bytes, 128-byte swizzle) and two of their scales per
//     stage into a 3-slot ring that the dequant warps free as soon as they
//     have read a stage;
//   * B producer warp: the B tiles of the stage's 4 groups (the pass's token
//     rows, bf16, 128-byte swizzled K-major, rows rounded up to 16) by bulk
//     copy into a 3-slot ring that the MMAs free;
//   * 16 dequant warps, thread = weight row = TMEM lane, two warps per lane
//     quarter and tile: set 0 takes groups 0-1 of each stage, set 1 groups
//     2-3. Per group a thread dequantizes its row to bf16 with the scale
//     folded in and stores it to the group's A slot of its tile in tensor
//     memory; the first group's store drains while the second group is
//     dequantized;
//   * 4 MMA warps, one per (tile, half of the stage's groups): one elected
//     lane of each issues 2 groups x 4 MMAs (M 128, N = tokens rounded up to 16,
//     K 16) per stage into its own accumulator, which runs over the whole
//     item. Per stage it waits once (the A groups of its tile and set
//     stored, which the dequant warps signal only after the stage's B tiles
//     have landed) and commits once (freeing its A slots and its use of the
//     B slot); after an item it commits to the accumulator barrier. An
//     mbarrier operation of the issuing thread waits for its MMAs in flight,
//     so the fewer per MMA the better; four issuers (four accumulators, so
//     that each accumulation order stays fixed) keep the tensor pipe fed;
//   * 4 epilogue warps, one per lane quarter: they look up the next item's
//     pass (and, for down, its token rows) while the item runs, then read
//     the accumulators back with tcgen05.ld, add each tile's two halves and
//     write h = SiLU(gate) * up (bf16, straight into down's B layout) or y
//     (fp32); the MMA warps wait for them before the next item's first MMA.
// Tensor memory: D 2 tiles x 2 halves x 64 columns, A 4 groups x 2 tiles x
// 32 columns. Every wait is bounded; a wait that runs out raises a CTA-wide
// abort flag, after which nothing waits any more; copies and MMAs in flight
// are drained (bounded) before the tensor memory is released, and bit 1 of
// the status word is set.

constexpr int kPqDq = 16;                            // dequant warps
constexpr int kPqEpi = kPqDq;                        // first of 4 epilogue warps (quarters 0-3)
constexpr int kPqProdW = kPqDq + 4;                  // weight producer warp
constexpr int kPqProdB = kPqDq + 5;                  // B producer warp
constexpr int kPqMma = kPqDq + 6;                    // first of 4 MMA warps
constexpr int kPqMmaWarps = 4;
constexpr int kPqThreads = 32 * (kPqDq + 6 + kPqMmaWarps);
constexpr int kPqWStages = 3;                        // weight ring: freed after dequant
constexpr int kPqBStages = 3;                        // B ring: freed by the MMAs
constexpr int kPqOffS = 256 * 128;                   // scales [256][4] f32
constexpr int kPqWStage = kPqOffS + 256 * 16;        // 36 KB of weights and scales
constexpr int kPqBGroup = kPfMaxN * 128;             // B: 64 rows x 128 B per group
constexpr int kPqBStage = 4 * kPqBGroup;             // 32 KB
constexpr int kPqOffBRing = kPqWStages * kPqWStage;
constexpr int kPqSmem = kPqOffBRing + kPqBStages * kPqBStage + 1024;
constexpr uint32_t kPqTmaBytes = 256 * 128 + 256 * 16;
constexpr uint32_t kPqTmemCols = 512;
constexpr uint32_t kPqD = 0;                         // accumulators: (tile, half) at (2 tile + half) x 64
constexpr uint32_t kPqA = 256;                       // A: group g, tile t at g x 64 + t x 32
constexpr uint32_t kPqWait = 1u << 24;

static_assert(kPqWStage % 1024 == 0 && kPqBStage % 1024 == 0,
              "stages must stay 1024-aligned for the 128B swizzle");
static_assert(kPqBGroup % 1024 == 0, "B tiles must stay 1024-aligned");
static_assert(kPqD + 4 * kPfMaxN <= kPqA && kPqA + 4 * 64 <= kPqTmemCols,
              "tensor memory: accumulators and A slots must fit the allocation");
static_assert(kPqEpi % 4 == 0, "epilogue warp q must sit in lane quarter q");

struct PqArgs {
    CUtensorMap wmap, smap;
    int mode;            // 0: gate_up, 1: down
    int K, G, tiles, k, I, H;
    const int32_t *offsets, *list, *uexp, *n_used, *pass_ofs;
    const int4 *ptab;    // pass table (expert, first list index, tokens), or null
    const uint16_t *b;   // B rows, bf16: x [T][H] or h [P][I]
    uint16_t *h;         // gate_up output [P][I] bf16
    float *y;            // down output [P][H] fp32
    int32_t *status;
};

struct PqShared {
    uint64_t wfull[kPqWStages], wempty[kPqWStages];
    uint64_t bfull[kPqBStages];
    uint64_t afull[2][2];                      // [set][tile]: the stage's two A groups stored
    uint64_t sdone[kPqMmaWarps][kPqBStages];   // issuer m's MMAs of the stage in B slot s done
    uint64_t dfull, dfree, mdone[kPqMmaWarps];
    uint32_t tmem;
    int abort;
};


__device__ __forceinline__ bool pq_try(uint64_t *mbar, uint32_t parity) {
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
__device__ __forceinline__ bool pq_wait(PqShared &sh, uint64_t *mbar, uint32_t parity) {
    volatile int *ab = &sh.abort;
    for (uint32_t i = 0; i < kPqWait; ++i) {
        if (pq_try(mbar, parity)) return true;
        if ((i & 15u) == 15u && *ab) return false;
    }
    *ab = 1;
    return false;
}

// pq_wait by every lane of a warp, with one answer for all of them, so the
// warp leaves its loop together (its .sync.aligned instructions need that).
__device__ __forceinline__ bool pq_wait_warp(PqShared &sh, uint64_t *mbar, uint32_t parity) {
    return __all_sync(0xffffffffu, pq_wait(sh, mbar, parity));
}

// Bounded wait that ignores the abort flag (draining work in flight).
__device__ __forceinline__ void pq_drain(uint64_t *mbar, uint32_t parity) {
    for (uint32_t i = 0; i < kPqWait; ++i)
        if (pq_try(mbar, parity)) return;
}

__device__ __forceinline__ void pq_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     tc05::smem_addr(mbar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void pq_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc05::smem_addr(mbar))
                 : "memory");
}

__device__ __forceinline__ void pq_tma3(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                        uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void pq_bulk(uint32_t dst, const void *src, uint32_t bytes,
                                        uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
        : "memory");
}

// tcgen05.mma (A in tensor memory) from a warp-uniform branch: every lane of
// the warp runs the instruction stream and elect.sync picks the lane that
// issues, so the operands the whole warp computes stay warp-uniform. A probe
// issued ~34 cycles per MMA this way against ~66 from a loop that a single
// lane runs (and ~16 cycles per MMA of tensor pipe at N 32 with two issuers).
__device__ __forceinline__ void pq_mma_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Commit of the MMAs issued by pq_mma_elect: with all 32 lanes active the
// same lane is elected, the one whose MMAs the commit tracks.
__device__ __forceinline__ void pq_commit_elect(uint64_t *mbar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            tc05::smem_addr(mbar))
        : "memory");
}

// Walks the passes (up to kPfMaxN pairs of one expert) in order.
struct PqCursor {
    int lo, pi, e, beg, ntok;
    __device__ __forceinline__ void seek(const PqArgs &a, int nu, int p) {
        if (a.ptab) {  // one load a pass instead of a search and walk
            pi = -1;
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
    __device__ __forceinline__ void to(const PqArgs &a, int p) {
        if (p == pi) return;
        if (a.ptab) {
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
        beg = b + pass * kPfMaxN;
        ntok = min(kPfMaxN, cnt - pass * kPfMaxN);
    }
};

__global__ void __launch_bounds__(kPqThreads, 1) k_prefill_tma(const __grid_constant__ PqArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ PqShared sh;
    // 1024-byte alignment by an offset on the shared array itself (keeps LDS)
    uint8_t *ring = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) tc05::tmem_alloc(&sh.tmem, kPqTmemCols);
    if (threadIdx.x == 32) {
        for (int s = 0; s < kPqWStages; ++s) {
            tc05::mbar_init(&sh.wfull[s], 1);
            tc05::mbar_init(&sh.wempty[s], kPqDq);
        }
        for (int s = 0; s < kPqBStages; ++s) {
            tc05::mbar_init(&sh.bfull[s], 1);
            for (int m = 0; m < kPqMmaWarps; ++m) tc05::mbar_init(&sh.sdone[m][s], 1);
        }
        for (int g = 0; g < 2; ++g)
            for (int t = 0; t < 2; ++t) tc05::mbar_init(&sh.afull[g][t], 4);  // 4 lane quarters
        tc05::mbar_init(&sh.dfull, kPqMmaWarps);
        tc05::mbar_init(&sh.dfree, 4);
        for (int m = 0; m < kPqMmaWarps; ++m) tc05::mbar_init(&sh.mdone[m], 1);
        sh.abort = 0;
        tc05::fence_mbar_init();
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = sh.tmem;

    // The grouping finished before the previous kernel (the x packing, or
    // gate_up) started, and the weights depend on no kernel, so the weight
    // producer never waits; everything that reads packed B or writes h / y does.
    if (warp != kPqProdW) pdl_wait();
    pdl_trigger();

    // with the pass table the grouping kernel also wrote the pass count
    // next to n_used (one load); else it is pass_ofs[n_used]
    int nu = 0, npass;
    if (a.ptab) {
        npass = a.n_used[1];
    } else {
        nu = *a.n_used;
        npass = nu > 0 ? a.pass_ofs[nu] : 0;
    }
    const int total_items = npass * a.tiles;
    // Items are dealt out round-robin (CTA c takes items c, c + grid, ...), so
    // at any time the CTAs work on ~grid consecutive items: the tiles of a
    // few passes, whose packed B and (passes of one expert) weights are then
    // read from DRAM once and served from L2 to the other CTAs. Contiguous
    // ranges would spread each pass's re-reads over the whole launch.
    const int i0 = (int)blockIdx.x, istep = (int)gridDim.x;
    const int n_items = i0 < total_items ? (total_items - i0 + istep - 1) / istep : 0;
    const int ns = a.G / 4;
    const int total = n_items * ns;  // stages of this CTA

    if (warp == kPqProdW) {
        // ---------------- weight producer (one thread)
        if (lane == 0) {
            PqCursor pc;
            if (total > 0) pc.seek(a, nu, i0 / a.tiles);
            int issued = 0;
            for (int j = 0; j < total; ++j) {
                const int ws = j % kPqWStages;
                if (j >= kPqWStages &&
                    !pq_wait(sh, &sh.wempty[ws], (uint32_t)(((j / kPqWStages) - 1) & 1)))
                    break;
                const int item = i0 + (j / ns) * istep, kb = j % ns;
                pc.to(a, item / a.tiles);
                const int tile = item % a.tiles;
                const int rowA = a.mode == 0 ? tile * 128 : tile * 256;
                const int rowB = a.mode == 0 ? a.I + tile * 128 : tile * 256 + 128;
                const uint32_t base = tc05::smem_addr(ring + ws * kPqWStage);
                const uint32_t fb = tc05::smem_addr(&sh.wfull[ws]);
                pq_expect_tx(&sh.wfull[ws], kPqTmaBytes);
                pq_tma3(base, &a.wmap, kb * 128, rowA, pc.e, fb);
                pq_tma3(base + 128 * 128, &a.wmap, kb * 128, rowB, pc.e, fb);
                pq_tma3(base + kPqOffS, &a.smap, kb * 4, rowA, pc.e, fb);
                pq_tma3(base + kPqOffS + 128 * 16, &a.smap, kb * 4, rowB, pc.e, fb);
                issued = j + 1;
            }
            // drain: every tensor copy issued must land before the CTA may exit
            for (int j = (issued > kPqWStages ? issued - kPqWStages : 0); j < issued; ++j)
                pq_drain(&sh.wfull[j % kPqWStages], (uint32_t)((j / kPqWStages) & 1));
        }
    } else if (warp == kPqProdB) {
        // ---------------- B producer (one thread): per stage the 4 groups'
        // packed B tiles of the pass, rows rounded up to 16, by bulk copy
        if (lane == 0) {
            PqCursor pc;
            if (total > 0) pc.seek(a, nu, i0 / a.tiles);
            int issued = 0;
            for (int j = 0; j < total; ++j) {
                const int bs = j % kPqBStages;
                // the slot is free once every issuer's MMAs of stage j - kPqBStages are done
                bool free = true;
                for (int m = 0; m < kPqMmaWarps && j >= kPqBStages && free; ++m)
                    free = pq_wait(sh, &sh.sdone[m][bs], (uint32_t)(((j / kPqBStages) - 1) & 1));
                if (!free) break;
                const int item = i0 + (j / ns) * istep, kb = j % ns, pi = item / a.tiles;
                pc.to(a, pi);
                const uint32_t bytes = (uint32_t)(((pc.ntok + 15) & ~15) * 128);
                const uint32_t dst = tc05::smem_addr(ring + kPqOffBRing + bs * kPqBStage);
                const uint32_t fb = tc05::smem_addr(&sh.bfull[bs]);
                pq_expect_tx(&sh.bfull[bs], 4 * bytes);
                for (int g = 0; g < 4; ++g)
                    pq_bulk(dst + g * kPqBGroup,
                            a.b + ((size_t)pi * a.G + 4 * kb + g) * (kPqBGroup / 2), bytes, fb);
                issued = j + 1;
            }
            // drain: every copy issued must land before the CTA may exit
            for (int j = (issued > kPqBStages ? issued - kPqBStages : 0); j < issued; ++j)
                pq_drain(&sh.bfull[j % kPqBStages], (uint32_t)((j / kPqBStages) & 1));
        }
    } else if (warp >= kPqMma) {
        // ---------------- MMA issue: warp kPqMma + m: tile m / 2, groups 2(m % 2), +1.
        // The whole warp runs the loop (warp-uniform operands); one elected
        // lane issues the MMAs and the commits. Every mbarrier operation of
        // the issuing lane after an MMA costs a few hundred cycles (it waits
        // for the MMAs issued so far to be taken up), so a stage has one wait
        // for its A groups and one commit.
        const int m = warp - kPqMma, t = m >> 1, hk = m & 1;
        PqCursor pc;
        if (total > 0) pc.seek(a, nu, i0 / a.tiles);
        const uint32_t dacc = tmem + kPqD + (uint32_t)(m * 64);
        const uint32_t a0 = tmem + kPqA + (uint32_t)(2 * hk * 64 + t * 32);
        // B descriptor of slot 0, group 2 hk; +1 in the address field = 16 bytes
        const uint64_t b0 = tc05::sdesc_sw128(
            tc05::smem_addr(ring + kPqOffBRing + 2 * hk * kPqBGroup));
        bool ok = true;
        for (int j = 0; j < total && ok; ++j) {
            const int bs = j % kPqBStages;
            const int it = j / ns, kb = j % ns;
            pc.to(a, (i0 + it * istep) / a.tiles);
            const uint32_t idesc = tc05::idesc_bf16_f32(128, (pc.ntok + 15) & ~15);
            // the accumulators are free once the epilogue has read the last item
            if (kb == 0 && it > 0) ok = pq_wait_warp(sh, &sh.dfree, (uint32_t)((it - 1) & 1));
            // A of this stage stored, and its B landed (the dequant warps check that)
            if (ok) ok = pq_wait_warp(sh, &sh.afull[hk][t], (uint32_t)(j & 1));
            if (!ok) break;
            tc05::fence_after_sync();
            const uint64_t bd = b0 + (uint64_t)((bs * kPqBStage) >> 4);
#pragma unroll
            for (int gg = 0; gg < 2; ++gg)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    pq_mma_elect(dacc, a0 + (uint32_t)(gg * 64 + kk * 8),
                                 bd + (uint64_t)((gg * kPqBGroup + kk * 32) >> 4), idesc,
                                 (kb > 0 || gg > 0 || kk > 0) ? 1u : 0u);
            // frees this issuer's A slots and its use of the B slot
            pq_commit_elect(&sh.sdone[m][bs]);
            if (kb == ns - 1) pq_commit_elect(&sh.dfull);
        }
        // the MMAs still in flight must finish before the tensor memory is freed
        pq_commit_elect(&sh.mdone[m]);
        pq_drain(&sh.mdone[m], 0);
    } else if (warp >= kPqEpi && warp < kPqEpi + 4) {
        // ---------------- epilogue: lane quarter q of both tiles
        const int q = warp & 3, r128 = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        PqCursor pc;
        if (total > 0) pc.seek(a, nu, i0 / a.tiles);
        for (int it = 0; it < n_items; ++it) {
            const int item = i0 + it * istep, tile = item % a.tiles;
            pc.to(a, item / a.tiles);
            const int ntok = pc.ntok, nblk = ((ntok + 15) & ~15) / 16;
            // down scatters to the pairs' rows: lane l holds pairs l and 32 + l
            int p0 = 0, p1 = 0;
            if (a.mode == 1) {
                if (lane < ntok) p0 = a.list[pc.beg + lane];
                if (lane + 32 < ntok) p1 = a.list[pc.beg + 32 + lane];
            }
            if (!pq_wait_warp(sh, &sh.dfull, (uint32_t)(it & 1))) break;
            tc05::fence_after_sync();
            if (a.mode == 0) {
                // h goes straight into down's packed B: pass pc.pi, group j0 / 64,
                // row n = token slot, column j0 % 64 in the dequant's K order (swizzled)
                const int j0 = tile * 128 + r128;
                const int kp = kperm_pos(j0 & 63);
                uint16_t *hp = a.h + ((size_t)pc.pi * (a.I / 64) + (j0 >> 6)) * (kPqBGroup / 2);
                // tile t, half h accumulates at kPqD + (2t + h) * 64: gate is tile 0,
                // up tile 1; 8 token columns at a time
                for (int c0 = 0; c0 < nblk * 16; c0 += 8) {
                    float gs[8];
                    uint32_t v0[8], v1[8];
                    tc05::tmem_ld8(tmem + lane_base + kPqD + c0, v0);
                    tc05::tmem_ld8(tmem + lane_base + kPqD + 64 + c0, v1);
                    tc05::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) gs[c] = __uint_as_float(v0[c]) + __uint_as_float(v1[c]);
                    tc05::tmem_ld8(tmem + lane_base + kPqD + 128 + c0, v0);
                    tc05::tmem_ld8(tmem + lane_base + kPqD + 192 + c0, v1);
                    tc05::tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int n = c0 + c;
                        float hv = 0.f;  // padded rows stay zero
                        if (n < ntok) {
                            const float g0 = gs[c];
                            hv = g0 / (1.0f + expf(-g0)) *
                                 (__uint_as_float(v0[c]) + __uint_as_float(v1[c]));
                        }
                        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                        hp[n * 64 + (((kp >> 3) ^ (n & 7)) << 3) + (kp & 7)] =
                            *reinterpret_cast<const uint16_t *>(&hb);
                    }
                }
            } else {
                const int row = tile * 256 + r128;
#pragma unroll 1
                for (int t = 0; t < 2; ++t)  // rows t * 128 + r128 of the tile
                    for (int c0 = 0; c0 < nblk * 16; c0 += 8) {
                        uint32_t d0[8], d1[8];
                        tc05::tmem_ld8(tmem + lane_base + kPqD + t * 128 + c0, d0);
                        tc05::tmem_ld8(tmem + lane_base + kPqD + t * 128 + 64 + c0, d1);
                        tc05::tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int n = c0 + c;
                            const int p = __shfl_sync(0xffffffffu, n < 32 ? p0 : p1, n & 31);
                            if (n < ntok)
                                a.y[(size_t)p * a.H + row + t * 128] =
                                    __uint_as_float(d0[c]) + __uint_as_float(d1[c]);
                        }
                    }
            }
            tc05::fence_before_sync();
            __syncwarp();
            if (lane == 0) pq_arrive(&sh.dfree);
        }
    } else {
        // ---------------- dequant warps
        const int set = warp >> 3, tt = (warp >> 2) & 1, q = warp & 3;
        const int r = tt * 128 + q * 32 + lane;     // stage row; TMEM lane q*32 + lane
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint32_t a_col = tmem + lane_base + kPqA + (uint32_t)(tt * 32);
        const int x7 = r & 7, ga = 2 * set;
        bool ok = true;
        for (int j = 0; j < total && ok; ++j) {
            const int ws = j % kPqWStages;
            ok = pq_wait_warp(sh, &sh.wfull[ws], (uint32_t)((j / kPqWStages) & 1));
            if (!ok) break;
            const uint8_t *sp = ring + ws * kPqWStage;
            const uint8_t *wr = sp + r * 128;
            const float2 sc = *reinterpret_cast<const float2 *>(sp + kPqOffS + r * 16 + ga * 4);
            const uint4 wa0 = *reinterpret_cast<const uint4 *>(wr + (((2 * ga) ^ x7) << 4));
            const uint4 wa1 = *reinterpret_cast<const uint4 *>(wr + (((2 * ga + 1) ^ x7) << 4));
            uint32_t A[32];
            pf_dequant_fast(wa0, wa1, sc.x, A);
            if (j > 0) {
                // the MMAs of the previous stage that read this warp's A slots are done
                ok = pq_wait_warp(sh, &sh.sdone[2 * tt + set][(j - 1) % kPqBStages],
                                  (uint32_t)(((j - 1) / kPqBStages) & 1));
                tc05::fence_after_sync();
            }
            if (!ok) break;
            tc05::tmem_st32(a_col + (uint32_t)(ga * 64), A);
            // the second group is dequantized while the first one's store drains
            {
                const uint4 wb0 = *reinterpret_cast<const uint4 *>(wr + (((2 * ga + 2) ^ x7) << 4));
                const uint4 wb1 = *reinterpret_cast<const uint4 *>(wr + (((2 * ga + 3) ^ x7) << 4));
                pf_dequant_fast(wb0, wb1, sc.y, A);
            }
            // this warp has read its rows of the stage: the weight slot may refill
            if (lane == 0) pq_arrive(&sh.wempty[ws]);
            tc05::tmem_st32(a_col + (uint32_t)((ga + 1) * 64), A);
            // the MMA warps wait on one barrier a stage: the first lane quarter
            // also checks that the stage's B tiles have landed
            if (q == 0) ok = pq_wait_warp(sh, &sh.bfull[j % kPqBStages], (uint32_t)((j / kPqBStages) & 1));
            tc05::tmem_wait_st();
            tc05::fence_before_sync();
            __syncwarp();
            if (!ok) break;
            if (lane == 0) pq_arrive(&sh.afull[set][tt]);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && sh.abort) atomicOr(a.status, 2);
    tc05::fence_after_sync();
    if (warp == 0) tc05::tmem_dealloc(tmem, kPqTmemCols);
}

// Packs the rows of x (bf16 [T][H]) that each pass uses into the MMA's B
// layout, each group's 64 values in the dequant's K order (kperm_pos):
// xp[pass][g][64 rows][64 bf16], row t = token slot t of the pass
// (zero from its token count up to the next multiple of 16), 128-byte
// swizzled. Grid (passes at most, ceil(G / 8)); warp w packs group
// 8 * blockIdx.y + w of pass blockIdx.x. The passes come from the grouping
// kernel's pass table, their count from the word after n_used.
__global__ void __launch_bounds__(256)
    k_pack_x(const uint16_t *__restrict__ x, int H, int k, const int32_t *list,
             const int32_t *n_used, const int4 *ptab, uint4 *xp) {
    pdl_wait();  // the grouping comes from the previous kernel
    pdl_trigger();
    const int pi = blockIdx.x;
    // the pass table entry and the pass count (next to n_used), one load each
    const int4 pt = ptab[pi];
    if (pi >= n_used[1]) return;
    const int beg = pt.y, ntok = pt.z;
    const int npad = (ntok + 15) & ~15;
    const int G = H / kGroup;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.y * 8 + warp;
    if (g >= G) return;
    uint4 *dst = xp + ((size_t)pi * G + g) * (kPfMaxN * 8);
    for (int c = lane; c < npad * 8; c += 32) {
        const int t = c >> 3, ch = c & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < ntok) {
            const int row = list[beg + t] / k;
            const uint4 u = *reinterpret_cast<const uint4 *>(x + (size_t)row * H + g * kGroup + ch * 8);
            // the dequant's K order (kperm_pos): elements (0,4,1,5,2,6,3,7) of the chunk
            v = make_uint4(prmt(u.x, u.z, 0x5410), prmt(u.x, u.z, 0x7632), prmt(u.y, u.w, 0x5410),
                           prmt(u.y, u.w, 0x7632));
        }
        dst[t * 8 + (ch ^ (t & 7))] = v;
    }
}

}  // namespace

cudaError_t launch_prefill(const MoeDims &m, int mode, const uint16_t *b, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, uint16_t *h, float *y,
                           int32_t *status, cudaStream_t st, const int4 *ptab) {
    if (tma_moe_supported(m)) {
        PqArgs q;
        memset(&q, 0, sizeof(q));
        q.mode = mode;
        q.k = k;
        q.I = m.I;
        q.H = m.H;
        q.offsets = offsets; q.list = list; q.uexp = uexp; q.n_used = n_used; q.pass_ofs = pass_ofs;
        q.ptab = ptab;
        q.b = b;
        q.h = h;
        q.y = y;
        q.status = status;
        bool ok;
        if (mode == 0) {
            q.K = m.H;
            q.tiles = m.I / 128;
            ok = encode_weight_maps(&q.wmap, &q.smap, m.gu_q, m.gu_s, m.E, 2 * m.I, m.H);
        } else {
            q.K = m.I;
            q.tiles = m.H / 256;
            ok = encode_weight_maps(&q.wmap, &q.smap, m.dn_q, m.dn_s, m.E, m.H, m.I);
        }
        q.G = q.K / kGroup;
        if (!ok) return cudaErrorInvalidValue;
        cudaError_t e = set_smem(k_prefill_tma, kPqSmem);
        if (e != cudaSuccess) return e;
        const int grid = sm_count() * max_ctas_per_sm(k_prefill_tma, kPqThreads, kPqSmem);
        return launch(k_prefill_tma, dim3(grid), dim3(kPqThreads), (size_t)kPqSmem, st, true, q);
    }
    PfArgs a{};
    a.k = k;
    a.offsets = offsets; a.list = list; a.uexp = uexp; a.n_used = n_used; a.pass_ofs = pass_ofs;
    a.h = h; a.y = y; a.I = m.I; a.H = m.H; a.mode = mode; a.status = status;
    a.b = b;
    if (mode == 0) {
        a.wq = m.gu_q; a.ws = m.gu_s;
        a.rows = 2 * m.I; a.K = m.H;
        a.eq = (size_t)2 * m.I * (m.H / 2); a.es = (size_t)2 * m.I * (m.H / 64);
        a.tiles = m.I / 128;
        a.by_pair = 0;
    } else {
        a.wq = m.dn_q; a.ws = m.dn_s;
        a.rows = m.H; a.K = m.I;
        a.eq = (size_t)m.H * (m.I / 2); a.es = (size_t)m.H * (m.I / 64);
        a.tiles = (m.H + 255) / 256;
        a.by_pair = 1;
    }
    cudaError_t e = set_smem(k_prefill, kPfSmem);
    if (e != cudaSuccess) return e;
    const int grid = sm_count() * max_ctas_per_sm(k_prefill, kPfThreads, kPfSmem);
    return launch(k_prefill, dim3(grid), dim3(kPfThreads), (size_t)kPfSmem, st, true, a);
}

int prefill_pass_tokens() { return kPfMaxN; }

cudaError_t launch_pack_x(const uint16_t *x, int H, int k, const int32_t *list,
                          const int32_t *n_used, const int4 *ptab, uint16_t *xp, int pmax,
                          cudaStream_t st) {
    if (pmax < 1) return cudaSuccess;
    return launch(k_pack_x, dim3(pmax, (H / kGroup + 7) / 8), dim3(256), 0, st, true, x, H, k,
                  list, n_used, ptab, reinterpret_cast<uint4 *>(xp));
}

}  // namespace qmv
