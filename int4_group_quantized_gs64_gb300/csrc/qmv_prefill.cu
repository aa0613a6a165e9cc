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

}  // namespace

cudaError_t launch_prefill(const MoeDims &m, int mode, const uint16_t *b, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, uint16_t *h, float *y,
                           int32_t *status, cudaStream_t st) {
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

}  // namespace qmv
