// qmv_moe.cu - MoE decode: top-k routing, token->expert grouping, fused
// gate+up with SiLU*mul, down projection and the weighted combine.
//
// colibri PR #418 "Vulkan backend: expert tier + dense + MLA attention on any
// Vulkan 1.2 GPU": commit "qmatmul_gate_up.comp + coli_vk_gate_up" (hidden =
// silu(gate(x)) * up(x), x read once for both), commit "coli_vk_expert_group"
// (K experts: fused gate+up+silu, then down, hidden kept on the device);
// PR #1338 "qwen36: Vulkan expert tier, and staged device-local uploads"
// (weighted accumulation of the expert outputs).
//
// Expert weights are read once per batch: moe_group turns the token->expert
// ids into per-expert pair lists, and every gate+up / down CTA works on one
// expert's row tile for all of that expert's tokens at once.
#include <float.h>
#include <limits.h>

#include <algorithm>

#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_route.cuh"
#include "qmv_rows.cuh"

namespace qmv {

namespace {

// ------------------------------------------------------------------ routing

// One warp per token; the token's logits are staged in shared memory once,
// lane L owns experts L, L+32, ... (E <= 1024).
constexpr int kRouteWarps = 8;

__global__ void __launch_bounds__(32 * kRouteWarps)
    k_route(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ ids,
            float *__restrict__ w) {
    __shared__ float sl[kRouteWarps][1024];
    // Launched with programmatic dependent launch: the logits may come from
    // the previous kernel and it may still read ids / w of an earlier call,
    // so wait for it before touching either; a dependent launched the same
    // way waits for this grid before reading ids.
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const int t = blockIdx.x * kRouteWarps + wl;
    if (t >= T) return;
    int my_id;
    float my_w;
    route_warp(logits + (size_t)t * E, E, k, sl[wl], my_id, my_w);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = my_w;
    }
}

// ------------------------------------------------------------------ grouping

// Exclusive block scan of three per-thread values (blockDim.x == 1024): warp
// scans, the warp totals through shared memory, and each warp adds the
// totals of the warps before it with one warp reduction per value (one
// barrier). The caller synchronises before it writes `tot` again.
__device__ __forceinline__ void block_scan3(int a, int b, int c, int &ea, int &eb, int &ec,
                                            int *tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b, ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, ia, o);
        const int y = __shfl_up_sync(0xFFFFFFFFu, ib, o);
        const int z = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        if (lane >= o) { ia += x; ib += y; ic += z; }
    }
    if (lane == 31) { tot[warp] = ia; tot[32 + warp] = ib; tot[64 + warp] = ic; }
    __syncthreads();
    const bool before = lane < warp;
    ea = (int)__reduce_add_sync(0xFFFFFFFFu, before ? (unsigned)tot[lane] : 0u) + ia - a;
    eb = (int)__reduce_add_sync(0xFFFFFFFFu, before ? (unsigned)tot[32 + lane] : 0u) + ib - b;
    ec = (int)__reduce_add_sync(0xFFFFFFFFu, before ? (unsigned)tot[64 + lane] : 0u) + ic - c;
}

// a / b for non-negative a, b: one 32-bit division when both fit in 32 bits
// (the plan's stage and cost numbers nearly always do), else the 64-bit one.
__device__ __forceinline__ long long div_nn(long long a, long long b) {
    if ((((unsigned long long)a | (unsigned long long)b) >> 32) == 0)
        return (long long)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// Grouping on one CTA of 1024 threads: counts by shared atomics; block scans
// give the offsets, the slots of the used experts and the pass offsets (one
// pass = up to kMaxTok pairs of one expert); then the warps place the pairs
// in parallel (below), keeping the lists ascending.
// res: bitmap of the experts this call serves (bit e % 32 of word e / 32), or
// null for all; pairs of other experts are left out of the lists without
// error. served (if not null): 1 for each pair that is grouped, else 0.
//
// With a work plan (pl && pl->ptab): the pass table and, for gate+up and for
// down, the first stage of every CTA, so that each CTA's stages carry the
// same cost (PlanArgs: weighted stages plus a cost per row tile's end). The
// stages of used expert u start at cost wpre[u] (exclusive scan of the
// experts' costs); CTA b starts at cost C * b / g of the total C, inside the
// pass and row tile that cost falls in, at the first stage whose start is
// not below it.
__device__ void group_cta(const int32_t *__restrict__ ids, int P, int E, int32_t *offsets,
                          int32_t *list, int32_t *uexp, int32_t *n_used, int32_t *pass_ofs,
                          int32_t *status, int pass_tok, const uint32_t *res = nullptr,
                          uint8_t *served = nullptr, const PlanArgs *pl = nullptr) {
    __shared__ int32_t cnt[1024], tot[96];
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = 0;
    cnt[tid] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = ids[p];
        const bool in = e >= 0 && e < E;
        if (!in) bad = 1;
        else if (expert_served(res, e)) atomicAdd(&cnt[e], 1);
        if (served) served[p] = in && expert_served(res, e) ? 1 : 0;
    }
    __syncthreads();
    const int c = tid < E ? cnt[tid] : 0;
    const int f = c > 0 ? 1 : 0;
    const int np = (c + pass_tok - 1) / pass_tok;
    int ec, ef, ep;
    block_scan3(c, f, np, ec, ef, ep, tot);
    // shared copies for the plan below (reading back the global ones would
    // cost a round trip to L2 for every dependent step): the expert offsets,
    // the used experts and their first passes, in the dynamic shared memory
    // (at least 32 E words; the routing's ids, if any, lie beyond 32 E)
    extern __shared__ int32_t group_smem[];
    int32_t *s_off = group_smem, *s_uexp = group_smem + (E + 1), *s_pofs = group_smem + 2 * (E + 1);
    if (tid < E) {
        offsets[tid] = ec;
        s_off[tid] = ec;
        if (f) {
            uexp[ef] = tid;
            s_uexp[ef] = tid;
            s_pofs[ef] = ep;
            if (pass_ofs) pass_ofs[ef] = ep;
        }
    }
    if (tid == E - 1) {
        offsets[E] = ec + c;
        s_off[E] = ec + c;
        *n_used = ef + f;
        // with a pass table (the library's own workspaces, whose n_used slot
        // has room) the pass count too, so that a reader needs one load
        if (pl && pl->ptab) n_used[1] = ep + np;
        s_pofs[ef + f] = ep + np;
        if (pass_ofs) pass_ofs[ef + f] = ep + np;
    }
    // the plan's arguments, read once
    const PlanArgs pa = pl ? *pl : PlanArgs{};
    // the pass table (expert, first list index, tokens of every pass)
    if (pa.ptab && f)
        for (int i = 0; i < np; ++i)
            pa.ptab[ep + i] = make_int4(tid, ec + i * pass_tok, min(pass_tok, c - i * pass_tok), 0);
    if (pa.ptab && pa.plan_gu) {
        // Cost of a pass of mode m: its T row tiles of N stages each, a stage
        // weighing w (kPlanW2, or for an expert's last pass by its token
        // count), plus kPlanItem at the end of each tile. Each used expert's
        // cost in both modes, scanned at once: the prefix of gate+up in
        // cnt[], that of down in s_wdn[].
        __shared__ int32_t nu_s;
        __shared__ long long wtot_s[2];
        int32_t *s_wdn = group_smem + 3 * (E + 1);
        auto pass_cost = [&](int m, int w) -> int {
            const int N = m ? pa.ns_dn : pa.ns_gu, T = (m ? pa.s_dn : pa.s_gu) / N;
            return T * (N * w + kPlanItem);
        };
        int wgu = 0, wdn = 0;
        if (f) {
            const int wl = c - (np - 1) * pass_tok > 4 ? kPlanW2 : kPlanW1;
            wgu = (np - 1) * pass_cost(0, kPlanW2) + pass_cost(0, wl);
            wdn = (np - 1) * pass_cost(1, kPlanW2) + pass_cost(1, wl);
        }
        int egu, edn, d2;
        __syncthreads();  // cnt[] (c) has been read: reuse it
        block_scan3(wgu, wdn, 0, egu, edn, d2, tot);
        if (f) {
            cnt[ef] = egu;
            s_wdn[ef] = edn;
        }
        if (tid == E - 1) {
            nu_s = ef + f;
            wtot_s[0] = (long long)egu + wgu;
            wtot_s[1] = (long long)edn + wdn;
        }
        __syncthreads();
        const int nu = nu_s;
        const int npass = nu > 0 ? s_pofs[nu] : 0;
        // (expert, first list index, tokens) of pass p, which is a pass of
        // used expert lo or the first pass of the next one (as in ptab)
        auto pass_at = [&](int p, int lo) -> int4 {
            if (p >= npass) return make_int4(0, 0, 0, 0);
            const int l = p >= s_pofs[lo + 1] ? lo + 1 : lo;
            const int e = s_uexp[l], i = p - s_pofs[l];
            const int ce = s_off[e + 1] - s_off[e];
            return make_int4(e, s_off[e] + i * pass_tok, min(pass_tok, ce - i * pass_tok), 0);
        };
        // one thread per (mode, CTA boundary b): both modes at once. CTA b
        // starts at cost C * b / g: in the pass, row tile and stage that cost
        // falls in, at the first stage whose start is not below it.
        const int g = pa.g;
        for (int idx = tid; idx < 2 * (g + 1); idx += blockDim.x) {
            const int m = idx / (g + 1), b = idx - m * (g + 1);
            const long long S = m ? pa.s_dn : pa.s_gu;
            const int N = m ? pa.ns_dn : pa.ns_gu, T = (int)(S / N);
            const int32_t *wp = m ? s_wdn : cnt;
            int32_t ub;
            int lo = 0;
            if (nu == 0) {
                ub = 0;
            } else if (b == g) {
                ub = (int32_t)(S * npass);
            } else {
                const long long cb = div_nn(wtot_s[m] * b, g);
                int hi = nu - 1;  // last used expert whose cost starts at or below cb
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (wp[mid] <= cb) lo = mid; else hi = mid - 1;
                }
                const int e = s_uexp[lo];
                const int ce = s_off[e + 1] - s_off[e];
                const int npe = (ce + pass_tok - 1) / pass_tok;
                const int wl = ce - (npe - 1) * pass_tok > 4 ? kPlanW2 : kPlanW1;
                const long long r = cb - wp[lo];
                const int i = (int)min((long long)(npe - 1), div_nn(r, pass_cost(m, kPlanW2)));
                const long long r2 = r - (long long)i * pass_cost(m, kPlanW2);
                const int wi = i < npe - 1 ? kPlanW2 : wl;
                const long long tc = (long long)N * wi + kPlanItem;  // a row tile of this pass
                const int it = (int)min((long long)(T - 1), div_nn(r2, tc));
                const long long r3 = r2 - (long long)it * tc;
                const long long st = min((long long)N, div_nn(r3 + wi - 1, wi));
                ub = (int32_t)(S * (s_pofs[lo] + i) + (long long)it * N + st);
            }
            const int4 t = pass_at((int)div_nn(ub, S), lo);  // the pass holding stage ub, if any
            (m ? pa.plan_dn : pa.plan_gu)[b] = make_int4(ub, t.x, t.y, t.z);
        }
    }
    // The list, in pair order within each expert. Up to 1024 pairs (a decode
    // micro-batch), warp w places the pairs of the experts e with e % 32 == w,
    // walking all pairs 32 at a time, so each expert's running position has one
    // writer. More pairs: warp w takes the w-th 32nd of the pairs; hist[w][e]
    // counts its pairs of expert e, a scan over w turns the counts into each
    // segment's first list position for e, and the warp places its pairs in
    // order, 32 at a time. Ranks among the lanes come from __match_any_sync. The
    // positions live in the dynamic shared memory (32 x E ints).
    __syncthreads();  // the scan's reads of tot[] and the plan's of group_smem are done
    if (P <= 1024) {
        int32_t *run = group_smem;
        if (tid < E) run[tid] = ec;
        __syncthreads();
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            const int e = p < P ? ids[p] : -1;
            const bool mine = p < P && e >= 0 && e < E && (e & 31) == warp && expert_served(res, e);
            if (__ballot_sync(0xFFFFFFFFu, mine) == 0) continue;
            // the lanes holding the same expert (other lanes get unique keys)
            const unsigned same = __match_any_sync(0xFFFFFFFFu, mine ? e : -1 - lane);
            const int rank = __popc(same & ((1u << lane) - 1u));
            const int after = __popc(same & ~((2u << lane) - 1u));
            if (mine) list[run[e] + rank] = p;
            __syncwarp();
            if (mine && after == 0) run[e] += rank + 1;
            __syncwarp();
        }
    } else {
        int32_t *hist = group_smem, *hw = group_smem + warp * E;
        const int seg = (P + 31) / 32, s0 = min(P, warp * seg), s1 = min(P, s0 + seg);
        for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int p = s0 + lane; p < s1; p += 32) {
            const int e = ids[p];
            if (e >= 0 && e < E && expert_served(res, e)) atomicAdd(&hw[e], 1);
        }
        __syncthreads();
        if (tid < E) {
            int at = ec;
            for (int w = 0; w < 32; ++w) {
                const int h = hist[w * E + tid];
                hist[w * E + tid] = at;
                at += h;
            }
        }
        __syncthreads();
        for (int base = s0; base < s1; base += 32) {
            const int p = base + lane;
            int e = p < s1 ? ids[p] : -1;
            const bool valid = p < s1 && e >= 0 && e < E && expert_served(res, e);
            if (!valid) e = -1 - lane;  // unique key: never matches another lane
            const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
            const int rank = __popc(same & ((1u << lane) - 1u));
            const int after = __popc(same & ~((2u << lane) - 1u));
            if (valid) list[hw[e] + rank] = p;
            __syncwarp();
            if (valid && after == 0) hw[e] += rank + 1;
            __syncwarp();
        }
    }
    if (tid == 0 && bad) atomicOr(status, 1);
}

// Splits groups g0 .. g0 + 31 of activation row r (1024 threads, one group
// a warp): per 64-wide group, max |v| -> power-of-two factor -> 16 fp16 hi/lo
// cells (int4 register order). sub: the tensor-map kernel's int4 form, with a
// (factor, offset_init) record per group (fac [G][2]); else fac [G].
__device__ void split_row_cta(const float *__restrict__ row, int K, int g0, uint4 *cells,
                              float *fac, bool sub) {
    __shared__ float buf[32][64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = K / kGroup;
    for (int g = g0 + warp; g < min(G, g0 + 32); g += blockDim.x >> 5) {
        const float a = row[g * kGroup + lane], b = row[g * kGroup + 32 + lane];
        const int e = split_exponent(warp_max(fmaxf(fabsf(a), fabsf(b))));
        const float mul = ldexpf(1.0f, e);
        buf[warp][lane] = a * mul;
        buf[warp][32 + lane] = b * mul;
        __syncwarp();
        if (sub) {
            const float sum = warp_sum(a * mul + b * mul);
            if (lane < 16) cells[(size_t)g * 16 + lane] = make_unit_s(buf[warp], lane);
            if (lane == 0)
                reinterpret_cast<float2 *>(fac)[g] = make_float2(ldexpf(1.0f, -e), offset_init(sum));
        } else {
            if (lane < 16) cells[(size_t)g * 16 + lane] = make_unit<false>(buf[warp], lane);
            if (lane == 0) fac[g] = ldexpf(1.0f, -e);
        }
        __syncwarp();
    }
}

// Pass and slot of the pairs of token t (pairs tk .. tk + k - 1), as the
// grouping of CTA 0 places them: the rank of a pair among the pairs of its
// expert from counting the earlier pairs with that expert (the lists are in
// pair order); then warp j takes pair j: its pass is the passes of all
// experts below its expert (from the shared counts, one warp reduction) plus
// rank / pass_tok, its slot the remainder. pass[j] = -1 for an id outside
// [0, E) or an expert not served.
__device__ void pair_slots_cta(const int32_t *__restrict__ ids, int P, int E, int k, int t,
                               int pass_tok, int *pass, int *slot, const uint32_t *res) {
    __shared__ int32_t cnt[1024], rank[32], eid[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    cnt[tid] = 0;
    if (tid < k) {
        const int e = ids[(size_t)t * k + tid];
        eid[tid] = (e >= 0 && e < E && expert_served(res, e)) ? e : -1;
        rank[tid] = 0;
    }
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e >= 0 && e < E && expert_served(res, e)) {
            atomicAdd(&cnt[e], 1);
            for (int j = 0; j < k; ++j)
                if (e == eid[j] && p < t * k + j) atomicAdd(&rank[j], 1);
        }
    }
    __syncthreads();
    if (warp < k) {
        const int e = eid[warp];
        int before = 0;
        for (int u = lane; u < e; u += 32) before += (cnt[u] + pass_tok - 1) / pass_tok;
        before = (int)__reduce_add_sync(0xFFFFFFFFu, (unsigned)before);
        if (lane == 0) {
            pass[warp] = e < 0 ? -1 : before + rank[warp] / pass_tok;
            slot[warp] = e < 0 ? 0 : rank[warp] % pass_tok;
        }
    }
    __syncthreads();
}

// Splits token row t into units once (the tensor-map kernel's int4 form) and
// writes them to each of its pairs' (pass, slot) in the pass-packed layout:
// in block (pi * ns + g / 4) of kPackedStage bytes, the record (factor,
// offset_init) at float2 slot * 4 + g % 4 and the units at byte
// kPackedHead + slot * 1024 + (g % 4) * 256. With 32 warps each warp has one
// group, g0 + warp: xa / xb are its values lane and 32 + lane, loaded by the
// caller (0 past the row's last group).
__device__ void split_row_packed_cta(int K, int g0, int k, const int *pass, const int *slot,
                                     uint8_t *pk, float xa, float xb) {
    __shared__ float buf[32][64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, G = K / kGroup, ns = G / 4;
    const int g = g0 + warp;
    if (g < G) {
        const float a = xa, b = xb;
        const int e = split_exponent(warp_max(fmaxf(fabsf(a), fabsf(b))));
        const float mul = ldexpf(1.0f, e);
        buf[warp][lane] = a * mul;
        buf[warp][32 + lane] = b * mul;
        const float2 rec = make_float2(ldexpf(1.0f, -e), offset_init(warp_sum(a * mul + b * mul)));
        __syncwarp();
        const uint4 u = make_unit_s(buf[warp], lane & 15);
        for (int j = lane >> 4; j < k; j += 2) {
            if (pass[j] < 0) continue;
            uint8_t *blk = pk + ((size_t)pass[j] * ns + g / 4) * kPackedStage;
            reinterpret_cast<uint4 *>(blk + kPackedHead + slot[j] * 1024 + (g % 4) * 256)[lane & 15] = u;
            if ((lane & 15) == 0) reinterpret_cast<float2 *>(blk)[slot[j] * 4 + g % 4] = rec;
        }
    }
}

// CTA 0 groups the pairs; CTA 1 + t * C + c splits groups 32c .. 32c + 31
// of token row t of x (C = ceil(H / 2048): one group a warp), per row or into
// the pass-packed layout when bit 0 of `form` is set; bit 1 selects the
// tensor-map kernel's int4 form for the per-row split (the packed layout is
// always in that form). CTA 0 first clears zero[0 ..
// nzero) (the call's status word and split counters), which later kernels
// read only after waiting for this one. Launched with programmatic dependent
// launch, every CTA waits for the previous kernel (routing writes ids).
__global__ void __launch_bounds__(1024)
    k_group_split(const int32_t *__restrict__ ids, int P, int E, int32_t *offsets, int32_t *list,
                  int32_t *uexp, int32_t *n_used, int32_t *pass_ofs, int32_t *status,
                  const float *__restrict__ x, int H, uint4 *xcells, float *xfac, int pass_tok,
                  int k, int form, int32_t *zero, int nzero, const uint32_t *res,
                  uint8_t *served, const float *__restrict__ logits, int32_t *ids_out,
                  float *w_out, PlanArgs plan) {
    pdl_wait();
    pdl_trigger();
    const bool packed = form & 1;
    // a packed-split CTA (32 warps, one group each) requests its x values
    // first, so that their latency overlaps routing and the slot scan
    float xa = 0.f, xb = 0.f;
    if (packed && blockIdx.x > 0) {
        const int G = H / kGroup, C = (G + 31) / 32;
        const int t = (blockIdx.x - 1) / C, g = 32 * ((blockIdx.x - 1) % C) + (threadIdx.x >> 5);
        if (g < G) {
            const float *src = x + (size_t)t * H + g * kGroup + (threadIdx.x & 31);
            xa = src[0];
            xb = src[32];
        }
    }
    if (logits) {
        // routing folded in: every CTA routes all T = P / k tokens itself (a
        // warp a token, the moe_route_topk code) into shared memory, so no
        // CTA waits for another; CTA 0 writes ids and w out
        extern __shared__ float route_smem[];  // [32 warps][E] rows, then ids
        const int T = P / k, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        int32_t *rids = reinterpret_cast<int32_t *>(route_smem + 32 * E);
        for (int t = warp; t < T; t += 32) {
            int my_id;
            float my_w;
            route_warp(logits + (size_t)t * E, E, k, route_smem + warp * E, my_id, my_w);
            if (lane < k) {
                rids[t * k + lane] = my_id;
                if (blockIdx.x == 0) {
                    ids_out[t * k + lane] = my_id;
                    w_out[t * k + lane] = my_w;
                }
            }
        }
        __syncthreads();
        ids = rids;
    }
    if (blockIdx.x == 0) {
        if (zero) {
            for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
            __syncthreads();
        }
        group_cta(ids, P, E, offsets, list, uexp, n_used, pass_ofs, status, pass_tok, res, served,
                  &plan);
    } else {
        const int G = H / kGroup, C = (G + 31) / 32;
        const int t = (blockIdx.x - 1) / C, g0 = 32 * ((blockIdx.x - 1) % C);
        if (packed) {
            __shared__ int pass[32], slot[32];
            pair_slots_cta(ids, P, E, k, t, pass_tok, pass, slot, res);
            split_row_packed_cta(H, g0, k, pass, slot, reinterpret_cast<uint8_t *>(xcells), xa, xb);
        } else {
            split_row_cta(x + (size_t)t * H, H, g0, xcells + (size_t)t * G * 16,
                          xfac + (size_t)t * G * ((form & 2) ? 2 : 1), (form & 2) != 0);
        }
    }
}

// Pass offsets for externally grouped pairs (the staged entry points).
__global__ void __launch_bounds__(1024)
    k_passes(const int32_t *__restrict__ offsets, const int32_t *__restrict__ uexp,
             const int32_t *__restrict__ n_used, int32_t *pass_ofs) {
    __shared__ int32_t tot[96];
    __shared__ int32_t s_last;
    const int nu = *n_used;
    int carry = 0;
    for (int base = 0; base < nu; base += 1024) {
        const int u = base + threadIdx.x;
        int np = 0;
        if (u < nu) {
            const int e = uexp[u];
            np = (offsets[e + 1] - offsets[e] + kMaxTok - 1) / kMaxTok;
        }
        int ea, eb, ec;
        block_scan3(np, 0, 0, ea, eb, ec, tot);
        if (u < nu) pass_ofs[u] = carry + ea;
        if (threadIdx.x == 1023) s_last = ea + np;
        __syncthreads();
        carry += s_last;
        __syncthreads();
    }
    if (threadIdx.x == 0) pass_ofs[nu] = carry;
}

// ------------------------------------------------------------------ expert items
//
// An item of the gate+up / down kernels is (pass, row tile): a pass is up to
// kMaxTok pairs of one expert. Items are numbered pass-major, so a CTA's
// contiguous item range mostly stays on one expert and pass.

struct PassInfo {
    int e, beg, ntok;  // expert, first list index of the pass, pairs in the pass
};

__device__ __forceinline__ PassInfo pass_info(int pi, const int32_t *pass_ofs,
                                              const int32_t *uexp, const int32_t *offsets,
                                              int nu) {
    int lo = 0, hi = nu - 1;  // largest u with pass_ofs[u] <= pi
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pass_ofs[mid] <= pi) lo = mid; else hi = mid - 1;
    }
    PassInfo r;
    r.e = uexp[lo];
    const int pass = pi - pass_ofs[lo];
    const int b = offsets[r.e], cnt = offsets[r.e + 1] - b;
    r.beg = b + pass * kMaxTok;
    r.ntok = min(kMaxTok, cnt - pass * kMaxTok);
    return r;
}

constexpr int kMoeWarps = 16;  // one CTA of 16 warps per SM
constexpr int kMoeStages = 4;
constexpr int kMoeRing = kMoeStages * kStageBytes;
constexpr int kMoeBudget = 64 * 1024;
constexpr int kGuRows = 16 * kMoeWarps / 2;  // hidden units per gate+up item (128)
constexpr int kDnRows = 16 * kMoeWarps;      // output rows per down item (256)
constexpr int kEpiBytes = (2 * kGuRows * kMaxTok + kMoeWarps * 64) * 4;

struct MoeTile {
    const uint8_t *q;   // weight pool
    const float *s;     // scale pool
    const int32_t *pass_ofs, *uexp, *offsets;
    size_t eq, es;      // per-expert strides (bytes, floats)
    size_t rowBytes;
    int G, tiles, nu, i0, rows_per_warp_tile_base, nrows_total;
    int gate_up;        // 1: warps 0-3 gate rows, 4-7 up rows (I = nrows_total / 2)
    mutable int c_pi = -1, c_e = 0;

    __device__ __forceinline__ TileSrc operator()(int item, int wp) const {
        const int it = i0 + item;
        const int pi = it / tiles, tl = it - pi * tiles;
        if (pi != c_pi) {
            c_e = pass_info(pi, pass_ofs, uexp, offsets, nu).e;
            c_pi = pi;
        }
        int row;
        if (gate_up) {
            const int I = nrows_total / 2;
            const int half = kMoeWarps / 2;
            row = (wp < half) ? tl * kGuRows + 16 * wp : I + tl * kGuRows + 16 * (wp - half);
        } else {
            row = tl * kDnRows + 16 * wp;
        }
        int nrows = nrows_total - row;
        if (nrows <= 0) { row = nrows_total - 1; nrows = 1; }
        return TileSrc{q + c_e * eq + (size_t)row * rowBytes, s + c_e * es + (size_t)row * G,
                       rowBytes, nrows};
    }
};


__device__ __forceinline__ void cta_items(int total, int &i0, int &i1) {
    i0 = (int)((long long)blockIdx.x * total / gridDim.x);
    i1 = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
}

// ------------------------------------------------------------------ gate + up + SiLU

template <int NB, class WS>
__device__ __forceinline__ void gate_up_item(WS &ws, int &cslot, int jt, const PassInfo &pinf,
                                             bool reuse, const StageCells &stage, int I, int k,
                                             float *h, uint4 *hcells, float *hfac, uint8_t *smem,
                                             const int *s_pair) {
    constexpr int half = kMoeWarps / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int ntok = pinf.ntok;
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kMoeWarps * kMoeRing);
    float *fac = reinterpret_cast<float *>(smem + kMoeWarps * kMoeRing + kMoeBudget);
    float *gbuf = fac + kMoeBudget / 256;
    float *hbuf = gbuf + kGuRows * kMaxTok;
    float *wbuf = hbuf + kGuRows * kMaxTok;
    float acc[NB][2];
    run_item<NB, false>(ws, cslot, cells, fac, kMoeBudget, ntok, reuse, stage, acc);

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
    __syncthreads();
    const int j0 = jt * kGuRows;
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
                const size_t hb = (size_t)s_pair[s] * I + j0;
                if (j0 + lr < I) h[hb + lr] = h0;
                if (j0 + lr + 8 < I) h[hb + lr + 8] = h1;
            }
        }
    }
    __syncthreads();
    // fp16 hi/lo units of h for the down projection: groups 2jt, 2jt+1 of h.
    const int Gd = I / kGroup;
    for (int idx = warp; idx < ntok * 2; idx += kMoeWarps) {
        const int s = idx >> 1, gg = idx & 1;
        const int gd = jt * 2 + gg;
        if (gd < Gd) {
            const float a = hbuf[(gg * 64 + lane) * kMaxTok + s];
            const float b = hbuf[(gg * 64 + 32 + lane) * kMaxTok + s];
            const int e = split_exponent(warp_max(fmaxf(fabsf(a), fabsf(b))));
            const float mul = ldexpf(1.0f, e);
            wbuf[warp * 64 + lane] = a * mul;
            wbuf[warp * 64 + 32 + lane] = b * mul;
            __syncwarp();
            const size_t cb = (size_t)s_pair[s] * Gd + gd;
            if (lane < 16) hcells[cb * 16 + lane] = make_unit<false>(wbuf + warp * 64, lane);
            if (lane == 0) hfac[cb] = ldexpf(1.0f, -e);
            __syncwarp();
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(32 * kMoeWarps, 1)
    k_gate_up(MoeDims m, const uint4 *__restrict__ xcells, const float *__restrict__ xfac, int k,
              const int32_t *__restrict__ offsets, const int32_t *__restrict__ list,
              const int32_t *__restrict__ uexp, const int32_t *__restrict__ n_used,
              const int32_t *__restrict__ pass_ofs, float *__restrict__ h,
              uint4 *__restrict__ hcells, float *__restrict__ hfac) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_rows[kMaxTok], s_pair[kMaxTok];
    pdl_wait();  // grouping and x cells come from the previous kernel
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = m.H, I = m.I, G = H / kGroup;
    const int nu = *n_used;
    if (nu == 0) return;
    const int tiles = (I + kGuRows - 1) / kGuRows;
    const int total = pass_ofs[nu] * tiles;
    int i0, i1;
    cta_items(total, i0, i1);
    if (i0 >= i1) return;
    MoeTile tile{m.gu_q, m.gu_s, pass_ofs, uexp, offsets, (size_t)2 * I * (H / 2),
                 (size_t)2 * I * G, (size_t)H / 2, G, tiles, nu, i0, 0, 2 * I, 1};
    WarpStream<false, kMoeStages, MoeTile> ws;
    ws.init(smem + warp * kMoeRing, tile, G, i1 - i0, warp, lane);
    ws.prologue();
    int cslot = 0;

    int cur_pi = -1;
    PassInfo pinf{};
    for (int it = 0; it < i1 - i0; ++it) {
        const int gi = i0 + it, pi = gi / tiles, jt = gi - pi * tiles;
        bool reuse = pi == cur_pi;
        if (!reuse) {
            pinf = pass_info(pi, pass_ofs, uexp, offsets, nu);
            cur_pi = pi;
            __syncthreads();  // previous item's epilogue is done with s_pair
            if (threadIdx.x < pinf.ntok) {
                const int p = list[pinf.beg + threadIdx.x];
                s_pair[threadIdx.x] = p;
                s_rows[threadIdx.x] = p / k;
            }
        }
        const StageCells stage{xcells, xfac, s_rows, pinf.ntok, G};
        if (pinf.ntok <= 4)
            gate_up_item<1>(ws, cslot, jt, pinf, reuse, stage, I, k, h, hcells, hfac, smem, s_pair);
        else
            gate_up_item<2>(ws, cslot, jt, pinf, reuse, stage, I, k, h, hcells, hfac, smem, s_pair);
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------ down

template <int NB, class WS>
__device__ __forceinline__ void down_item(WS &ws, int &cslot, int tl, const PassInfo &pinf,
                                          bool reuse, const StageCells &stage, int H, float *y,
                                          uint8_t *smem, const int *s_pair) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    uint4 *cells = reinterpret_cast<uint4 *>(smem + kMoeWarps * kMoeRing);
    float *fac = reinterpret_cast<float *>(smem + kMoeWarps * kMoeRing + kMoeBudget);
    float acc[NB][2];
    run_item<NB, false>(ws, cslot, cells, fac, kMoeBudget, pinf.ntok, reuse, stage, acc);
    const int row0 = tl * kDnRows + 16 * warp;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int s = 4 * nb + q;
        if (s < pinf.ntok) {
            const size_t yb = (size_t)s_pair[s] * H;
            if (row0 + gid < H) y[yb + row0 + gid] = acc[nb][0];
            if (row0 + gid + 8 < H) y[yb + row0 + gid + 8] = acc[nb][1];
        }
    }
}

__global__ void __launch_bounds__(32 * kMoeWarps, 1)
    k_down(MoeDims m, const uint4 *__restrict__ hcells, const float *__restrict__ hfac,
           const int32_t *__restrict__ offsets, const int32_t *__restrict__ list,
           const int32_t *__restrict__ uexp, const int32_t *__restrict__ n_used,
           const int32_t *__restrict__ pass_ofs, float *__restrict__ y) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int s_pair[kMaxTok];
    // The grouping was complete before the previous kernel started its main
    // work, so the item map and the weights can be read before the wait.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = m.H, I = m.I, G = I / kGroup;
    const int nu = *n_used;
    if (nu == 0) { pdl_wait(); pdl_trigger(); return; }
    const int tiles = (H + kDnRows - 1) / kDnRows;
    const int total = pass_ofs[nu] * tiles;
    int i0, i1;
    cta_items(total, i0, i1);
    MoeTile tile{m.dn_q, m.dn_s, pass_ofs, uexp, offsets, (size_t)H * (I / 2), (size_t)H * G,
                 (size_t)I / 2, G, tiles, nu, i0, 0, H, 0};
    WarpStream<false, kMoeStages, MoeTile> ws;
    ws.init(smem + warp * kMoeRing, tile, G, i1 - i0, warp, lane);
    ws.prologue();
    int cslot = 0;
    pdl_wait();  // h cells come from the gate+up kernel
    pdl_trigger();

    int cur_pi = -1;
    PassInfo pinf{};
    for (int it = 0; it < i1 - i0; ++it) {
        const int gi = i0 + it, pi = gi / tiles, tl = gi - pi * tiles;
        const bool reuse = pi == cur_pi;
        if (!reuse) {
            pinf = pass_info(pi, pass_ofs, uexp, offsets, nu);
            cur_pi = pi;
            __syncthreads();
            if (threadIdx.x < pinf.ntok) s_pair[threadIdx.x] = list[pinf.beg + threadIdx.x];
        }
        const StageCells stage{hcells, hfac, s_pair, pinf.ntok, G};
        if (pinf.ntok <= 4)
            down_item<1>(ws, cslot, tl, pinf, reuse, stage, H, y, smem, s_pair);
        else
            down_item<2>(ws, cslot, tl, pinf, reuse, stage, H, y, smem, s_pair);
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------ combine

// out[t] = sum_j w[t][j] * y[t*k + j] over the served slots, j in order (one
// fused multiply-add each). V = 4: four consecutive outputs a thread with
// 16-byte loads (H a multiple of 4, out 16-byte aligned), so the k loads of
// a thread are in flight together.
template <int V>
__global__ void __launch_bounds__(256)
    k_combine(const float *__restrict__ y, const int32_t *__restrict__ ids,
              const float *__restrict__ w, int k, int E, int H, float *__restrict__ out,
              const uint32_t *res, int early) {
    // the token's pairs: weight, and whether the pair is combined (k <= 1024)
    __shared__ float s_w[1024];
    __shared__ unsigned char s_on[1024];
    const int t = blockIdx.y;
    auto stage = [&]() {
        for (int j = threadIdx.x; j < k; j += blockDim.x) {
            const int p = t * k + j;
            const int e = ids[p];
            const bool on = e >= 0 && e < E && expert_served(res, e);
            s_on[j] = on ? 1 : 0;
            s_w[j] = on ? w[p] : 0.0f;
        }
    };
    // ids, w and res are read before the wait when they predate the previous
    // kernel (early), so that only y's loads follow it
    if (early) stage();
    pdl_wait();
    pdl_trigger();
    if (!early) stage();
    __syncthreads();
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (i >= H) return;
    float o[V];
#pragma unroll
    for (int v = 0; v < V; ++v) o[v] = 0.0f;
    // the y rows of all pairs are in bounds: load them independently (the
    // skipped pairs' values are never used), add in pair order
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        const float *yr = y + (size_t)(t * k + j) * H + i;
        const float wp = s_w[j];
        const bool on = s_on[j] != 0;
        if (V == 4) {
            const float4 v4 = *reinterpret_cast<const float4 *>(yr);
            if (on) {
                o[0] = fmaf(wp, v4.x, o[0]);
                o[1] = fmaf(wp, v4.y, o[1]);
                o[2] = fmaf(wp, v4.z, o[2]);
                o[3] = fmaf(wp, v4.w, o[3]);
            }
        } else {
            const float v1 = yr[0];
            if (on) o[0] = fmaf(wp, v1, o[0]);
        }
    }
    if (V == 4)
        *reinterpret_cast<float4 *>(out + (size_t)t * H + i) = make_float4(o[0], o[1], o[2], o[3]);
    else
        out[(size_t)t * H + i] = o[0];
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

size_t moe_smem() { return engine_smem(kMoeWarps, kMoeStages, kMoeBudget, kEpiBytes); }

int moe_grid(void (*k)(MoeDims, const uint4 *, const float *, int, const int32_t *,
                       const int32_t *, const int32_t *, const int32_t *, const int32_t *,
                       float *, uint4 *, float *)) {
    return sm_count() * max_ctas_per_sm(k, 32 * kMoeWarps, moe_smem());
}

}  // namespace

// ------------------------------------------------------------------ launchers

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    return launch(k_route, dim3((T + kRouteWarps - 1) / kRouteWarps), dim3(32 * kRouteWarps), 0,
                  st, true, logits, T, E, k, ids, w);
}

cudaError_t launch_group(const int32_t *ids, int P, int E, int32_t *offsets, int32_t *list,
                         int32_t *uexp, int32_t *n_used, int32_t *status, cudaStream_t st) {
    const size_t smem = group_smem_bytes(E);
    cudaError_t e = set_smem(k_group_split, std::max(smem, (size_t)49 * 1024));
    if (e != cudaSuccess) return e;
    return launch(k_group_split, dim3(1), dim3(1024), smem, st, false, ids, P, E, offsets, list, uexp,
                  n_used, (int32_t *)nullptr, status, (const float *)nullptr, 64,
                  (uint4 *)nullptr, (float *)nullptr, (int)kMaxTok, 1, 0, (int32_t *)nullptr, 0,
                  (const uint32_t *)nullptr, (uint8_t *)nullptr, (const float *)nullptr,
                  (int32_t *)nullptr, (float *)nullptr, PlanArgs{});
}

cudaError_t launch_group_split(const int32_t *ids, int T, int k, int E, int32_t *offsets,
                               int32_t *list, int32_t *uexp, int32_t *n_used, int32_t *pass_ofs,
                               int32_t *status, const float *x, int H, void *xcells, float *xfac,
                               cudaStream_t st, int pass_tok, bool packed, int32_t *zero,
                               int nzero, bool pdl, const uint32_t *res, uint8_t *served,
                               const float *logits, int32_t *ids_out, float *w_out, bool sub,
                               const PlanArgs *plan) {
    const int C = (H / kGroup + 31) / 32;  // CTAs per token row
    // dynamic shared memory: the routing rows and ids, or the grouping's
    // per-warp expert counts, whichever is larger (the counts reuse the
    // routing rows after routing)
    const size_t smem = std::max(logits ? route_smem_bytes(T, E, k) : 0, group_smem_bytes(E));
    {
        // with the static shared memory, even a small dynamic part needs the
        // opt-in (set_smem only opts in above 48 KB)
        cudaError_t e = set_smem(k_group_split, std::max(smem, (size_t)49 * 1024));
        if (e != cudaSuccess) return e;
    }
    return launch(k_group_split, dim3(x ? 1 + T * C : 1), dim3(1024), smem, st, pdl, ids, T * k,
                  E, offsets, list, uexp, n_used, pass_ofs, status, x, H,
                  static_cast<uint4 *>(xcells), xfac, pass_tok, k,
                  (packed ? 1 : 0) | ((packed || sub) ? 2 : 0), zero, nzero, res, served, logits,
                  ids_out, w_out, plan ? *plan : PlanArgs{});
}

size_t group_smem_bytes(int E) { return (size_t)32 * E * sizeof(int32_t); }

size_t route_smem_bytes(int T, int E, int k) {
    return (size_t)32 * E * sizeof(float) + (size_t)T * k * sizeof(int32_t);
}

cudaError_t launch_passes(const int32_t *offsets, const int32_t *uexp, const int32_t *n_used,
                          int32_t *pass_ofs, cudaStream_t st, bool pdl) {
    return launch(k_passes, dim3(1), dim3(1024), 0, st, pdl, offsets, uexp, n_used, pass_ofs);
}

cudaError_t launch_gate_up(const MoeDims &m, const void *xcells, const float *xfac, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hcells,
                           float *hfac, cudaStream_t st) {
    const size_t smem = moe_smem();
    cudaError_t e = set_smem(k_gate_up, smem);
    if (e != cudaSuccess) return e;
    return launch(k_gate_up, dim3(moe_grid(k_gate_up)), dim3(32 * kMoeWarps), smem, st, true, m,
                  static_cast<const uint4 *>(xcells), xfac, k, offsets, list, uexp, n_used,
                  pass_ofs, h, static_cast<uint4 *>(hcells), hfac);
}

cudaError_t launch_down(const MoeDims &m, const void *hcells, const float *hfac,
                        const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                        const int32_t *n_used, const int32_t *pass_ofs, float *y, cudaStream_t st) {
    const size_t smem = moe_smem();
    cudaError_t e = set_smem(k_down, smem);
    if (e != cudaSuccess) return e;
    const int grid = sm_count() * max_ctas_per_sm(k_down, 32 * kMoeWarps, smem);
    return launch(k_down, dim3(grid), dim3(32 * kMoeWarps), smem, st, true, m,
                  static_cast<const uint4 *>(hcells), hfac, offsets, list, uexp, n_used, pass_ofs,
                  y);
}

cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E,
                           int H, float *out, cudaStream_t st, bool pdl, const uint32_t *res,
                           bool early) {
    if (T == 0) return cudaSuccess;
    const int ea = early && pdl ? 1 : 0;
    if (H % 4 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(y) & 15) == 0)
        return launch(k_combine<4>, dim3((H / 4 + 255) / 256, T), dim3(256), 0, st, pdl, y, ids, w,
                      k, E, H, out, res, ea);
    return launch(k_combine<1>, dim3((H + 255) / 256, T), dim3(256), 0, st, pdl, y, ids, w, k, E, H,
                  out, res, ea);
}

MoeWorkspace moe_ws_layout(int E, int H, int I, int T, int k) {
    MoeWorkspace L{};
    const size_t P = (size_t)T * k;
    size_t o = 0;
    L.status = o;
    L.sk_cnt = o + 4;
    L.status_bytes = 4 + 4 * 2 * (size_t)kSkMaxCtas;
    o = align256(o + L.status_bytes);
    L.offsets = o; o = align256(o + 4 * (size_t)(E + 1));
    L.list = o; o = align256(o + 4 * P);
    L.uexp = o; o = align256(o + 4 * (size_t)E);
    L.n_used = o; o = align256(o + 8);  // n_used, then the pass count
    L.pass_ofs = o; o = align256(o + 4 * (size_t)(E + 1));
    L.xcells = o; o = align256(o + 4 * (size_t)T * H);
    L.xfac = o; o = align256(o + 8 * (size_t)T * (H / 64));  // up to 8 bytes a group
    L.h = o; o = align256(o + 4 * P * I);
    L.hcells = o; o = align256(o + 4 * P * I);
    L.hfac = o; o = align256(o + 8 * P * (I / 64));
    L.y = o; o = align256(o + 4 * P * H);
    L.sk_part = o; o = align256(o + 4 * (size_t)kSkMaxCtas * kSkPartFloats);
    // a pass holds up to kMaxTok pairs of one expert: at most P / kMaxTok + min(E, P) passes
    const size_t pm = std::min(P, (P + kMaxTok - 1) / kMaxTok + std::min((size_t)E, P));
    L.pmax = (int)pm;
    const size_t sh = (size_t)H / (4 * kGroup), si = (size_t)I / (4 * kGroup);  // stages
    L.xpk = o; o = align256(o + pm * sh * kPackedStage);
    L.hpk = o; o = align256(o + pm * si * kPackedStage);
    L.ptab = o; o = align256(o + 16 * pm);
    L.plan = o; o = align256(o + 16 * 2 * ((size_t)kSkMaxCtas + 1));
    L.total = o;
    return L;
}

PrefillWorkspace prefill_ws_layout(int E, int H, int I, int T, int k) {
    PrefillWorkspace L{};
    const size_t P = (size_t)T * k;
    size_t o = 0;
    L.status = o; o = align256(o + 4);
    L.offsets = o; o = align256(o + 4 * (size_t)(E + 1));
    L.list = o; o = align256(o + 4 * P);
    L.uexp = o; o = align256(o + 4 * (size_t)E);
    L.n_used = o; o = align256(o + 8);  // n_used, then the pass count
    L.pass_ofs = o; o = align256(o + 4 * (size_t)(E + 1));
    L.h = o; o = align256(o + 2 * P * I);
    L.y = o; o = align256(o + 4 * P * H);
    // packed B operands of the tensor-map path: a pass holds up to 64 pairs of
    // one expert, so there are at most P / 64 + min(E, P) passes
    const size_t pm = std::min(P, (P + 63) / 64 + std::min((size_t)E, P));
    L.pmax = (int)pm;
    L.ptab = o; o = align256(o + 16 * pm);
    L.xp = o; o = align256(o + pm * (size_t)(H / 64) * 8192);
    L.hp = o; o = align256(o + pm * (size_t)(I / 64) * 8192);
    L.total = o;
    return L;
}

}  // namespace qmv
