// qmv_moe_one.cu - the expert FFN of one decode token in a single launch.
//
// Math (colibri PR #418, "qmatmul_gate_up.comp + coli_vk_gate_up",
// "coli_vk_expert_group", "grouped scales in the Vulkan kernels"): for each
// routed expert e_p with weight w_p, h_p = SiLU(G_p x) * (U_p x) and
// out = sum_p w_p * D_p h_p; per 64-group the exact products (nibble - 8) * v
// are summed and the group scale is applied in fp32 to that partial sum.
// Operands are exact fp16 weights and fp16 hi + lo activations with one
// power-of-two factor per 64-group (the fragment layout of qmv_device.cuh),
// multiplied by warp MMAs with fp32 accumulation.
//
// With one token every expert is read once and the whole layer is only a
// few MB, so the separate grouping, gate+up, down and combine launches cost
// more than the bytes. Here one cooperative launch (one CTA per SM) does it:
//   * at start, a producer warp requests the CTA's whole share of weights
//     and scales by bulk copy: gate+up tiles t = CTA, CTA + grid, ... (a tile
//     is 8 gate rows and the 8 up rows of the same hidden units; one
//     transaction barrier each) and down row tiles (16 output rows of every
//     routed expert);
//   * while they land, the 8 compute warps split x into activation units;
//   * gate+up, tile by tile as each lands: the 8 warps split the tile's
//     64-groups, their partial sums are added in warp order and one thread
//     per hidden unit writes h;
//   * one grid-wide barrier (every h written);
//   * down: warp p splits expert p's h into units and computes its 16-row
//     tile; out = sum_p w_p y_p is added in expert order.
// Every result is written by exactly one thread after a fixed-order sum, so
// the output does not depend on timing.
//
// Waits are bounded: a copy or barrier wait that runs out sets bit 1 of the
// status word (the outputs are then not valid) and the kernel goes on. CTA 0
// clears the status word at the start, so a call needs no memset first. An
// expert id outside [0, E) sets bit 0 and contributes nothing; so does, with
// no error, an expert outside the call's residency bitmap.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "qmv_internal.h"
#include "qmv_launch.cuh"
#include "qmv_route.cuh"
#include "qmv_rows.cuh"
#include "tc05.cuh"

namespace qmv {

namespace {

constexpr int kOWarps = 8;                  // compute warps; warp kOWarps issues the copies
constexpr int kOThreads = 32 * (kOWarps + 1);
constexpr int kOMaxT1 = 64;                 // gate+up tiles per CTA (one barrier each)
constexpr uint32_t kOWait = 1u << 24;
constexpr int kOMaxK = 32;              // routed experts per token
constexpr int kOSmemMax = 220 * 1024;   // dynamic shared memory budget

struct OneArgs {
    // the weight pools as 3-D tensor maps (128 bytes, row, 128-byte chunk of
    // the row), boxes of 8 (gate+up) / 16 (down) whole rows, 128-byte
    // swizzle: one copy per box, and a row's 16-byte chunks land XOR-ed with
    // the row index, so a warp's 8-byte loads of 8 rows hit distinct banks
    CUtensorMap map_gu;
    CUtensorMap map_dn;
    const uint8_t *gu_q;   // gate+up weights [E][2I][H/2]
    const float *gu_s;     // their scales [E][2I][H/64]
    const uint8_t *dn_q;   // down weights [E][H][I/2]
    const float *dn_s;     // their scales [E][H][I/64]
    int E, H, I, k;
    const float *x;        // [H]
    const int32_t *ids;    // [k]
    const float *w;        // [k]
    float *h;              // [k][I] (workspace)
    float *out;            // [H]
    int32_t *status;       // cleared by CTA 0 at the start
    const uint32_t *res;   // served experts' bitmap, or null for all
    uint8_t *served;       // [k]: 1 = pair computed (CTA 0 writes it), or null
    const float *logits;   // [E]: route in-kernel (ids / w then outputs), or null
    int32_t *ids_out;      // routed ids [k] (CTA 0 writes them) when logits != null
    float *w_out;          // their weights [k]
    // shared-memory layout (byte offsets from the aligned base)
    int n1, n2;            // gate+up tiles, down row tiles per CTA (at most)
    int o_xu, o_xf, o_w1, o_s1, o_w2, o_s2, o_hu, o_hf, o_red, o_scr, o_lg;
};

struct OneShared {
    uint64_t mb1[kOMaxT1]; // gate+up tile i landed
    uint64_t mb2;          // down copies landed
    int ids[kOMaxK];
    float w[kOMaxK];
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc05::smem_addr(mbar))
        : "memory");
}

__device__ __forceinline__ void tma_g2s3(uint32_t dst, const CUtensorMap *map, int c1,
                                         uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(0), "r"(tc05::smem_addr(mbar))
        : "memory");
}

// Byte o of row r of a box of R rows loaded through a swizzled map (R a
// multiple of 8, box base 1024-byte aligned): the box is [chunk][row][128 B]
// with the 16-byte units of each 128-byte line XOR-ed with the row mod 8.
__device__ __forceinline__ const uint8_t *swz(const uint8_t *box, int R, int r, int o) {
    return box + (((o >> 7) * R + r) << 7) + ((((o >> 4) & 7) ^ (r & 7)) << 4) + (o & 15);
}

__device__ __forceinline__ void expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     tc05::smem_addr(mbar)),
                 "r"(bytes)
                 : "memory");
}

// The compute warps only (the producer warp does not take part).
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kOWarps) : "memory");
}

// Grid barrier count of this kernel on this device: zero when the library
// is loaded and never reset. Launches are cooperative, of one CTA per SM,
// and a launch takes no ticket before every CTA of the launch before it
// has taken its own (a CTA of the next launch starts only where one of this
// launch has exited, after the barrier), so launch n holds tickets
// [n * grid, (n + 1) * grid) and its CTAs wait for the count to reach
// (n + 1) * grid. No clearing between calls: no memset node in the graph.
__device__ unsigned long long g_one_bar;

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// All CTAs of the (cooperative) grid: every write before it is visible to
// every read after it. Bounded; returns false if it gave up.
__device__ __forceinline__ bool grid_barrier() {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        unsigned long long t;  // release: this CTA's writes before the barrier
        asm volatile("atom.add.release.gpu.u64 %0, [%1], 1;" : "=l"(t) : "l"(&g_one_bar) : "memory");
        const unsigned long long target = (t / gridDim.x + 1) * gridDim.x;
        uint32_t i = 0;
        while (ld_acquire64(&g_one_bar) < target) {
            if (++i == kOWait) {
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
    }
    __syncthreads();
    return ok != 0;
}

// Groups c = w, w + nw, ... < n of a row-major source (64 floats per group
// at src + 64 c, read through L2) -> activation units and factors in shared
// memory; w / nw: this warp's index among the nw warps that share the work.
// A warp takes up to 8 groups at once (loads, maxima and conversions of the 8
// interleave), with 64 floats of scratch per group.
__device__ __forceinline__ void split_groups(const float *src, int n, uint4 *units, float *fac,
                                             float *scratch, int w, int nw) {
    const int lane = threadIdx.x & 31;
    for (int c0 = w; c0 < n; c0 += 8 * nw) {
        float va[8], vb[8], m[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i * nw;
            va[i] = c < n ? __ldcg(src + (size_t)c * kGroup + lane) : 0.f;
            vb[i] = c < n ? __ldcg(src + (size_t)c * kGroup + 32 + lane) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(va[i]), fabsf(vb[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xffffffffu, m[i], o));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i * nw;
            const int e = split_exponent(m[i]);  // |e| <= 126: 2^e is a normal float
            scratch[i * 64 + lane] = va[i] * __int_as_float((127 + e) << 23);
            scratch[i * 64 + 32 + lane] = vb[i] * __int_as_float((127 + e) << 23);
            if (lane == 0 && c < n) fac[c] = __int_as_float((127 - e) << 23);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = 2 * j + (lane >> 4), c = c0 + i * nw;
            if (c < n) units[c * 16 + (lane & 15)] = make_unit<false>(scratch + i * 64, lane & 15);
        }
        __syncwarp();
    }
}

// Rows src[p][n * 64] (p < rows_n, read through L2: other CTAs wrote them)
// -> units[p][g][16] and factors fac[p][g] in shared memory, by the nt
// threads t < nt, four threads per 64-group. Thread quarter q of a group
// holds values 16q .. 16q+15, exactly the values of the group's units
// (mh, q, part), so each thread builds its four units from its own values;
// the group's max |v| takes two shuffles. Same arithmetic as split_groups.
__device__ __forceinline__ void split_rows_quad(const float *src, int rows_n, int n, uint4 *units,
                                                float *fac, int t, int nt) {
    const int nq = rows_n * n * 4;
    for (int base = 0; base < nq; base += nt) {  // uniform trip count: shuffles below
        const int idx = base + t;
        const bool valid = idx < nq;
        const int c = valid ? idx >> 2 : 0, q = idx & 3;  // c = p * n + g
        float v[16];
        const float4 *s4 = reinterpret_cast<const float4 *>(src + (size_t)c * kGroup + 16 * q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 f = valid ? __ldcg(s4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
        }
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
        const int e = split_exponent(am);  // |e| <= 126: 2^e is a normal float
        const float mul = __int_as_float((127 + e) << 23);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= mul;
        if (valid) {
#pragma unroll
            for (int mh = 0; mh < 2; ++mh)
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    uint32_t r[4];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        int k0, k1, k2, k3;
                        frag_ks<false>(2 * mh + i, 0, k0, k1, k2, k3);  // local to the quad
                        r[2 * i] = pack_half2(split_part(v[k0], part), split_part(v[k1], part));
                        r[2 * i + 1] = pack_half2(split_part(v[k2], part), split_part(v[k3], part));
                    }
                    units[c * 16 + (mh * 4 + q) * 2 + part] = make_uint4(r[0], r[1], r[2], r[3]);
                }
            if (q == 0) fac[c] = __int_as_float((127 - e) << 23);
        }
    }
}

// Lane (gid, q) of a warp: MMA over one 64-group of a 16-row tile in shared
// memory (row gid: row r0 of box b0 with R0 rows; row gid + 8: row r8 of box
// b8 with R8 rows; the group at byte 32 g of a row) against that group's
// activation units bu (one token: every B column is token 0). Adds
// scale * factor * (hi + lo) of rows gid / gid + 8 to c0 / c8 (meaningful in
// lanes q == 0).
__device__ __forceinline__ void tile_group_one(const uint8_t *b0, int R0, int r0, const uint8_t *b8,
                                               int R8, int r8, int g, const uint4 (&bu)[1][2],
                                               float f, float s0, float s8, float &c0, float &c8) {
    const int lane = threadIdx.x & 31, q = lane & 3;
    const int o = g * 32 + 8 * q;
    const uint2 w0 = *reinterpret_cast<const uint2 *>(swz(b0, R0, r0, o));
    const uint2 w8 = *reinterpret_cast<const uint2 *>(swz(b8, R8, r8, o));
    float d[1][4];
    tile_group_int4<1>(w0, w8, bu, d);
    c0 = fmaf(s0 * f, d[0][0] + d[0][1], c0);
    c8 = fmaf(s8 * f, d[0][2] + d[0][3], c8);
}

__device__ __forceinline__ void load_units(const uint4 *u, uint4 (&bu)[1][2]) {
    const int lane = threadIdx.x & 31, q = lane & 3, part = (lane >> 2) & 1;
    bu[0][0] = u[q * 2 + part];
    bu[0][1] = u[(4 + q) * 2 + part];
}

__global__ void __launch_bounds__(kOThreads, 1) k_moe_one(const __grid_constant__ OneArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ OneShared sh;
    uint8_t *base = smem_raw + ((1024u - (tc05::smem_addr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int H = a.H, I = a.I, k = a.k;
    const int GH = H / kGroup, GI = I / kGroup;
    const int tiles1 = k * (I / 8), tiles2 = H / 16;
    const int b = blockIdx.x, grid = gridDim.x;
    const int rb1 = H / 2, rb2 = I / 2;                        // row bytes
    const uint32_t t1w = 16u * rb1, t1s = 16u * GH * 4;       // gate+up tile: rows, scales
    const uint32_t e2w = 16u * rb2, e2s = 16u * GI * 4;       // down rows of one expert
    const int n1 = b < tiles1 ? (tiles1 - b + grid - 1) / grid : 0;
    const int n2 = b < tiles2 ? (tiles2 - b + grid - 1) / grid : 0;

    // the call's status word: cleared here, before any bit of this call is set
    // (bit 0 by CTA 0 below, bit 1 only after the grid barrier)
    if (b == 0 && threadIdx.x == 0) *a.status = 0;
    if (a.logits && warp == 0) {
        // every CTA routes the token itself (the same top-k as moe_route_topk)
        int my_id;
        float my_w;
        route_warp(a.logits, a.E, k, reinterpret_cast<float *>(base + a.o_lg), my_id, my_w);
        if (lane < k) {
            sh.ids[lane] = my_id;
            sh.w[lane] = my_w;
            if (b == 0) {
                a.ids_out[lane] = my_id;
                a.w_out[lane] = my_w;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < k) {
        int e = a.logits ? sh.ids[threadIdx.x] : a.ids[threadIdx.x];
        if (e < 0 || e >= a.E) {
            if (b == 0) atomicOr(a.status, 1);
            e = -1;
        } else if (!expert_served(a.res, e)) {
            e = -1;  // not resident: left to the caller, no error
        }
        sh.ids[threadIdx.x] = e;
        if (!a.logits) sh.w[threadIdx.x] = a.w[threadIdx.x];
        if (b == 0 && a.served) a.served[threadIdx.x] = e >= 0 ? 1 : 0;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < n1; ++i) tc05::mbar_init(&sh.mb1[i], 1);
        tc05::mbar_init(&sh.mb2, 1);
        tc05::fence_mbar_init();
    }
    __syncthreads();

    bool timed_out = false;
    if (warp == kOWarps) {
        // ---- producer: every copy of the CTA's share, requested at once (a
        // few large bulk copies: the copy engine takes commands one by one):
        // per gate+up tile its 8 gate rows, its 8 up rows and their scales,
        // then per down row tile and expert 16 rows and their scales
        if (lane == 0) {
            uint32_t bytes2 = 0;
            for (int p = 0; p < k; ++p)
                if (sh.ids[p] >= 0) bytes2 += (uint32_t)n2 * (e2w + e2s);
            expect_tx(&sh.mb2, bytes2);
            for (int i = 0; i < n1; ++i) {
                const int t = b + i * grid, p = t / (I / 8), u0 = 8 * (t % (I / 8)), e = sh.ids[p];
                expect_tx(&sh.mb1[i], e >= 0 ? t1w + t1s : 0u);
                if (e < 0) continue;
                const uint32_t dw = tc05::smem_addr(base + a.o_w1 + i * t1w);
                const uint32_t ds = tc05::smem_addr(base + a.o_s1 + i * t1s);
                const size_t rg = (size_t)e * 2 * I + u0, ru = rg + I;   // gate / up rows
                tma_g2s3(dw, &a.map_gu, (int)rg, &sh.mb1[i]);
                tma_g2s3(dw + 8u * rb1, &a.map_gu, (int)ru, &sh.mb1[i]);
                bulk_g2s(ds, a.gu_s + rg * GH, 8u * GH * 4, &sh.mb1[i]);
                bulk_g2s(ds + 8u * GH * 4, a.gu_s + ru * GH, 8u * GH * 4, &sh.mb1[i]);
            }
            for (int i = 0; i < n2; ++i)
                for (int p = 0; p < k; ++p) {
                    const int e = sh.ids[p];
                    if (e < 0) continue;
                    const int slot = i * k + p;
                    const size_t r0 = (size_t)e * H + 16 * (b + i * grid);
                    tma_g2s3(tc05::smem_addr(base + a.o_w2 + slot * e2w), &a.map_dn, (int)r0,
                             &sh.mb2);
                    bulk_g2s(tc05::smem_addr(base + a.o_s2 + slot * e2s), a.dn_s + r0 * GI,
                             16u * GI * 4, &sh.mb2);
                }
        }
        __syncwarp();
    } else {
        // ---- x -> activation units (each CTA its own copy)
        uint4 *xu = reinterpret_cast<uint4 *>(base + a.o_xu);
        float *xf = reinterpret_cast<float *>(base + a.o_xf);
        float *red = reinterpret_cast<float *>(base + a.o_red);
        float *scratch = reinterpret_cast<float *>(base + a.o_scr) + warp * 8 * 64;
        split_groups(a.x, GH, xu, xf, scratch, warp, kOWarps);
        compute_sync();

        // ---- gate+up, tile by tile as each lands: warp w takes groups w,
        // w + 8, ... of the tile; the partial sums red[tile][warp][16] are then
        // added in warp order
        for (int i = 0; i < n1; ++i) {
            if (!tc05::mbar_wait(&sh.mb1[i], 0, kOWait)) timed_out = true;
            const uint8_t *rows = base + a.o_w1 + i * t1w;   // gate box, then up box
            const float *sc = reinterpret_cast<const float *>(base + a.o_s1 + i * t1s);
            float c0 = 0.f, c8 = 0.f;
            for (int g = warp; g < GH; g += kOWarps) {
                uint4 bu[1][2];
                load_units(xu + g * 16, bu);
                tile_group_one(rows, 8, gid, rows + 8 * rb1, 8, gid, g, bu, xf[g],
                               sc[gid * GH + g], sc[(gid + 8) * GH + g], c0, c8);
            }
            if (q == 0) {
                red[(i * kOWarps + warp) * 16 + gid] = c0;
                red[(i * kOWarps + warp) * 16 + 8 + gid] = c8;
            }
        }
        compute_sync();
        for (int c = threadIdx.x; c < n1 * 8; c += 32 * kOWarps) {
            const int i = c >> 3, u = c & 7, t = b + i * grid;
            const int p = t / (I / 8), u0 = 8 * (t % (I / 8));
            float gv = 0.f, uv = 0.f;
            for (int w = 0; w < kOWarps; ++w) {
                gv += red[(i * kOWarps + w) * 16 + u];
                uv += red[(i * kOWarps + w) * 16 + 8 + u];
            }
            const float hv = sh.ids[p] >= 0 ? gv / (1.0f + expf(-gv)) * uv : 0.f;
            a.h[(size_t)p * I + u0 + u] = hv;
        }
    }

    if (!grid_barrier()) timed_out = true;

    if (warp < kOWarps) {
        // ---- h -> activation units (each CTA its own copy), then down + combine
        uint4 *hu = reinterpret_cast<uint4 *>(base + a.o_hu);
        float *hf = reinterpret_cast<float *>(base + a.o_hf);
        float *red = reinterpret_cast<float *>(base + a.o_red);
        // all compute threads split h (k rows of I), four threads a group
        split_rows_quad(a.h, k, GI, hu, hf, threadIdx.x, 32 * kOWarps);
        compute_sync();
        if (!tc05::mbar_wait(&sh.mb2, 0, kOWait)) timed_out = true;
        for (int i = 0; i < n2; ++i) {
            for (int p = warp; p < k; p += kOWarps) {
                float c0 = 0.f, c8 = 0.f;
                if (sh.ids[p] >= 0) {
                    const uint8_t *rows = base + a.o_w2 + (i * k + p) * e2w;  // one 16-row box
                    const float *sc =
                        reinterpret_cast<const float *>(base + a.o_s2 + (i * k + p) * e2s);
                    for (int g = 0; g < GI; ++g) {
                        uint4 bu[1][2];
                        load_units(hu + (p * GI + g) * 16, bu);
                        tile_group_one(rows, 16, gid, rows, 16, gid + 8, g, bu, hf[p * GI + g],
                                       sc[gid * GI + g], sc[(gid + 8) * GI + g], c0, c8);
                    }
                }
                if (q == 0) {
                    red[p * 16 + gid] = c0;
                    red[p * 16 + 8 + gid] = c8;
                }
            }
            compute_sync();
            if (threadIdx.x < 16) {
                float o = 0.f;
                for (int p = 0; p < k; ++p)
                    if (sh.ids[p] >= 0) o = fmaf(sh.w[p], red[p * 16 + threadIdx.x], o);
                a.out[16 * (b + i * grid) + threadIdx.x] = o;
            }
            compute_sync();
        }
    }
    if (timed_out && lane == 0) atomicOr(a.status, 2);
    // copies still in flight (only after a wait ran out) land before exit
    if (warp == kOWarps && lane == 0) {
        for (int i = 0; i < n1; ++i) tc05::mbar_wait(&sh.mb1[i], 0, kOWait);
        tc05::mbar_wait(&sh.mb2, 0, kOWait);
    }
    __syncthreads();
}

inline size_t up16(size_t v) { return (v + 15) & ~(size_t)15; }
inline size_t up1k(size_t v) { return (v + 1023) & ~(size_t)1023; }

// Shared-memory layout for (H, I, k) on a grid of `grid` CTAs; false if it
// does not fit.
bool one_layout(const MoeDims &m, int k, int grid, OneArgs &a, size_t &smem) {
    const int GH = m.H / kGroup, GI = m.I / kGroup;
    const int tiles1 = k * (m.I / 8), tiles2 = m.H / 16;
    a.n1 = (tiles1 + grid - 1) / grid;
    a.n2 = (tiles2 + grid - 1) / grid;
    // weight boxes at 1024-byte aligned offsets (the 128-byte swizzle's atom)
    const size_t t1w = 16 * (size_t)(m.H / 2), t1s = 16 * (size_t)GH * 4;
    const size_t e2w = 16 * (size_t)(m.I / 2), e2s = 16 * (size_t)GI * 4;
    size_t o = 0;
    a.o_w1 = (int)o; o = up1k(o + (size_t)a.n1 * t1w);
    a.o_w2 = (int)o; o = up1k(o + (size_t)a.n2 * k * e2w);
    a.o_s1 = (int)o; o = up16(o + (size_t)a.n1 * t1s);
    a.o_s2 = (int)o; o = up16(o + (size_t)a.n2 * k * e2s);
    a.o_xu = (int)o; o = up16(o + (size_t)GH * 256);
    a.o_xf = (int)o; o = up16(o + (size_t)GH * 4);
    a.o_hu = (int)o; o = up16(o + (size_t)k * GI * 256);
    a.o_hf = (int)o; o = up16(o + (size_t)k * GI * 4);
    a.o_red = (int)o; o = up16(o + (size_t)std::max(a.n1 * kOWarps * 16, kOMaxK * 16) * 4);
    a.o_scr = (int)o; o = up16(o + (size_t)kOWarps * 8 * 64 * 4);
    a.o_lg = (int)o; o = up16(o + (size_t)1024 * 4);  // one routing row (E <= 1024)
    smem = o + 1024;
    return smem <= (size_t)kOSmemMax && a.n1 <= kOMaxT1;
}

}  // namespace

bool moe_one_supported(const MoeDims &m, int k) {
    // whole rows per box: row bytes (H / 2, I / 2) a multiple of 128, at most 32 KB
    if (k < 1 || k > kOMaxK || m.H % 256 || m.I % 256 || m.H > 65536 || m.I > 65536) return false;
    OneArgs a;
    size_t smem = 0;
    return one_layout(m, k, sm_count(), a, smem);
}

cudaError_t launch_moe_one(const MoeDims &m, const float *x, const int32_t *ids, const float *w,
                           int k, float *h, float *out, int32_t *status, cudaStream_t st,
                           const uint32_t *res, uint8_t *served, const float *logits,
                           int32_t *ids_out, float *w_out) {
    OneArgs a;
    memset(&a, 0, sizeof(a));
    size_t smem = 0;
    const int grid = sm_count();
    if (!one_layout(m, k, grid, a, smem)) return cudaErrorInvalidValue;
    a.gu_q = m.gu_q; a.gu_s = m.gu_s; a.dn_q = m.dn_q; a.dn_s = m.dn_s;
    a.E = m.E; a.H = m.H; a.I = m.I; a.k = k;
    a.x = x; a.ids = ids; a.w = w; a.h = h; a.out = out; a.status = status;
    a.res = res; a.served = served;
    a.logits = logits; a.ids_out = ids_out; a.w_out = w_out;
    if (!encode_rows_swizzled(&a.map_gu, m.gu_q, (long long)m.E * 2 * m.I, m.H / 2, 8) ||
        !encode_rows_swizzled(&a.map_dn, m.dn_q, (long long)m.E * m.H, m.I / 2, 16))
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem(k_moe_one, smem);
    if (e != cudaSuccess) return e;
    if (max_ctas_per_sm(k_moe_one, kOThreads, smem) < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kOThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_moe_one, a);
}

}  // namespace qmv
