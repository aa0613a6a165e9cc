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

#include "qmv_internal.h"
#include "qmv_rows.cuh"

namespace qmv {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ------------------------------------------------------------------ routing

// One warp per token; lane L owns experts L, L+32, ... (E <= 1024).
__global__ void __launch_bounds__(256)
    k_route(const float *__restrict__ logits, int T, int E, int k, int32_t *__restrict__ ids,
            float *__restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *l = logits + (size_t)t * E;
    uint32_t taken = 0u;
    int my_id = 0;
    float my_l = -INFINITY;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int i = 0; lane + 32 * i < E; ++i) {
            if ((taken >> i) & 1u) continue;
            const int e = lane + 32 * i;
            float v = l[e];
            if (v != v) v = -INFINITY;  // NaN never ahead of a finite logit
            if (v > bv || (v == bv && e < bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) { my_id = bi; my_l = bv; }
    }
    const float mx = __shfl_sync(0xFFFFFFFFu, my_l, 0);
    float ev = 0.0f;
    if (lane < k) ev = (mx == -INFINITY) ? 1.0f : expf(my_l - mx);
    const float z = warp_sum(ev);
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = ev / z;
    }
}

// ------------------------------------------------------------------ grouping

// One CTA of 1024 threads. Counting by shared atomics, a block scan for the
// offsets, and a single warp that fills the lists in pair order (ranks from
// __match_any_sync), which keeps every list ascending.
__global__ void __launch_bounds__(1024)
    k_group(const int32_t *__restrict__ ids, int P, int E, int32_t *__restrict__ offsets,
            int32_t *__restrict__ list, int32_t *__restrict__ uexp, int32_t *__restrict__ n_used,
            int32_t *__restrict__ status) {
    __shared__ int32_t cnt[1024], run[1024];
    __shared__ int32_t warp_tot[32], warp_tot2[32];
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) bad = 0;
    for (int e = tid; e < 1024; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = ids[p];
        if (e < 0 || e >= E) bad = 1;
        else atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // Exclusive scans over the experts: counts -> offsets, used flags -> uexp slots.
    const int c = tid < E ? cnt[tid] : 0;
    const int f = c > 0 ? 1 : 0;
    int ic = c, ifl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, ic, o);
        const int b = __shfl_up_sync(0xFFFFFFFFu, ifl, o);
        if (lane >= o) { ic += a; ifl += b; }
    }
    if (lane == 31) { warp_tot[warp] = ic; warp_tot2[warp] = ifl; }
    __syncthreads();
    if (warp == 0) {
        int a = warp_tot[lane], b = warp_tot2[lane];
        int ia = a, ib = b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x1 = __shfl_up_sync(0xFFFFFFFFu, ia, o);
            const int x2 = __shfl_up_sync(0xFFFFFFFFu, ib, o);
            if (lane >= o) { ia += x1; ib += x2; }
        }
        warp_tot[lane] = ia - a;   // exclusive prefix of warp totals
        warp_tot2[lane] = ib - b;
    }
    __syncthreads();
    const int excl = warp_tot[warp] + ic - c;
    const int exflag = warp_tot2[warp] + ifl - f;
    if (tid < E) {
        offsets[tid] = excl;
        run[tid] = excl;
        if (f) uexp[exflag] = tid;
    }
    if (tid == E - 1) {
        offsets[E] = excl + c;
        *n_used = exflag + f;
    }
    __syncthreads();
    if (warp == 0) {
        const unsigned lt = (1u << lane) - 1u;
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            int e = p < P ? ids[p] : -1;
            const bool valid = p < P && e >= 0 && e < E;
            if (!valid) e = -1 - lane;  // unique key: never matches another lane
            const unsigned mask = __match_any_sync(0xFFFFFFFFu, e);
            const int rank = __popc(mask & lt);
            if (valid) list[run[e] + rank] = p;
            __syncwarp();
            if (valid && rank == 0) run[e] += __popc(mask);
            __syncwarp();
        }
    }
    if (tid == 0 && bad) atomicOr(status, 1);
}

// ------------------------------------------------------------------ activation split

// One CTA per row: max |v| -> power-of-two rescale, then the fragment cells.
__global__ void __launch_bounds__(256)
    k_split(const float *__restrict__ v, int K, uint4 *__restrict__ cells,
            float *__restrict__ fac) {
    __shared__ float red[8];
    const int r = blockIdx.x, tid = threadIdx.x;
    const float *row = v + (size_t)r * K;
    float m = 0.0f;
    for (int k = tid; k < K; k += blockDim.x) m = fmaxf(m, fabsf(row[k]));
    m = warp_max(m);
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    if (tid < 32) {
        float mm = tid < (int)(blockDim.x >> 5) ? red[tid] : 0.0f;
        mm = warp_max(mm);
        if (tid == 0) red[0] = mm;
    }
    __syncthreads();
    const int e = split_exponent(red[0]);
    const float mul = ldexpf(1.0f, e);
    if (tid == 0) fac[r] = ldexpf(1.0f, -e);
    const int G = K / kGroup;
    uint4 *out = cells + (size_t)r * G * 16;
    for (int c = tid; c < G * 16; c += blockDim.x) {
        const int g = c >> 4, m4 = (c >> 2) & 3, q = c & 3;
        int k0, k1, k2, k3;
        frag_ks<false>(g, m4, q, k0, k1, k2, k3);
        out[c] = make_cell(row[k0] * mul, row[k1] * mul, row[k2] * mul, row[k3] * mul);
    }
}

// ------------------------------------------------------------------ gate + up + SiLU

struct ExpertTokens {
    int e, beg, cnt;
};

__device__ __forceinline__ bool expert_of_block(const int32_t *offsets, const int32_t *uexp,
                                                const int32_t *n_used, int tiles,
                                                ExpertTokens &et, int &tile) {
    const int u = blockIdx.x / tiles;
    tile = blockIdx.x - u * tiles;
    if (u >= *n_used) return false;
    et.e = uexp[u];
    et.beg = offsets[et.e];
    et.cnt = offsets[et.e + 1] - et.beg;
    return true;
}

// Warps 0,1: gate rows j0 + 16w; warps 2,3: the matching up rows. One tile =
// 32 hidden units for every token of the expert.
template <int NB>
__device__ __forceinline__ void gate_up_pass(const MoeDims &m, const uint4 *xcells,
                                             const float *xfac, int k, const int32_t *list,
                                             const ExpertTokens &et, int tok0, int ntok, int j0,
                                             float *h, uint4 *cells, int *s_rows, int *s_pair,
                                             float *s_fac, float *s_gate) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int H = m.H, I = m.I, G = H / kGroup;
    const int rowInMat = (warp < 2) ? (j0 + 16 * warp) : (I + j0 + 16 * (warp - 2));
    const size_t eq = (size_t)et.e * 2 * I * (H / 2);
    const size_t es = (size_t)et.e * 2 * I * G;
    const int rA = rowInMat + gid, rB = rowInMat + gid + 8;

    WeightRing<false> ring;
    ring.init(m.gu_q + eq + (size_t)rA * (H / 2), m.gu_q + eq + (size_t)rB * (H / 2),
              m.gu_s + es + (size_t)rA * G, m.gu_s + es + (size_t)rB * G, G, q);
    ring.prologue();

    if (threadIdx.x < ntok) {
        const int p = list[et.beg + tok0 + threadIdx.x];
        const int t = p / k;
        s_pair[threadIdx.x] = p;
        s_rows[threadIdx.x] = t;
        s_fac[threadIdx.x] = xfac[t];
    }
    StageFromCells stage{xcells, s_rows, ntok, G, cells};
    float acc[NB][2];
    rows_mainloop<NB, false>(ring, cells, ntok, stage, acc);

    // gate warps publish g; up warps form h = SiLU(g) * u.
    if (warp < 2) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q;
            if (s < ntok) {
                s_gate[(16 * warp + gid) * kMaxTok + s] = acc[nb][0] * s_fac[s];
                s_gate[(16 * warp + gid + 8) * kMaxTok + s] = acc[nb][1] * s_fac[s];
            }
        }
    }
    __syncthreads();
    if (warp >= 2) {
        const int lr = 16 * (warp - 2) + gid;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const int s = 4 * nb + q;
            if (s < ntok) {
                const float u0 = acc[nb][0] * s_fac[s], u1 = acc[nb][1] * s_fac[s];
                const float g0 = s_gate[lr * kMaxTok + s], g1 = s_gate[(lr + 8) * kMaxTok + s];
                const size_t hb = (size_t)s_pair[s] * I + j0;
                h[hb + lr] = g0 / (1.0f + expf(-g0)) * u0;
                h[hb + lr + 8] = g1 / (1.0f + expf(-g1)) * u1;
            }
        }
    }
    __syncthreads();  // s_gate / s_pair reused by the next pass
}

__global__ void __launch_bounds__(kCtaThreads)
    k_gate_up(MoeDims m, const uint4 *__restrict__ xcells, const float *__restrict__ xfac, int k,
              const int32_t *__restrict__ offsets, const int32_t *__restrict__ list,
              const int32_t *__restrict__ uexp, const int32_t *__restrict__ n_used,
              float *__restrict__ h) {
    extern __shared__ uint4 cells[];
    __shared__ int s_rows[kMaxTok], s_pair[kMaxTok];
    __shared__ float s_fac[kMaxTok];
    __shared__ float s_gate[32 * kMaxTok];
    const int tiles = m.I / 32;
    ExpertTokens et;
    int tile;
    if (!expert_of_block(offsets, uexp, n_used, tiles, et, tile)) return;
    const int j0 = tile * 32;
    for (int tok0 = 0; tok0 < et.cnt; tok0 += kMaxTok) {
        const int ntok = min(kMaxTok, et.cnt - tok0);
        if (ntok <= 4)
            gate_up_pass<1>(m, xcells, xfac, k, list, et, tok0, ntok, j0, h, cells, s_rows, s_pair,
                            s_fac, s_gate);
        else if (ntok <= 8)
            gate_up_pass<2>(m, xcells, xfac, k, list, et, tok0, ntok, j0, h, cells, s_rows, s_pair,
                            s_fac, s_gate);
        else
            gate_up_pass<4>(m, xcells, xfac, k, list, et, tok0, ntok, j0, h, cells, s_rows, s_pair,
                            s_fac, s_gate);
    }
}

// ------------------------------------------------------------------ down

template <int NB>
__device__ __forceinline__ void down_pass(const MoeDims &m, const uint4 *hcells, const float *hfac,
                                          const int32_t *list, const ExpertTokens &et, int tok0,
                                          int ntok, int i0, float *y, uint4 *cells, int *s_pair,
                                          float *s_fac) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
    const int H = m.H, I = m.I, G = I / kGroup;
    const int row0 = i0 + 16 * warp;
    const int rA = min(row0 + gid, H - 1), rB = min(row0 + gid + 8, H - 1);
    const size_t eq = (size_t)et.e * H * (I / 2);
    const size_t es = (size_t)et.e * H * G;

    WeightRing<false> ring;
    ring.init(m.dn_q + eq + (size_t)rA * (I / 2), m.dn_q + eq + (size_t)rB * (I / 2),
              m.dn_s + es + (size_t)rA * G, m.dn_s + es + (size_t)rB * G, G, q);
    ring.prologue();

    if (threadIdx.x < ntok) {
        const int p = list[et.beg + tok0 + threadIdx.x];
        s_pair[threadIdx.x] = p;
        s_fac[threadIdx.x] = hfac[p];
    }
    StageFromCells stage{hcells, s_pair, ntok, G, cells};
    float acc[NB][2];
    rows_mainloop<NB, false>(ring, cells, ntok, stage, acc);
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int s = 4 * nb + q;
        if (s < ntok) {
            const size_t yb = (size_t)s_pair[s] * H;
            if (row0 + gid < H) y[yb + row0 + gid] = acc[nb][0] * s_fac[s];
            if (row0 + gid + 8 < H) y[yb + row0 + gid + 8] = acc[nb][1] * s_fac[s];
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kCtaThreads)
    k_down(MoeDims m, const uint4 *__restrict__ hcells, const float *__restrict__ hfac,
           const int32_t *__restrict__ offsets, const int32_t *__restrict__ list,
           const int32_t *__restrict__ uexp, const int32_t *__restrict__ n_used,
           float *__restrict__ y) {
    extern __shared__ uint4 cells[];
    __shared__ int s_pair[kMaxTok];
    __shared__ float s_fac[kMaxTok];
    const int tiles = (m.H + 16 * kWarps - 1) / (16 * kWarps);
    ExpertTokens et;
    int tile;
    if (!expert_of_block(offsets, uexp, n_used, tiles, et, tile)) return;
    const int i0 = tile * 16 * kWarps;
    for (int tok0 = 0; tok0 < et.cnt; tok0 += kMaxTok) {
        const int ntok = min(kMaxTok, et.cnt - tok0);
        if (ntok <= 4)
            down_pass<1>(m, hcells, hfac, list, et, tok0, ntok, i0, y, cells, s_pair, s_fac);
        else if (ntok <= 8)
            down_pass<2>(m, hcells, hfac, list, et, tok0, ntok, i0, y, cells, s_pair, s_fac);
        else
            down_pass<4>(m, hcells, hfac, list, et, tok0, ntok, i0, y, cells, s_pair, s_fac);
    }
}

// ------------------------------------------------------------------ combine

__global__ void __launch_bounds__(256)
    k_combine(const float *__restrict__ y, const int32_t *__restrict__ ids,
              const float *__restrict__ w, int k, int E, int H, float *__restrict__ out) {
    const int t = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= H) return;
    float o = 0.0f;
    for (int j = 0; j < k; ++j) {
        const int p = t * k + j;
        const int e = ids[p];
        if (e >= 0 && e < E) o = fmaf(w[p], y[(size_t)p * H + i], o);
    }
    out[(size_t)t * H + i] = o;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

// ------------------------------------------------------------------ launchers

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int per = 8;  // tokens (warps) per CTA
    k_route<<<(T + per - 1) / per, 32 * per, 0, st>>>(logits, T, E, k, ids, w);
    return cudaGetLastError();
}

cudaError_t launch_group(const int32_t *ids, int P, int E, int32_t *offsets, int32_t *list,
                         int32_t *uexp, int32_t *n_used, int32_t *status, cudaStream_t st) {
    k_group<<<1, 1024, 0, st>>>(ids, P, E, offsets, list, uexp, n_used, status);
    return cudaGetLastError();
}

cudaError_t launch_split(const float *v, int R, int K, void *cells, float *fac, cudaStream_t st) {
    if (R == 0) return cudaSuccess;
    k_split<<<R, 256, 0, st>>>(v, K, static_cast<uint4 *>(cells), fac);
    return cudaGetLastError();
}

cudaError_t launch_gate_up(const MoeDims &m, const void *xcells, const float *xfac, int T, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, float *h, cudaStream_t st) {
    const int P = T * k;
    const int maxU = P < m.E ? P : m.E;
    if (maxU == 0) return cudaSuccess;
    const int tiles = m.I / 32;
    const size_t smem = (size_t)kCellBudget;
    k_gate_up<<<maxU * tiles, kCtaThreads, smem, st>>>(
        m, static_cast<const uint4 *>(xcells), xfac, k, offsets, list, uexp, n_used, h);
    return cudaGetLastError();
}

cudaError_t launch_down(const MoeDims &m, const void *hcells, const float *hfac, int T, int k,
                        const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                        const int32_t *n_used, float *y, cudaStream_t st) {
    const int P = T * k;
    const int maxU = P < m.E ? P : m.E;
    if (maxU == 0) return cudaSuccess;
    const int tiles = (m.H + 16 * kWarps - 1) / (16 * kWarps);
    const size_t smem = (size_t)kCellBudget;
    k_down<<<maxU * tiles, kCtaThreads, smem, st>>>(m, static_cast<const uint4 *>(hcells), hfac,
                                                    offsets, list, uexp, n_used, y);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E,
                           int H, float *out, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    dim3 grid((H + 255) / 256, T);
    k_combine<<<grid, 256, 0, st>>>(y, ids, w, k, E, H, out);
    return cudaGetLastError();
}

MoeWorkspace moe_ws_layout(int E, int H, int I, int T, int k) {
    MoeWorkspace L{};
    const size_t P = (size_t)T * k;
    size_t o = 0;
    L.status = o; o = align256(o + 4);
    L.offsets = o; o = align256(o + 4 * (size_t)(E + 1));
    L.list = o; o = align256(o + 4 * P);
    L.uexp = o; o = align256(o + 4 * (size_t)E);
    L.n_used = o; o = align256(o + 4);
    L.xcells = o; o = align256(o + 4 * (size_t)T * H);
    L.xfac = o; o = align256(o + 4 * (size_t)T);
    L.h = o; o = align256(o + 4 * P * I);
    L.hcells = o; o = align256(o + 4 * P * I);
    L.hfac = o; o = align256(o + 4 * P);
    L.y = o; o = align256(o + 4 * P * H);
    L.total = o;
    return L;
}

}  // namespace qmv
