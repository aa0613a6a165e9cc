// qmv_route.cuh - top-k routing of one token by one warp, shared by the
// routing kernel and the single-launch one-token FFN.
//
// Math (colibri PR #418, "coli_vk_expert_group"; the reading of the routing
// rule): the k experts with the largest fp32 logits, equal logits keeping the
// lower expert index first, in descending logit order; weights are the
// softmax over all experts restricted to the chosen k and renormalised, i.e.
// exp(l_e - l_max) / sum over the chosen. NaN logits are treated as -inf, so
// they are never chosen ahead of a finite logit.
#pragma once

#include <climits>
#include <cmath>

namespace qmv {

// Order-preserving 32-bit key of a non-NaN float (larger float, larger key;
// -0 must have been folded into +0) and its inverse. -inf has key 0x007FFFFF,
// so key 0 means "no candidate".
__device__ __forceinline__ uint32_t route_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float route_val(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Offers candidate (kk, e) to a lane's best (k1, i1) and second best (k2, i2);
// candidates arrive in increasing e, so equal keys keep the lower index ahead.
__device__ __forceinline__ void route_offer(uint32_t kk, int e, uint32_t &k1, int &i1,
                                            uint32_t &k2, int &i2) {
    if (kk > k1) {
        k2 = k1;
        i2 = i1;
        k1 = kk;
        i1 = e;
    } else if (kk > k2) {
        k2 = kk;
        i2 = e;
    }
}

// Warp-wide: logits l[0 .. E) (E <= 1024, k <= min(E, 32)) -> lane j < k gets
// the j-th expert id and its weight. row: 1024 words of this warp's shared
// memory (the experts' keys, for a lane that runs out of cached candidates).
//
// Lane L owns experts L, L + 32, ...; it keeps its best and second-best
// (key, index). Each of the k rounds takes the warp's largest key and, among
// lanes holding it, the lowest index (two warp reductions); the winning lane
// moves its second best up, and only a lane that wins a third time rescans
// its experts (skipping the ones taken).
__device__ __forceinline__ void route_warp(const float *__restrict__ l, int E, int k, float *row,
                                           int &my_id, float &my_w) {
    const int lane = threadIdx.x & 31;
    uint32_t *keys = reinterpret_cast<uint32_t *>(row);
    uint32_t k1 = 0u, k2 = 0u;
    int i1 = INT_MAX, i2 = INT_MAX;
    constexpr int kBatch = 8;  // logit loads in flight per lane
    for (int e0 = lane; e0 < E; e0 += 32 * kBatch) {
        float v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + 32 * u;
            v[u] = e < E ? l[e] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int e = e0 + 32 * u;
            if (e < E) {
                float x = v[u];
                if (x != x) x = -INFINITY;  // NaN never ahead of a finite logit
                if (x == 0.f) x = 0.f;      // -0 ties with +0 (then the lower index wins)
                const uint32_t kk = route_key(x);
                keys[e] = kk;
                route_offer(kk, e, k1, i1, k2, i2);
            }
        }
    }
    __syncwarp();
    uint32_t taken = 0u;  // bit i: expert lane + 32 i chosen
    bool second_known = true;
    my_id = 0;
    float my_l = -INFINITY;
    for (int j = 0; j < k; ++j) {
        const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, k1);
        const uint32_t mi =
            __reduce_min_sync(0xFFFFFFFFu, (k1 == mk && mk != 0u) ? (uint32_t)i1 : 0xFFFFFFFFu);
        if (lane == j) {
            my_id = (int)mi;
            my_l = route_val(mk);
        }
        if (mk != 0u && (int)(mi & 31u) == lane) {
            taken |= 1u << (mi >> 5);
            if (second_known) {
                k1 = k2;
                i1 = i2;
                second_known = false;
            } else {
                k1 = k2 = 0u;
                i1 = i2 = INT_MAX;
                for (int i = 0; lane + 32 * i < E; ++i) {
                    const int e = lane + 32 * i;
                    if (!((taken >> i) & 1u)) route_offer(keys[e], e, k1, i1, k2, i2);
                }
                second_known = true;
            }
        }
    }
    const float mx = __shfl_sync(0xFFFFFFFFu, my_l, 0);
    float ev = 0.0f;
    if (lane < k) ev = (mx == -INFINITY) ? 1.0f : expf(my_l - mx);
    float z = ev;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    my_w = ev / z;
}

}  // namespace qmv
