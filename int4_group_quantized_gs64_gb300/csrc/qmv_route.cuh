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

// Warp-wide: logits l[0 .. E) (E <= 1024) -> lane j < k gets the j-th expert
// id and its weight. row: 1024 floats of this warp's shared memory.
__device__ __forceinline__ void route_warp(const float *__restrict__ l, int E, int k, float *row,
                                           int &my_id, float &my_w) {
    const int lane = threadIdx.x & 31;
    for (int e = lane; e < E; e += 32) {
        const float v = l[e];
        row[e] = (v != v) ? -INFINITY : v;  // NaN never ahead of a finite logit
    }
    __syncwarp();
    uint32_t taken = 0u;
    my_id = 0;
    float my_l = -INFINITY;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int i = 0; lane + 32 * i < E; ++i) {
            if ((taken >> i) & 1u) continue;
            const int e = lane + 32 * i;
            const float v = row[e];
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
    float z = ev;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    my_w = ev / z;
}

}  // namespace qmv
