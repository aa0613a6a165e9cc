// qmv_internal.h - launchers behind the C ABI (host side, no validation here:
// the ABI layer checks every argument before calling these).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qmv {

// Dense GEMV, any S (passes of up to 16 tokens).
cudaError_t launch_dense_int4(const uint8_t *wq, const float *scales, int N, int K,
                              const float *x, float *y, int S, cudaStream_t st);
cudaError_t launch_dense_int8(const int8_t *w, const float *row_scale, int N, int K,
                              const float *x, float *y, int S, cudaStream_t st);

struct MoeDims {
    const uint8_t *gu_q;
    const float *gu_s;
    const uint8_t *dn_q;
    const float *dn_s;
    int E, H, I;
};

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         cudaStream_t st);
cudaError_t launch_group(const int32_t *ids, int P, int E, int32_t *offsets, int32_t *list,
                         int32_t *uexp, int32_t *n_used, int32_t *status, cudaStream_t st);
// Activation rows [R][K] fp32 -> fragment cells [R][K/64][4][4] uint4 + fac[R] (2^-sigma).
cudaError_t launch_split(const float *v, int R, int K, void *cells, float *fac, cudaStream_t st);
cudaError_t launch_gate_up(const MoeDims &m, const void *xcells, const float *xfac, int T, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, float *h, cudaStream_t st);
cudaError_t launch_down(const MoeDims &m, const void *hcells, const float *hfac, int T, int k,
                        const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                        const int32_t *n_used, float *y, cudaStream_t st);
cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E,
                           int H, float *out, cudaStream_t st);

// Workspace layout of the whole decode FFN.
struct MoeWorkspace {
    size_t status, offsets, list, uexp, n_used, xcells, xfac, h, hcells, hfac, y, total;
};
MoeWorkspace moe_ws_layout(int E, int H, int I, int T, int k);

}  // namespace qmv
