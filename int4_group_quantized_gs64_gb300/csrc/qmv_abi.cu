// qmv_abi.cu - the extern "C" entry points declared in include/qmv.h.
//
// Every entry point validates its arguments on the host and returns a
// negative qmv_status before enqueuing anything (so a failed call leaves its
// outputs alone, as the pages require of a failed take: colibri PR #1338,
// fake-Vulkan gate comment), then calls the launchers of qmv_internal.h.
#include <stdint.h>

#include "../../include/qmv.h"
#include "qmv_internal.h"

namespace {

constexpr int kMaxK = 65536;
constexpr int kMaxE = 1024;
constexpr int kMaxPairs = 1 << 20;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline cudaStream_t cs(qmv_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? QMV_OK : QMV_ECUDA; }

int check_moe(const qmv_moe_int4 *m) {
    if (!m || !m->gu_q || !m->gu_s || !m->dn_q || !m->dn_s) return QMV_EINVAL;
    if (m->gs != 64 || m->E < 1 || m->E > kMaxE) return QMV_EINVAL;
    if (m->H < 64 || m->I < 64 || m->H % 64 || m->I % 64 || m->H > kMaxK || m->I > kMaxK)
        return QMV_ESHAPE;
    if (!aligned(m->gu_q, 16) || !aligned(m->dn_q, 16) || !aligned(m->gu_s, 4) ||
        !aligned(m->dn_s, 4))
        return QMV_EALIGN;
    return QMV_OK;
}

qmv::MoeDims dims(const qmv_moe_int4 *m) {
    return qmv::MoeDims{m->gu_q, m->gu_s, m->dn_q, m->dn_s, m->E, m->H, m->I};
}

int check_group_args(const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                     const int32_t *n_used) {
    if (!offsets || !list || !uexp || !n_used) return QMV_EINVAL;
    if (!aligned(offsets, 4) || !aligned(list, 4) || !aligned(uexp, 4) || !aligned(n_used, 4))
        return QMV_EALIGN;
    return QMV_OK;
}

int ffn_check(const qmv_moe_int4 *m, int T, int k, void *ws, size_t ws_bytes,
                     qmv::MoeWorkspace &L) {
    int r = check_moe(m);
    if (r) return r;
    if (T < 1 || k < 1 || k > m->E || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    L = qmv::moe_ws_layout(m->E, m->H, m->I, T, k);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return QMV_EWORKSPACE;
    return QMV_OK;
}

// The phases keep the activation units pass-packed (two copies per stage in
// the tensor-map kernel) when that kernel runs and a token's pairs fit the
// grouping kernel's per-token slots.
bool packed_units(const qmv_moe_int4 *m, int T, int k) {
    return qmv::tma_moe_supported(dims(m), (long long)T * k) && k <= 32;
}

// The tensor-map kernels run this call (shape, alignment, and a stage count
// that their 32-bit stage numbers hold).
bool tma_path(const qmv_moe_int4 *m, int T, int k) {
    return qmv::tma_moe_supported(dims(m), (long long)T * k);
}

bool one_token(const qmv_moe_int4 *m, int k) {
    const qmv::MoeDims d = dims(m);
    return k >= 1 && k <= m->E && qmv::tma_moe_supported(d) && qmv::moe_one_supported(d, k);
}

template <class T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

}  // namespace

extern "C" {

int qmv_version(void) { return 100; }

int qmv_test_split_skew(int ns) {
    const int old = qmv::g_split_skew_ns;
    qmv::g_split_skew_ns = ns > 0 ? ns : 0;
    return old;
}

const char *qmv_status_str(int status) {
    switch (status) {
        case QMV_OK: return "ok";
        case QMV_EINVAL: return "invalid argument";
        case QMV_ESHAPE: return "unsupported shape";
        case QMV_EWORKSPACE: return "workspace missing, misaligned or too small";
        case QMV_ECUDA: return "CUDA launch failed";
        case QMV_ETIMEOUT: return "device wait timed out";
        case QMV_EALIGN: return "pointer misaligned";
        default: return "unknown status";
    }
}

size_t qmv_gemv_workspace_bytes(int K, int S) {
    if (K < 64 || K % 64 || K > kMaxK || S < 1) return 0;
    return qmv::gemv_ws_bytes(K, S);
}

int qmv_int4_gs(const uint8_t *wq, const float *scales, int N, int K, int gs, const float *x,
                float *y, int S, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!wq || !scales || !x || !y || N < 1 || S < 1 || gs != 64) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(wq, 16) || !aligned(scales, 4) || !aligned(x, 4) || !aligned(y, 4))
        return QMV_EALIGN;
    if (!ws || !aligned(ws, 256) || ws_bytes < qmv_gemv_workspace_bytes(K, S)) return QMV_EWORKSPACE;
    return from_cuda(qmv::launch_gemv_int4(wq, scales, N, K, x, y, S, ws, cs(stream)));
}

int qmv_int4_gs_bf16(const uint8_t *wq, const float *scales, int N, int K, int gs, const float *x,
                     uint16_t *y_bf16, int S, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!wq || !scales || !x || !y_bf16 || N < 1 || S < 1 || gs != 64) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(wq, 16) || !aligned(scales, 4) || !aligned(x, 4) || !aligned(y_bf16, 2))
        return QMV_EALIGN;
    if (!ws || !aligned(ws, 256) || ws_bytes < qmv_gemv_workspace_bytes(K, S)) return QMV_EWORKSPACE;
    return from_cuda(
        qmv::launch_gemv_int4(wq, scales, N, K, x, nullptr, S, ws, cs(stream), y_bf16));
}

int qmv_int4_gs_pair(const uint8_t *wq0, const float *s0, int N0, const uint8_t *wq1,
                     const float *s1, int N1, int K, int gs, const float *x, float *y0, float *y1,
                     int S, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!wq0 || !s0 || !wq1 || !s1 || !x || !y0 || !y1 || N0 < 1 || N1 < 1 || S < 1 || gs != 64)
        return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(wq0, 16) || !aligned(wq1, 16) || !aligned(s0, 4) || !aligned(s1, 4) ||
        !aligned(x, 4) || !aligned(y0, 4) || !aligned(y1, 4))
        return QMV_EALIGN;
    if (!ws || !aligned(ws, 256) || ws_bytes < qmv_gemv_workspace_bytes(K, S)) return QMV_EWORKSPACE;
    return from_cuda(
        qmv::launch_gemv_int4_pair(wq0, s0, N0, wq1, s1, N1, K, x, y0, y1, S, ws, cs(stream)));
}

int qmv_int3_gs(const uint8_t *wq3, const float *scales, int N, int K, int gs, const float *x,
                float *y, int S, qmv_stream_t stream) {
    if (!wq3 || !scales || !x || !y || N < 1 || S < 1 || gs != 64) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(wq3, 4) || !aligned(scales, 4) || !aligned(x, 16) || !aligned(y, 4))
        return QMV_EALIGN;
    return from_cuda(qmv::launch_gemv_int3(wq3, scales, N, K, x, y, S, cs(stream)));
}

int qmv_int8_row(const int8_t *w, const float *row_scale, int N, int K, const float *x, float *y,
                 int S, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!w || !row_scale || !x || !y || N < 1 || S < 1) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(w, 16) || !aligned(row_scale, 4) || !aligned(x, 4) || !aligned(y, 4))
        return QMV_EALIGN;
    if (!ws || !aligned(ws, 256) || ws_bytes < qmv_gemv_workspace_bytes(K, S)) return QMV_EWORKSPACE;
    return from_cuda(qmv::launch_gemv_int8(w, row_scale, N, K, x, y, S, ws, cs(stream)));
}

int qmv_int8_row_bf16(const int8_t *w, const float *row_scale, int N, int K, const float *x,
                      uint16_t *y_bf16, int S, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!w || !row_scale || !x || !y_bf16 || N < 1 || S < 1) return QMV_EINVAL;
    if (K < 64 || K % 64 || K > kMaxK) return QMV_ESHAPE;
    if (!aligned(w, 16) || !aligned(row_scale, 4) || !aligned(x, 4) || !aligned(y_bf16, 2))
        return QMV_EALIGN;
    if (!ws || !aligned(ws, 256) || ws_bytes < qmv_gemv_workspace_bytes(K, S)) return QMV_EWORKSPACE;
    return from_cuda(
        qmv::launch_gemv_int8(w, row_scale, N, K, x, nullptr, S, ws, cs(stream), y_bf16));
}

int moe_route_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                   qmv_stream_t stream) {
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > E || k > 32) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!logits || !ids || !w) return QMV_EINVAL;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(w, 4)) return QMV_EALIGN;
    return from_cuda(qmv::launch_route(logits, T, E, k, ids, w, cs(stream)));
}

int moe_group(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *list,
              int32_t *uexp, int32_t *n_used, int32_t *status, qmv_stream_t stream) {
    if (T < 0 || k < 1 || E < 1 || E > kMaxE || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (!status || (T > 0 && !ids)) return QMV_EINVAL;
    int r = check_group_args(offsets, list, uexp, n_used);
    if (r) return r;
    if (!aligned(status, 4) || (ids && !aligned(ids, 4))) return QMV_EALIGN;
    return from_cuda(qmv::launch_group(ids, T * k, E, offsets, list, uexp, n_used, status,
                                       cs(stream)));
}

size_t moe_workspace_bytes(const qmv_moe_int4 *m, int T, int k) {
    if (check_moe(m) || T < 0 || k < 1 || (int64_t)T * k > kMaxPairs) return 0;
    return qmv::moe_ws_layout(m->E, m->H, m->I, T, k).total;
}

int moe_gate_up_silu(const qmv_moe_int4 *m, const float *x, int T, int k, const int32_t *offsets,
                     const int32_t *list, const int32_t *uexp, const int32_t *n_used, float *h,
                     void *ws, size_t ws_bytes, qmv_stream_t stream) {
    int r = check_moe(m);
    if (r) return r;
    if (T < 0 || k < 1 || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!x || !h) return QMV_EINVAL;
    if ((r = check_group_args(offsets, list, uexp, n_used))) return r;
    if (!aligned(x, 4) || !aligned(h, 4)) return QMV_EALIGN;
    const qmv::MoeWorkspace L = qmv::moe_ws_layout(m->E, m->H, m->I, T, k);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return QMV_EWORKSPACE;
    char *b = static_cast<char *>(ws);
    int32_t *pass_ofs = reinterpret_cast<int32_t *>(b + L.pass_ofs);
    float *xfac = reinterpret_cast<float *>(b + L.xfac);
    const cudaStream_t st = cs(stream);
    int32_t *cnt = reinterpret_cast<int32_t *>(b + L.sk_cnt);
    float *part = reinterpret_cast<float *>(b + L.sk_part);
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * qmv::kSkMaxCtas, st);
    if (e == cudaSuccess) e = qmv::launch_passes(offsets, uexp, n_used, pass_ofs, st, false);
    if (e == cudaSuccess)
        e = qmv::launch_split(x, T, m->H, b + L.xcells, xfac, st, tma_path(m, T, k));
    if (e == cudaSuccess) {
        float *hfac = reinterpret_cast<float *>(b + L.hfac);
        if (tma_path(m, T, k))
            e = qmv::launch_moe_tma(dims(m), 0, b + L.xcells, xfac, k, offsets, list, uexp, n_used,
                                    pass_ofs, h, b + L.hcells, hfac, nullptr,
                                    reinterpret_cast<int32_t *>(b + L.status), cnt, part, st);
        else
            e = qmv::launch_gate_up(dims(m), b + L.xcells, xfac, k, offsets, list, uexp, n_used,
                                    pass_ofs, h, b + L.hcells, hfac, st);
    }
    return from_cuda(e);
}

int moe_down(const qmv_moe_int4 *m, const float *h, int T, int k, const int32_t *offsets,
             const int32_t *list, const int32_t *uexp, const int32_t *n_used, float *y, void *ws,
             size_t ws_bytes, qmv_stream_t stream) {
    int r = check_moe(m);
    if (r) return r;
    if (T < 0 || k < 1 || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!h || !y) return QMV_EINVAL;
    if ((r = check_group_args(offsets, list, uexp, n_used))) return r;
    if (!aligned(h, 4) || !aligned(y, 4)) return QMV_EALIGN;
    const qmv::MoeWorkspace L = qmv::moe_ws_layout(m->E, m->H, m->I, T, k);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return QMV_EWORKSPACE;
    char *b = static_cast<char *>(ws);
    int32_t *pass_ofs = reinterpret_cast<int32_t *>(b + L.pass_ofs);
    float *hfac = reinterpret_cast<float *>(b + L.hfac);
    const cudaStream_t st = cs(stream);
    int32_t *cnt = reinterpret_cast<int32_t *>(b + L.sk_cnt) + qmv::kSkMaxCtas;
    float *part = reinterpret_cast<float *>(b + L.sk_part);
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int32_t) * qmv::kSkMaxCtas, st);
    if (e == cudaSuccess) e = qmv::launch_passes(offsets, uexp, n_used, pass_ofs, st, false);
    if (e == cudaSuccess)
        e = qmv::launch_split(h, T * k, m->I, b + L.hcells, hfac, st, tma_path(m, T, k));
    if (e == cudaSuccess) {
        if (tma_path(m, T, k))
            e = qmv::launch_moe_tma(dims(m), 1, b + L.hcells, hfac, k, offsets, list, uexp, n_used,
                                    pass_ofs, nullptr, nullptr, nullptr, y,
                                    reinterpret_cast<int32_t *>(b + L.status), cnt, part, st);
        else
            e = qmv::launch_down(dims(m), b + L.hcells, hfac, offsets, list, uexp, n_used, pass_ofs,
                                 y, st);
    }
    return from_cuda(e);
}

int moe_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E, int H,
                float *out, qmv_stream_t stream) {
    if (T < 0 || k < 1 || E < 1 || H < 1 || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!y || !ids || !w || !out) return QMV_EINVAL;
    if (!aligned(y, 4) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(out, 4)) return QMV_EALIGN;
    return from_cuda(qmv::launch_combine(y, ids, w, T, k, E, H, out, cs(stream), false));
}

}  // extern "C"

namespace {

// The prepare phase with an optional residency bitmap and served mask.
int prepare_impl(const qmv_moe_int4 *m, const float *x, int T, const int32_t *ids, int k,
                 void *ws, size_t ws_bytes, qmv_stream_t stream, const uint32_t *res,
                 uint8_t *served, const float *logits = nullptr, int32_t *ids_out = nullptr,
                 float *w_out = nullptr) {
    qmv::MoeWorkspace L;
    int r = ffn_check(m, T, k, ws, ws_bytes, L);
    if (r) return r;
    if (!x || !ids) return QMV_EINVAL;
    if (!aligned(x, 4) || !aligned(ids, 4)) return QMV_EALIGN;
    const bool pk = packed_units(m, T, k);
    // the packed path also gets the work plan of the gate+up and down kernels
    qmv::PlanArgs plan{};
    if (pk) {
        plan.ptab = at<int4>(ws, L.ptab);
        plan.plan_gu = at<int4>(ws, L.plan);
        plan.plan_dn = at<int4>(ws, L.plan) + qmv::kSkMaxCtas + 1;
        plan.s_gu = ((m->I + 127) / 128) * (m->H / 256);
        plan.s_dn = ((m->H + 255) / 256) * (m->I / 256);
        plan.ns_gu = m->H / 256;
        plan.ns_dn = m->I / 256;
        plan.g = qmv::tma_grid();
    }
    // the grouping kernel clears the status word and the split counters itself
    return from_cuda(qmv::launch_group_split(
        ids, T, k, m->E, at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.list),
        at<int32_t>(ws, L.uexp), at<int32_t>(ws, L.n_used), at<int32_t>(ws, L.pass_ofs),
        at<int32_t>(ws, L.status), x, m->H, at<void>(ws, pk ? L.xpk : L.xcells),
        (pk ? nullptr : at<float>(ws, L.xfac)), cs(stream), 8, pk, at<int32_t>(ws, L.status),
        (int)(L.status_bytes / 4), true, res, served, logits, ids_out, w_out,
        tma_path(m, T, k), pk ? &plan : nullptr));
}

// Whole FFN (moe_expert_ffn_int4 with res == served == null).
int ffn_impl(const qmv_moe_int4 *m, const uint32_t *res, const float *x, int T,
             const int32_t *ids, const float *w, int k, float *out, uint8_t *served, void *ws,
             size_t ws_bytes, qmv_stream_t stream);

}  // namespace

extern "C" {

int moe_ffn_prepare(const qmv_moe_int4 *m, const float *x, int T, const int32_t *ids, int k,
                    void *ws, size_t ws_bytes, qmv_stream_t stream) {
    return prepare_impl(m, x, T, ids, k, ws, ws_bytes, stream, nullptr, nullptr);
}

int moe_ffn_gate_up(const qmv_moe_int4 *m, int T, int k, void *ws, size_t ws_bytes,
                    qmv_stream_t stream) {
    qmv::MoeWorkspace L;
    int r = ffn_check(m, T, k, ws, ws_bytes, L);
    if (r) return r;
    if (tma_path(m, T, k)) {
        const bool pk = packed_units(m, T, k);
        return from_cuda(qmv::launch_moe_tma(
            dims(m), 0, at<void>(ws, pk ? L.xpk : L.xcells), (pk ? nullptr : at<float>(ws, L.xfac)), k,
            at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.list), at<int32_t>(ws, L.uexp),
            at<int32_t>(ws, L.n_used), at<int32_t>(ws, L.pass_ofs), at<float>(ws, L.h),
            at<void>(ws, pk ? L.hpk : L.hcells), (pk ? nullptr : at<float>(ws, L.hfac)), nullptr,
            at<int32_t>(ws, L.status), at<int32_t>(ws, L.sk_cnt), at<float>(ws, L.sk_part),
            cs(stream), pk, pk ? at<int4>(ws, L.ptab) : nullptr,
            pk ? at<int4>(ws, L.plan) : nullptr));
    }
    return from_cuda(qmv::launch_gate_up(
        dims(m), at<void>(ws, L.xcells), at<float>(ws, L.xfac), k, at<int32_t>(ws, L.offsets),
        at<int32_t>(ws, L.list), at<int32_t>(ws, L.uexp), at<int32_t>(ws, L.n_used),
        at<int32_t>(ws, L.pass_ofs), at<float>(ws, L.h), at<void>(ws, L.hcells),
        at<float>(ws, L.hfac), cs(stream)));
}

int moe_ffn_down(const qmv_moe_int4 *m, int T, int k, void *ws, size_t ws_bytes,
                 qmv_stream_t stream) {
    qmv::MoeWorkspace L;
    int r = ffn_check(m, T, k, ws, ws_bytes, L);
    if (r) return r;
    if (tma_path(m, T, k)) {
        const bool pk = packed_units(m, T, k);
        return from_cuda(qmv::launch_moe_tma(
            dims(m), 1, at<void>(ws, pk ? L.hpk : L.hcells), (pk ? nullptr : at<float>(ws, L.hfac)), k,
            at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.list), at<int32_t>(ws, L.uexp),
            at<int32_t>(ws, L.n_used), at<int32_t>(ws, L.pass_ofs), nullptr, nullptr, nullptr,
            at<float>(ws, L.y), at<int32_t>(ws, L.status), at<int32_t>(ws, L.sk_cnt) + qmv::kSkMaxCtas,
            at<float>(ws, L.sk_part), cs(stream), pk, pk ? at<int4>(ws, L.ptab) : nullptr,
            pk ? at<int4>(ws, L.plan) + qmv::kSkMaxCtas + 1 : nullptr));
    }
    return from_cuda(qmv::launch_down(dims(m), at<void>(ws, L.hcells), at<float>(ws, L.hfac),
                                      at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.list),
                                      at<int32_t>(ws, L.uexp), at<int32_t>(ws, L.n_used),
                                      at<int32_t>(ws, L.pass_ofs), at<float>(ws, L.y), cs(stream)));
}

int moe_ffn_combine(const qmv_moe_int4 *m, const int32_t *ids, const float *w, int T, int k,
                    float *out, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    qmv::MoeWorkspace L;
    int r = ffn_check(m, T, k, ws, ws_bytes, L);
    if (r) return r;
    if (!ids || !w || !out) return QMV_EINVAL;
    if (!aligned(ids, 4) || !aligned(w, 4) || !aligned(out, 4)) return QMV_EALIGN;
    return from_cuda(qmv::launch_combine(at<float>(ws, L.y), ids, w, T, k, m->E, m->H, out,
                                         cs(stream), true));
}

int moe_weight_path(const qmv_moe_int4 *m) {
    const int r = check_moe(m);
    if (r) return r;
    return qmv::tma_moe_supported(dims(m)) ? 1 : 0;
}

int moe_one_token_path(const qmv_moe_int4 *m, int k) {
    const int r = check_moe(m);
    if (r) return r;
    return one_token(m, k) ? 1 : 0;
}

int moe_expert_ffn_int4(const qmv_moe_int4 *m, const float *x, int T, const int32_t *ids,
                        const float *w, int k, float *out, void *ws, size_t ws_bytes,
                        qmv_stream_t stream) {
    return ffn_impl(m, nullptr, x, T, ids, w, k, out, nullptr, ws, ws_bytes, stream);
}

int moe_route_expert_ffn_int4(const qmv_moe_int4 *m, const float *logits, const float *x, int T,
                              int k, int32_t *ids, float *w, float *out, void *ws, size_t ws_bytes,
                              qmv_stream_t stream) {
    int r = check_moe(m);
    if (r) return r;
    if (T < 0 || k < 1 || k > m->E || k > 32 || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!logits || !ids || !w) return QMV_EINVAL;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(w, 4)) return QMV_EALIGN;
    if (T == 1 && one_token(m, k)) {
        qmv::MoeWorkspace L;
        if ((r = ffn_check(m, T, k, ws, ws_bytes, L))) return r;
        if (!x || !out) return QMV_EINVAL;
        if (!aligned(x, 4) || !aligned(out, 4)) return QMV_EALIGN;
        // one token: routing inside the single cooperative launch, which
        // clears the status word itself
        return from_cuda(qmv::launch_moe_one(dims(m), x, nullptr, nullptr, k, at<float>(ws, L.h),
                                             out, at<int32_t>(ws, L.status), cs(stream), nullptr,
                                             nullptr, logits, ids, w));
    }
    if (T <= 32 && packed_units(m, T, k)) {
        // a decode micro-batch: the grouping kernel routes the tokens itself
        qmv::MoeWorkspace L;
        if ((r = ffn_check(m, T, k, ws, ws_bytes, L))) return r;
        if (!x || !out) return QMV_EINVAL;
        if (!aligned(x, 4) || !aligned(out, 4)) return QMV_EALIGN;
        if ((r = prepare_impl(m, x, T, ids, k, ws, ws_bytes, stream, nullptr, nullptr, logits,
                              ids, w)))
            return r;
        if ((r = moe_ffn_gate_up(m, T, k, ws, ws_bytes, stream))) return r;
        if ((r = moe_ffn_down(m, T, k, ws, ws_bytes, stream))) return r;
        // ids and w come from the grouping kernel, three launches back
        return from_cuda(qmv::launch_combine(at<float>(ws, L.y), ids, w, T, k, m->E, m->H, out,
                                             cs(stream), true, nullptr, true));
    }
    if ((r = moe_route_topk(logits, T, m->E, k, ids, w, stream))) return r;
    return moe_expert_ffn_int4(m, x, T, ids, w, k, out, ws, ws_bytes, stream);
}

int moe_expert_ffn_int4_resident(const qmv_moe_int4 *m, const uint32_t *resident, const float *x,
                                 int T, const int32_t *ids, const float *w, int k, float *out,
                                 uint8_t *served, void *ws, size_t ws_bytes, qmv_stream_t stream) {
    if (!resident || !served) return QMV_EINVAL;
    if (!aligned(resident, 4)) return QMV_EALIGN;
    return ffn_impl(m, resident, x, T, ids, w, k, out, served, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {

int ffn_impl(const qmv_moe_int4 *m, const uint32_t *res, const float *x, int T,
             const int32_t *ids, const float *w, int k, float *out, uint8_t *served, void *ws,
             size_t ws_bytes, qmv_stream_t stream) {
    if (T == 0 && !check_moe(m) && k >= 1 && k <= m->E) return QMV_OK;
    qmv::MoeWorkspace L;
    int r = ffn_check(m, T, k, ws, ws_bytes, L);
    if (r) return r;
    if (!x || !ids || !w || !out) return QMV_EINVAL;
    if (!aligned(x, 4) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(out, 4)) return QMV_EALIGN;
    const cudaStream_t st = cs(stream);
    if (T == 1 && one_token(m, k)) {
        // one token: a single cooperative launch (it clears the status word)
        return from_cuda(qmv::launch_moe_one(dims(m), x, ids, w, k, at<float>(ws, L.h), out,
                                             at<int32_t>(ws, L.status), st, res, served));
    }
    if ((r = prepare_impl(m, x, T, ids, k, ws, ws_bytes, stream, res, served))) return r;
    if ((r = moe_ffn_gate_up(m, T, k, ws, ws_bytes, stream))) return r;
    if ((r = moe_ffn_down(m, T, k, ws, ws_bytes, stream))) return r;
    // ids, w and res are call inputs, older than this call's first kernel
    return from_cuda(qmv::launch_combine(at<float>(ws, L.y), ids, w, T, k, m->E, m->H, out, st,
                                         true, res, true));
}

}  // namespace

extern "C" {

size_t moe_prefill_workspace_bytes(const qmv_moe_int4 *m, int T, int k) {
    if (check_moe(m) || m->I % 128 || T < 0 || k < 1 || (int64_t)T * k > kMaxPairs) return 0;
    return qmv::prefill_ws_layout(m->E, m->H, m->I, T, k).total;
}

int moe_expert_ffn_int4_prefill(const qmv_moe_int4 *m, const uint16_t *x_bf16, int T,
                                const int32_t *ids, const float *w, int k, float *out, void *ws,
                                size_t ws_bytes, qmv_stream_t stream) {
    int r = check_moe(m);
    if (r) return r;
    if (m->I % 128) return QMV_ESHAPE;
    if (T < 0 || k < 1 || k > m->E || (int64_t)T * k > kMaxPairs) return QMV_EINVAL;
    if (T == 0) return QMV_OK;
    if (!x_bf16 || !ids || !w || !out) return QMV_EINVAL;
    if (!aligned(x_bf16, 16) || !aligned(ids, 4) || !aligned(w, 4) || !aligned(out, 4))
        return QMV_EALIGN;
    const qmv::PrefillWorkspace L = qmv::prefill_ws_layout(m->E, m->H, m->I, T, k);
    if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return QMV_EWORKSPACE;
    const cudaStream_t st = cs(stream);
    const qmv::MoeDims d = dims(m);
    int32_t *status = at<int32_t>(ws, L.status);
    int32_t *offsets = at<int32_t>(ws, L.offsets), *list = at<int32_t>(ws, L.list);
    int32_t *uexp = at<int32_t>(ws, L.uexp), *n_used = at<int32_t>(ws, L.n_used);
    int32_t *pass_ofs = at<int32_t>(ws, L.pass_ofs);
    uint16_t *h = at<uint16_t>(ws, L.h);
    float *y = at<float>(ws, L.y);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    {
        // the grouping also writes the pass table, which the x packing reads
        qmv::PlanArgs pt{};
        pt.ptab = at<int4>(ws, L.ptab);
        if (e == cudaSuccess)
            e = qmv::launch_group_split(ids, T, k, m->E, offsets, list, uexp, n_used, pass_ofs,
                                        status, nullptr, m->H, nullptr, nullptr, st,
                                        qmv::prefill_pass_tokens(), false, nullptr, 0, false,
                                        nullptr, nullptr, nullptr, nullptr, nullptr, false, &pt);
    }
    if (qmv::tma_moe_supported(d)) {
        // tensor-map path: B operands packed per pass (x by a packing kernel,
        // h by the gate_up kernel itself)
        uint16_t *xp = at<uint16_t>(ws, L.xp), *hp = at<uint16_t>(ws, L.hp);
        if (e == cudaSuccess)
            e = qmv::launch_pack_x(x_bf16, m->H, k, list, n_used, at<int4>(ws, L.ptab), xp,
                                   L.pmax, st);
        if (e == cudaSuccess)
            e = qmv::launch_prefill(d, 0, xp, k, offsets, list, uexp, n_used, pass_ofs, hp, y,
                                    status, st, at<int4>(ws, L.ptab));
        if (e == cudaSuccess)
            e = qmv::launch_prefill(d, 1, hp, k, offsets, list, uexp, n_used, pass_ofs, hp, y,
                                    status, st, at<int4>(ws, L.ptab));
    } else {
        if (e == cudaSuccess)
            e = qmv::launch_prefill(d, 0, x_bf16, k, offsets, list, uexp, n_used, pass_ofs, h, y,
                                    status, st);
        if (e == cudaSuccess)
            e = qmv::launch_prefill(d, 1, h, k, offsets, list, uexp, n_used, pass_ofs, h, y,
                                    status, st);
    }
    if (e == cudaSuccess)  // ids and w are call inputs
        e = qmv::launch_combine(y, ids, w, T, k, m->E, m->H, out, st, true, nullptr, true);
    return from_cuda(e);
}

}  // extern "C"
