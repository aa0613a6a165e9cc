// qmv_internal.h - launchers behind the C ABI (host side, no validation here:
// the ABI layer checks every argument before calling these).
#pragma once

#include <cuda.h>

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "qmv_layout.h"

namespace qmv {

// Dense GEMV, any S (passes of up to 16 tokens). scratch: dense_scratch_bytes(K, S).
size_t dense_scratch_bytes(int K, int S);
cudaError_t launch_dense_int4(const uint8_t *wq, const float *scales, int N, int K,
                              const float *x, float *y, int S, void *scratch, cudaStream_t st);
cudaError_t launch_dense_int8(const int8_t *w, const float *row_scale, int N, int K,
                              const float *x, float *y, int S, void *scratch, cudaStream_t st);

// The GEMV entry points' workspace (status word, split counters, activation
// units, partial sums): gemv_ws_bytes(K, S) bytes. int4 runs on the
// tensor-map kernel (qmv_moe_tma.cu, dense mode) when tma_dense_supported().
size_t gemv_ws_bytes(int K, int S);
// ybf (optional): write y rounded to bf16 there instead of fp32 into y.
cudaError_t launch_gemv_int4(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                             float *y, int S, void *ws, cudaStream_t st, uint16_t *ybf = nullptr);
cudaError_t launch_gemv_int8(const int8_t *w, const float *row_scale, int N, int K,
                             const float *x, float *y, int S, void *ws, cudaStream_t st,
                             uint16_t *ybf = nullptr);
// int3-g64 two-plane rows [N][K/64 * 24 bytes], fp32 x [S][K] (16-byte aligned).
cudaError_t launch_gemv_int3(const uint8_t *wq, const float *scales, int N, int K, const float *x,
                             float *y, int S, cudaStream_t st);
// The same on the warp MMA in one launch (k_int3_ks_x), for up to 4 tokens,
// K a multiple of 256, 16-byte aligned rows and x's units within 64 KB.
bool int3_one_launch(const uint8_t *wq, int K, int S);
cudaError_t launch_gemv_int3_mma(const uint8_t *wq, const float *scales, int N, int K,
                                 const float *x, float *y, int S, cudaStream_t st);
// Two int4 GEMVs against the same x: one activation split; one launch when
// both matrices take the tensor-map kernel, else two.
cudaError_t launch_gemv_int4_pair(const uint8_t *wq0, const float *s0, int N0, const uint8_t *wq1,
                                  const float *s1, int N1, int K, const float *x, float *y0,
                                  float *y1, int S, void *ws, cudaStream_t st);

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
// Work plan of the tensor-map FFN kernels, written by the grouping kernel
// (ptab == null: none). A pass is up to kMaxTok pairs of one expert; the CTAs
// of gate+up (and of down) split the passes' stages so that every CTA gets
// the same cost: a stage with at most 4 tokens costs kPlanW1, one with more
// kPlanW2 (its MMAs cover two token blocks), and the end of every item (a
// row tile's last stage: its epilogue) kPlanItem more.
constexpr int kPlanW1 = 3, kPlanW2 = 4, kPlanItem = 4;
struct PlanArgs {
    int4 *ptab;        // [passes]: (expert, first list index, tokens, 0)
    int4 *plan_gu;     // [g + 1]: (first stage of each gate+up CTA, then the total;
                       //  and the expert, first list index and tokens of the pass
                       //  holding that stage), so a CTA starts with one load
    int4 *plan_dn;     // [g + 1]: the same for down
    int s_gu, s_dn;    // stages per pass: row tiles x stages per tile
    int ns_gu, ns_dn;  // stages per row tile (an item)
    int g;             // CTAs of the tensor-map kernel
};
// CTAs of a tensor-map decode launch.
int tma_grid();
// Test hook of the tensor-map kernel's split items: the consumers of odd CTAs
// start this many ns late (0: off). Set through qmv_test_split_skew.
extern int g_split_skew_ns;

// Grouping plus the split of the T activation rows, in one launch (with
// logits: routing too, ids / w then written to ids_out / w_out). With
// packed == true the units go to the pass-packed layout (see MoeWorkspace)
// instead of per-row cells; zero[0 .. nzero) is cleared first; pdl: launched
// with programmatic dependent launch. Per-row cells are in the tensor-map
// kernel's int4 form when sub == true (see launch_split); packed units always are.
cudaError_t launch_group_split(const int32_t *ids, int T, int k, int E, int32_t *offsets,
                               int32_t *list, int32_t *uexp, int32_t *n_used, int32_t *pass_ofs,
                               int32_t *status, const float *x, int H, void *xcells, float *xfac,
                               cudaStream_t st, int pass_tok = 8, bool packed = false,
                               int32_t *zero = nullptr, int nzero = 0, bool pdl = false,
                               const uint32_t *res = nullptr, uint8_t *served = nullptr,
                               const float *logits = nullptr, int32_t *ids_out = nullptr,
                               float *w_out = nullptr, bool sub = false,
                               const PlanArgs *plan = nullptr);
// Shared memory of the grouping kernel when it also routes (logits != null):
// every CTA routes the T tokens itself, so T * k pairs and E logits a warp.
size_t route_smem_bytes(int T, int E, int k);
size_t group_smem_bytes(int E);  // the grouping's per-warp expert counts, 32 x E ints
cudaError_t launch_passes(const int32_t *offsets, const int32_t *uexp, const int32_t *n_used,
                          int32_t *pass_ofs, cudaStream_t st, bool pdl);
// Activation rows [R][K] fp32 -> fragment cells [R][K/64][16] uint4 + factors [R][K/64],
// or, with sub == true, the tensor-map kernel's int4 form: cells with the
// high-nibble values divided by 16 and records (factor, offset_init) [R][K/64][2].
cudaError_t launch_split(const float *v, int R, int K, void *cells, float *fac, cudaStream_t st,
                         bool sub = false);
cudaError_t launch_gate_up(const MoeDims &m, const void *xcells, const float *xfac, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hcells,
                           float *hfac, cudaStream_t st);
cudaError_t launch_down(const MoeDims &m, const void *hcells, const float *hfac,
                        const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                        const int32_t *n_used, const int32_t *pass_ofs, float *y, cudaStream_t st);
// early (with pdl): ids, w and res were written before the previous kernel
// started (call inputs, or written by a kernel at least two launches back),
// so the combine reads them before it waits for y.
cudaError_t launch_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E,
                           int H, float *out, cudaStream_t st, bool pdl,
                           const uint32_t *res = nullptr, bool early = false);

// Prefill (tcgen05): mode 0 = gate+up+SiLU (B = x bf16 rows, writes h bf16),
// mode 1 = down (B = h bf16 rows, writes y fp32). Passes of prefill_pass_tokens().
// ptab: the grouping kernel's pass table, or null (then the passes are found
// through pass_ofs, uexp and offsets).
cudaError_t launch_prefill(const MoeDims &m, int mode, const uint16_t *b, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, uint16_t *h, float *y,
                           int32_t *status, cudaStream_t st, const int4 *ptab = nullptr);
int prefill_pass_tokens();
// Tensor-map prefill (tma_moe_supported shapes): B operands packed per pass,
// [pass][K/64][64 rows][64 bf16], 128-byte swizzled, rows beyond the pass's
// tokens zero. launch_pack_x packs x; the gate_up launch writes h packed
// (argument h) and down reads it (argument b).
cudaError_t launch_pack_x(const uint16_t *x, int H, int k, const int32_t *list,
                          const int32_t *n_used, const int4 *ptab, uint16_t *xp, int pmax,
                          cudaStream_t st);

// TMA-fed decode kernels (qmv_moe_tma.cu): mode 0 = gate+up (cells = x units,
// writes h, h units, h factors), mode 1 = down (cells = h units, writes y).
// The weight stages of all items are shared out evenly over the CTAs; an item
// split between CTAs leaves partial sums in `part` and the last CTA to finish
// it (counted in cnt, which must be zero at launch and is zero again after
// the kernel) adds them and writes the item.
// P: the call's token-expert pairs (0: shape and alignment only).
bool tma_moe_supported(const MoeDims &m, long long P = 0);
// 3-D tensor maps of a weight pool [E][rows][K/2] (box 128 B x box_rows rows,
// 128-byte swizzle) and of its scales [E][rows][K/64] (box 4 x box_rows rows).
bool encode_weight_maps(CUtensorMap *wmap, CUtensorMap *smap, const uint8_t *wq, const float *ws,
                        int E, int rows, int K, int box_rows = 128);
bool tma_dense_supported(const uint8_t *wq, const float *scales, int N, int K, int S);
// A row-major byte matrix [rows][row_bytes] as a 3-D tensor map (128 bytes,
// row, 128-byte chunk), boxes of box_rows whole rows with the 128-byte
// swizzle (in shared memory: [chunk][row][128 B], 16-byte units XOR-ed with
// the row mod 8). row_bytes a multiple of 128, at most 32768.
bool encode_rows_swizzled(CUtensorMap *map, const uint8_t *base, long long rows, int row_bytes,
                          int box_rows);
// wq2 != null: a second matrix [N2][K/2] against the same activations, its
// row tiles after the first's in the same launch, output y2 [S][N2].
cudaError_t launch_dense_tma(const uint8_t *wq, const float *scales, int N, int K, int S,
                             const void *cells, const float *cfac, float *y, int32_t *status,
                             int32_t *cnt, float *part, cudaStream_t st,
                             const uint8_t *wq2 = nullptr, const float *scales2 = nullptr,
                             int N2 = 0, float *y2 = nullptr, uint16_t *ybf = nullptr);
// packed: the activation units (cells, cfac) and, for gate+up, the units of
// h it writes (hcells, hfac) are in the pass-packed layout; else per row.
// ptab / plan (optional): the grouping kernel's pass table and this mode's
// CTA stage boundaries (PlanArgs); without them the kernel splits the stages
// evenly and walks the passes through pass_ofs.
cudaError_t launch_moe_tma(const MoeDims &m, int mode, const void *cells, const float *cfac, int k,
                           const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                           const int32_t *n_used, const int32_t *pass_ofs, float *h, void *hcells,
                           float *hfac, float *y, int32_t *status, int32_t *cnt, float *part,
                           cudaStream_t st, bool packed = false, const int4 *ptab = nullptr,
                           const int4 *plan = nullptr);

// Single-launch expert FFN of one token (cooperative grid, qmv_moe_one.cu);
// it clears the status word itself.
bool moe_one_supported(const MoeDims &m, int k);
cudaError_t launch_moe_one(const MoeDims &m, const float *x, const int32_t *ids, const float *w,
                           int k, float *h, float *out, int32_t *status,
                           cudaStream_t st, const uint32_t *res = nullptr,
                           uint8_t *served = nullptr, const float *logits = nullptr,
                           int32_t *ids_out = nullptr, float *w_out = nullptr);

// Workspace layout of the MoE entry points (256-byte aligned segments). The
// status word and the split counters (kSkMaxCtas for gate+up, then kSkMaxCtas
// for down) are adjacent, so one memset of status_bytes clears them all.
// Pass-packed activation units (kPackedStage blocks, qmv_layout.h): xpk
// holds x for gate+up, hpk h for down.
struct MoeWorkspace {
    size_t status, sk_cnt, status_bytes, offsets, list, uexp, n_used, pass_ofs, xcells, xfac, h,
        hcells, hfac, y, sk_part, xpk, hpk, ptab, plan, total;
    int pmax;  // passes, at most
};
MoeWorkspace moe_ws_layout(int E, int H, int I, int T, int k);

struct PrefillWorkspace {
    size_t status, offsets, list, uexp, n_used, pass_ofs, ptab, h, y, xp, hp, total;
    int pmax;  // passes, at most
};
PrefillWorkspace prefill_ws_layout(int E, int H, int I, int T, int k);

}  // namespace qmv
