/*
 * qmv.h - C ABI of the GB300 (sm_103a) quantized matrix-vector library.
 *
 * Quantized formats (colibri PR #418 "Vulkan backend: expert tier + dense +
 * MLA attention on any Vulkan 1.2 GPU"):
 *   int4-gs64  two offset-binary nibbles per byte, value = nibble - 8
 *              (commit "opt-in Vulkan int4/int8 quantized GEMV"), element 2j
 *              in the LOW nibble of byte j and 2j+1 in the high nibble (the
 *              pages do not state the order; this is the library's reading),
 *              bytes in K order; one fp32 scale per 64 consecutive K values
 *              applied to that group's partial dot product (commit "grouped
 *              scales in the Vulkan kernels", fmt 4, group size 64).
 *              Weights [rows][K/2] uint8, scales [rows][K/64] fp32, row-major.
 *   int8-row   int8 weights [rows][K] with one fp32 scale per row (same
 *              GEMV commit, fmt 1).
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers (memory the caller allocated on
 *     the current CUDA device). The caller owns every buffer; the library
 *     never allocates, frees or synchronises.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and is complete when the stream is. Calls can be
 *     captured into CUDA graphs.
 *   - Arguments are validated on the host before anything is enqueued. On a
 *     nonzero return nothing was enqueued and no output was touched.
 *   - Shapes are row-major and contiguous. K, H and I must be multiples of 64.
 *   - Activations may have any finite fp32 value; each kernel rescales them
 *     by a power of two internally, which changes no result bit pattern beyond
 *     the stated tolerance.
 *   - Accuracy: the fp32 paths return y with
 *         |y - y_exact| <= 2e-5 * sum_k |w_k * x_k|
 *     per output (w the dequantized weight), the bf16 prefill path with 1e-2.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so CUDA callers pass their streams unchanged. */
typedef struct CUstream_st *qmv_stream_t;

typedef enum {
    QMV_OK = 0,
    QMV_EINVAL = -1,     /* null pointer, bad count, unsupported group size   */
    QMV_ESHAPE = -2,     /* a dimension is not a multiple of 64 or too large   */
    QMV_EWORKSPACE = -3, /* workspace pointer null, misaligned or too small    */
    QMV_ECUDA = -4,      /* a CUDA launch failed (see cudaGetLastError)        */
    QMV_ETIMEOUT = -5,   /* a bounded device-side wait gave up                 */
    QMV_EALIGN = -6      /* a pointer is not aligned as documented             */
} qmv_status;

/* Library version as 10000*major + 100*minor + patch. */
int qmv_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *qmv_status_str(int status);

/* Test hook, not part of the method: from the next launch on, the compute
 * warps of every odd CTA of the tensor-map MoE and dense kernels start `ns`
 * nanoseconds late (0 turns it off; negative values are taken as 0). Items
 * whose stages two CTAs share then meet every order of arrival, so tests can
 * check that the output does not depend on it. Process-wide, host only,
 * enqueues nothing; not thread-safe against concurrent launches. Returns the
 * previous value. */
int qmv_test_split_skew(int ns);

/* ---------------------------------------------------------------- GEMV */

/* Scratch needed by qmv_int4_gs / qmv_int8_row for S tokens of length K, in
 * bytes (a multiple of 256; 0 for unsupported sizes). It holds a status word
 * (the first int32, cleared by every call: bit 1 = a bounded device wait ran
 * out and y is not valid), counters and partial sums for row tiles shared
 * between thread blocks (about 4 MB, independent of K and S), and the
 * activations, converted into fp16 hi/lo fragments with one power-of-two
 * factor per 64-wide group before the weights are streamed. */
size_t qmv_gemv_workspace_bytes(int K, int S);

/* Dense int4 grouped-scale GEMV (colibri PR #418, commits "opt-in Vulkan
 * int4/int8 quantized GEMV" and "grouped scales in the Vulkan kernels"):
 *     y[s][i] = sum_g scales[i][g] * sum_{k in group g} (nibble(i,k) - 8) * x[s][k]
 *   wq      [N][K/2] uint8, 16-byte aligned
 *   scales  [N][K/gs] fp32, 4-byte aligned
 *   x       [S][K] fp32, 4-byte aligned
 *   y       [S][N] fp32 (written, fp32-accumulated)
 *   ws      device scratch of at least qmv_gemv_workspace_bytes(K, S) bytes,
 *           256-byte aligned, not shared with a concurrent call
 *   gs must be 64; K a multiple of 64; 1 <= N, 1 <= S, K <= 65536.
 * Up to 4 tokens whose activations fit 64 KB of fragments (S * K <= 16384)
 * run as one launch: every thread block converts x itself and streams its
 * 16-row tiles through per-warp cp.async rings, K split over the warps.
 * Otherwise, when N is a multiple of 16, K/64 a multiple of 4 and wq and
 * scales are 16-byte aligned, the weights stream through tensor-map (TMA)
 * copies with the row tiles' work shared evenly over all SMs; other shapes
 * use per-warp cp.async rings. All give the same results up to fp32
 * summation order.
 * Errors: QMV_EINVAL (null pointer, gs != 64, N or S < 1), QMV_ESHAPE (K),
 *         QMV_EALIGN, QMV_EWORKSPACE, QMV_ECUDA. */
int qmv_int4_gs(const uint8_t *wq, const float *scales, int N, int K, int gs, const float *x,
                float *y, int S, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* qmv_int4_gs with a bf16 output (colibri PR #418: the commit "vk_matmul_qt
 * routes a resident int4/int8 matmul_qt through coli_vk_matmul", whose dense
 * projections feed the next layer, and the rmsnorm / coli_vk_attn_qprep
 * chain that consumes them on the device; bf16 is the reading of the
 * activation type that chain passes on). The sum is formed exactly as in
 * qmv_int4_gs, in fp32, and each output is then rounded to the nearest bf16
 * value, ties to even:
 *   y_bf16  [S][N] bf16 bit patterns (uint16_t, 2-byte aligned; written)
 *   every other argument, the workspace and the errors as qmv_int4_gs.
 * For the same inputs and workspace size the result is the fp32 output of
 * qmv_int4_gs rounded to bf16, bit for bit. */
int qmv_int4_gs_bf16(const uint8_t *wq, const float *scales, int N, int K, int gs, const float *x,
                     uint16_t *y_bf16, int S, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* Two int4-gs64 GEMVs against the same activations (colibri PR #418, commit
 * "qmatmul staged-x length fix": matmul_pair stages x once for the q_a and
 * kv_a projections, 6144 -> (2048, 576), and records both in one submit):
 *     y0 = W0 x and y1 = W1 x, each exactly as qmv_int4_gs computes it
 *   wq0 [N0][K/2] and wq1 [N1][K/2] uint8, 16-byte aligned
 *   s0 [N0][K/gs], s1 [N1][K/gs] fp32; x [S][K]; y0 [S][N0]; y1 [S][N1] fp32
 *   ws      device scratch of at least qmv_gemv_workspace_bytes(K, S) bytes
 *           (the same as one GEMV), 256-byte aligned
 * x is converted into fp16 hi/lo fragments once. For up to 4 tokens with
 * S * K <= 16384 (see qmv_int4_gs) the row tiles of both matrices are one
 * work sequence of the single-launch kernel; otherwise, when both matrices
 * qualify for the tensor-map path, of one tensor-map launch; otherwise the
 * two GEMVs run one after the other (the status word then reports the second).
 * Errors: as qmv_int4_gs. */
int qmv_int4_gs_pair(const uint8_t *wq0, const float *s0, int N0, const uint8_t *wq1,
                     const float *s1, int N1, int K, int gs, const float *x, float *y0, float *y1,
                     int S, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* Dense int3-g64 GEMV over two-plane rows (colibri PR #418, the fmt-5
 * commit: 24 bytes per 64-group, lanes striding the 16-value low-plane words,
 * the high-plane word pre-shifted to bit 0, group scales applied to the word
 * partials). The pages name the planes but print no byte; the layout read
 * here: in each 24-byte group, bytes 0..15 hold 2 low bits per element
 * (element e at bits 2(e%4) of byte e/4) and bytes 16..23 one high bit per
 * element (bit e%8 of byte 16 + e/8); code = low | high << 2, value = code - 4.
 *     y[s][i] = sum_g scales[i][g] * sum_{k in group g} (code(i,k) - 4) * x[s][k]
 *   wq3     [N][K/64 * 24] uint8, 4-byte aligned
 *   scales  [N][K/gs] fp32, 4-byte aligned
 *   x       [S][K] fp32, 16-byte aligned
 *   y       [S][N] fp32 (written, fp32-accumulated)
 *   gs must be 64; K a multiple of 64; 1 <= N, 1 <= S, K <= 65536. No
 *   workspace: on the CUDA cores, each warp walks its rows and decodes each
 *   32-bit low-plane word once for up to 4 tokens; x is staged per CTA in up
 *   to 96 KB of shared memory (read from global memory when K > 24576).
 * Errors: QMV_EINVAL, QMV_ESHAPE (K), QMV_EALIGN, QMV_ECUDA. */
int qmv_int3_gs(const uint8_t *wq3, const float *scales, int N, int K, int gs, const float *x,
                float *y, int S, qmv_stream_t stream);

/* Dense int8 per-row-scale GEMV (same commit, fmt 1):
 *     y[s][i] = row_scale[i] * sum_k w[i][k] * x[s][k]
 *   w [N][K] int8 (16-byte aligned), row_scale [N] fp32, x [S][K] fp32, y [S][N] fp32,
 *   ws as for qmv_int4_gs. K a multiple of 64, K <= 65536; N, S >= 1.
 *   Errors as qmv_int4_gs. */
int qmv_int8_row(const int8_t *w, const float *row_scale, int N, int K, const float *x,
                 float *y, int S, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* qmv_int8_row with a bf16 output (as qmv_int4_gs_bf16): the fp32 result of
 * qmv_int8_row rounded to the nearest bf16, ties to even, into
 *   y_bf16  [S][N] bf16 bit patterns (uint16_t, 2-byte aligned; written);
 *   every other argument, the workspace and the errors as qmv_int8_row. */
int qmv_int8_row_bf16(const int8_t *w, const float *row_scale, int N, int K, const float *x,
                      uint16_t *y_bf16, int S, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* The dense int4-gs64 GEMV of qmv_int4_gs for callers that cannot allocate
 * device memory: code that must never make the device synchronise (cudaMalloc
 * and cudaFree can), hosts that forbid device allocation after start-up, and
 * C callers with nowhere to keep a workspace between calls. Same arguments as
 * qmv_int4_gs, minus the workspace, and the same results up to the order of
 * the fp32 additions: it always runs the per-warp cp.async kernel, never the
 * tensor-map kernel that qmv_int4_gs takes when N % 16 == 0, so results are
 * not bit-identical to qmv_int4_gs and its speed differs on such shapes. The
 * pages have no counterpart of this entry point.
 *   Scratch: one file-scope device array inside the library (266,240 bytes,
 *   held by every GPU that loads the library until the process exits), so
 *   S * K must be at most 65536; larger calls return QMV_EWORKSPACE and
 *   enqueue nothing.
 *   Every call looks up the array's device address in the current context (a
 *   host call, cudaGetSymbolAddress), so a device reset does not leave a stale
 *   address behind. The first call on a device may load the library's module
 *   there, which allocates the array and can synchronise: make one call per
 *   device at start-up, before any stream capture and before any code that
 *   must not synchronise.
 *   Every call uses the same array and overwrites all of it that it reads, so
 *   nothing carries over between calls, but calls whose work overlaps on the
 *   GPU (different streams, or different host threads on one device) race on
 *   it: order them on one stream.
 *   Allocates nothing itself: no cudaMalloc, cudaFree or allocating library
 *   call. */
int qmv_int4_gs_noalloc(const uint8_t *wq, const float *scales, int N, int K, int gs,
                        const float *x, float *y, int S, qmv_stream_t stream);

/* ---------------------------------------------------------------- MoE */

/* Device-resident int4-gs64 expert weights (the analogue of the pages'
 * uploaded-once weight handle). All experts live in one pool each:
 *   gu_q [E][2I][H/2] uint8: gate rows 0..I-1, then up rows I..2I-1 (reading:
 *        the pages fuse gate and up but do not state the stacking order)
 *   gu_s [E][2I][H/64] fp32
 *   dn_q [E][H][I/2] uint8, dn_s [E][H][I/64] fp32
 * The descriptor itself is a HOST struct; it is read during the call only. */
typedef struct {
    const uint8_t *gu_q;
    const float *gu_s;
    const uint8_t *dn_q;
    const float *dn_s;
    int32_t E, H, I, gs;
} qmv_moe_int4;

/* Top-k routing: for each token, the k experts with the largest logits
 * (fp32 comparison; equal logits keep the lower expert index first), in
 * descending logit order, with weights = softmax over all experts restricted
 * to the chosen k and renormalised to sum to one (equivalently
 * exp(l_e - l_max) / sum over the chosen). NaN logits are never chosen
 * ahead of finite ones.
 *   logits [T][E] fp32; ids [T][k] int32 (written); w [T][k] fp32 (written).
 *   1 <= k <= min(E, 32), E <= 1024, T >= 0 (T == 0 enqueues nothing). */
int moe_route_topk(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                   qmv_stream_t stream);

/* Token -> expert grouping (so each expert's weights are read once per batch,
 * colibri PR #418 "coli_vk_expert_group"). Pair p = t*k + j.
 *   offsets [E+1] int32: exclusive prefix sum of the per-expert pair counts
 *   list    [T*k] int32: pair ids grouped by expert, ascending inside a group
 *   uexp    [E]   int32: the experts with at least one pair, ascending
 *   n_used  [1]   int32: how many entries of uexp are valid
 *   status  [1]   int32: OR-ed with 1 when an id is outside [0, E); such a
 *                 pair is left out of every list. Not cleared by this call.
 *   T*k <= 1 << 20, E <= 1024. */
int moe_group(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *list,
              int32_t *uexp, int32_t *n_used, int32_t *status, qmv_stream_t stream);

/* Fused gate+up with SiLU*mul for every grouped pair (colibri PR #418,
 * commit "qmatmul_gate_up.comp + coli_vk_gate_up"): for each expert e in
 * uexp and each pair p = t*k + j routed to e,
 *     h[p][c] = SiLU(gate_e[c] . x[t]) * (up_e[c] . x[t]),   SiLU(g) = g / (1 + e^-g)
 *   x [T][H] fp32; h [T*k][I] fp32 (rows of pairs that no expert serves are
 *   left untouched). offsets/list/uexp/n_used as written by moe_group.
 *   ws: device scratch of at least moe_workspace_bytes(m, T, k) bytes,
 *   256-byte aligned (the activations are converted into it first). */
int moe_gate_up_silu(const qmv_moe_int4 *m, const float *x, int T, int k,
                     const int32_t *offsets, const int32_t *list, const int32_t *uexp,
                     const int32_t *n_used, float *h, void *ws, size_t ws_bytes,
                     qmv_stream_t stream);

/* Down projection of every grouped pair (colibri PR #418, "coli_vk_expert_group"):
 *     y[p][i] = down_e[i] . h[p]          y [T*k][H] fp32 (pairs not served: untouched)
 * and the weighted combine (PR #1338, weighted accumulation of expert outputs):
 *     out[t][i] = sum_{j < k, ids[t][j] valid} w[t][j] * y[t*k + j][i]
 *   summed in slot order, so results are deterministic. out [T][H] fp32.
 *   moe_down takes the same workspace as moe_gate_up_silu. moe_combine reads
 *   ids to skip pairs whose id is outside [0, E). */
int moe_down(const qmv_moe_int4 *m, const float *h, int T, int k, const int32_t *offsets,
             const int32_t *list, const int32_t *uexp, const int32_t *n_used, float *y,
             void *ws, size_t ws_bytes, qmv_stream_t stream);
int moe_combine(const float *y, const int32_t *ids, const float *w, int T, int k, int E, int H,
                float *out, qmv_stream_t stream);

/* Workspace of the MoE entry points that take one, in bytes (256-byte aligned segments). */
size_t moe_workspace_bytes(const qmv_moe_int4 *m, int T, int k);

/* Whole MoE expert FFN for a decode micro-batch (colibri PR #418,
 * "coli_vk_expert_group": fused gate+up+SiLU, then down, hidden kept on the
 * device; PR #1338: weighted accumulation). Equivalent to moe_group,
 * moe_gate_up_silu, moe_down and moe_combine in sequence:
 *     out[t] = sum_j w[t][j] * down_e(SiLU(gate_e x[t]) * up_e x[t]),  e = ids[t][j]
 *   x [T][H] fp32, ids [T][k] int32, w [T][k] fp32, out [T][H] fp32.
 *   ws: device workspace of at least moe_workspace_bytes(m, T, k) bytes,
 *   256-byte aligned, owned by the caller, not shared between concurrent calls.
 *   The first int32 of ws is a device status word, cleared at the start of
 *   the call: bit 0 = an id outside [0, E) (that pair skipped, as moe_group),
 *   bit 1 = a bounded wait on the weight stream ran out (out not valid).
 *   One token (T == 1) with moe_one_token_path(m, k) == 1 runs as a single
 *   cooperative kernel (all CTAs resident, one grid-wide barrier between
 *   gate+up and down); the result is the same. */
int moe_expert_ffn_int4(const qmv_moe_int4 *m, const float *x, int T, const int32_t *ids,
                        const float *w, int k, float *out, void *ws, size_t ws_bytes,
                        qmv_stream_t stream);

/* Routing and expert FFN of a decode micro-batch in one call: moe_route_topk
 * on logits [T][E] (ids [T][k] and w [T][k] are written, as that call writes
 * them), then moe_expert_ffn_int4 with those ids and weights; same
 * workspace, limits and status word (1 <= k <= min(E, 32)). With one token
 * and moe_one_token_path(m, k) == 1 the routing runs inside the
 * single-launch FFN kernel (every thread block routes the token itself; the
 * first writes ids and w), so the call is one kernel after the status clear.
 * With 2..32 tokens on the tensor-map path the grouping kernel routes the
 * tokens itself the same way, which saves the routing launch.
 * Errors: those of moe_route_topk and moe_expert_ffn_int4. */
int moe_route_expert_ffn_int4(const qmv_moe_int4 *m, const float *logits, const float *x, int T,
                              int k, int32_t *ids, float *w, float *out, void *ws, size_t ws_bytes,
                              qmv_stream_t stream);

/* moe_expert_ffn_int4 over the resident experts only (colibri PR #418,
 * "Vulkan expert tier ... overlapped with CPU rows": the GPU computes the
 * experts of its registry while the CPU computes the rest; PR #1338,
 * "Validation": a miss returns no mask bit):
 *     out[t] = sum over served slots j of w[t][j] * down_e(SiLU(gate_e x[t]) * up_e x[t])
 *     served[t][j] = 1 if e = ids[t][j] is in [0, E) and bit e % 32 of
 *                    resident[e / 32] is set, else 0
 *   resident  device bitmap [ceil(E / 32)] uint32, 4-byte aligned
 *   served    device [T][k] uint8, written
 *   others and the workspace as moe_expert_ffn_int4. A token with no served
 *   slot gets out[t] = 0. The caller adds the unserved slots' terms itself.
 *   A non-resident id is not an error; status bit 0 still flags ids outside
 *   [0, E). Errors: those of moe_expert_ffn_int4, plus QMV_EINVAL for a null
 *   resident or served and QMV_EALIGN for a misaligned resident. */
int moe_expert_ffn_int4_resident(const qmv_moe_int4 *m, const uint32_t *resident, const float *x,
                                 int T, const int32_t *ids, const float *w, int k, float *out,
                                 uint8_t *served, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* The four phases of moe_expert_ffn_int4, for callers that interleave other
 * work or time the phases (the pages split their expert group the same way
 * into issue and take). All four take the same workspace; each phase reads
 * what the previous one left there, so they must run in this order on one
 * stream, with T and k unchanged:
 *   moe_ffn_prepare  clears the status word, groups the pairs (moe_group) and
 *                    converts x into fp16 hi/lo cells with per-group factors;
 *   moe_ffn_gate_up  h = SiLU(gate x) * up x for every served pair, kept in the
 *                    workspace both as fp32 and as cells for the down pass;
 *   moe_ffn_down     y = down h per pair, in the workspace;
 *   moe_ffn_combine  out[t] = sum_j w[t][j] * y[t*k + j], slot order. */
int moe_ffn_prepare(const qmv_moe_int4 *m, const float *x, int T, const int32_t *ids, int k,
                    void *ws, size_t ws_bytes, qmv_stream_t stream);
int moe_ffn_gate_up(const qmv_moe_int4 *m, int T, int k, void *ws, size_t ws_bytes,
                    qmv_stream_t stream);
int moe_ffn_down(const qmv_moe_int4 *m, int T, int k, void *ws, size_t ws_bytes,
                 qmv_stream_t stream);
int moe_ffn_combine(const qmv_moe_int4 *m, const int32_t *ids, const float *w, int T, int k,
                    float *out, void *ws, size_t ws_bytes, qmv_stream_t stream);

/* Which weight stream the decode gate+up and down kernels of this descriptor
 * use (no counterpart on the pages; it names the kernel a profile shows):
 *   1  tensor-map bulk copies (TMA) into an mbarrier-guarded ring, taken when
 *      H/64 and I/64 are multiples of 4 and the four pools are 16-byte aligned;
 *   0  per-warp cp.async rings otherwise.
 * Both compute the same result. Host only, enqueues nothing.
 * Errors: those of the descriptor check shared by every MoE call (QMV_EINVAL,
 * QMV_ESHAPE, QMV_EALIGN). */
int moe_weight_path(const qmv_moe_int4 *m);

/* Whether moe_expert_ffn_int4 with T == 1 and this k runs the single-launch
 * kernel (1) or the grouped phases (0). The single launch is taken when the
 * weight pools suit the tensor-map path (moe_weight_path == 1), H and I are
 * multiples of 256, 1 <= k <= 32, and one CTA's share of the layer's weights
 * fits in its shared memory. No counterpart on the pages; it names the kernel
 * a profile shows. Host only, enqueues nothing.
 * Errors: those of the descriptor check shared by every MoE call. */
int moe_one_token_path(const qmv_moe_int4 *m, int k);

/* Workspace of moe_expert_ffn_int4_prefill, in bytes (0 for unsupported sizes). */
size_t moe_prefill_workspace_bytes(const qmv_moe_int4 *m, int T, int k);

/* Batched MoE prefill on the tcgen05 tensor cores (colibri PR #418 PR summary
 * names cooperative-matrix prefill kernels as the next step for batched
 * prompts; the math is that of moe_expert_ffn_int4):
 *     out[t] = sum_j w[t][j] * down_e(SiLU(gate_e x[t]) * up_e x[t]),  e = ids[t][j]
 * with bf16 operands and fp32 accumulation: the weights are dequantized to
 * bf16 with their group scale folded in, h is rounded to bf16 between the two
 * projections; expected accuracy |out - exact| <= 1e-2 * sum |w * down * h|.
 *   x_bf16 [T][H] bfloat16 bit patterns, 16-byte aligned; ids [T][k] int32;
 *   w [T][k] fp32; out [T][H] fp32.
 *   Each expert's tokens are processed in passes of up to 64, each pass
 *   reading the expert's weights once. I must be a multiple of 128.
 *   ws: at least moe_prefill_workspace_bytes(m, T, k) bytes, 256-byte aligned;
 *   its first int32 is a status word: bit 0 = an id outside [0, E) (pair
 *   skipped), bit 1 = a tensor-core wait timed out (output not valid). */
int moe_expert_ffn_int4_prefill(const qmv_moe_int4 *m, const uint16_t *x_bf16, int T,
                                const int32_t *ids, const float *w, int k, float *out, void *ws,
                                size_t ws_bytes, qmv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
