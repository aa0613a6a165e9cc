/*
 * qmv_oracle.c - plain, slow, fp64 CPU oracle for the int4-gs64 / int8
 * quantized GEMV and the MoE expert FFN built on it.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The CUDA library shares
 * no code, header, table or constant with it, and neither includes the other.
 *
 * Sources (the pages are pull-request threads of the "colibri" engine):
 *  [PR418]  colibri PR #418 "Vulkan backend: expert tier + dense + MLA
 *           attention on any Vulkan 1.2 GPU" - commit messages:
 *             "opt-in Vulkan int4/int8 quantized GEMV" (int4 decodes as
 *               nibble - 8, offset binary; int8 with a per-row scale),
 *             "qmatmul_gate_up.comp + coli_vk_gate_up" (hidden =
 *               silu(gate(x)) * up(x), x read once for both),
 *             "coli_vk_expert_group" (K experts: fused gate+up+silu, then
 *               down, hidden kept on the device),
 *             "grouped scales in the Vulkan kernels" (fmt 4: one scale per
 *               gs inputs applied to the packed-word partial; gs a multiple
 *               of 8 so a word never straddles a group),
 *             PR summary, "Correctness" (CPU-reference exactness harness).
 *  [PR1338] colibri PR #1338 "qwen36: Vulkan expert tier, and staged
 *           device-local uploads" - the fake-Vulkan gate comment (int4-gs64
 *           arrives as fmt 4 / grp 64 at half a byte per element; the
 *           weighted accumulation of expert outputs is checked lane by lane).
 *
 * Readings where the pages are silent:
 *  R1 nibble order: element 2j of a row is the LOW nibble of byte j,
 *     element 2j+1 the HIGH nibble; bytes run in K order.
 *  R2 scales are fp32, row-major [rows][K/gs].
 *  R3 the stacked gate+up tensor holds gate rows 0..I-1, then up rows I..2I-1.
 *  R4 routing: softmax over all experts, select the k largest logits (fp32
 *     compare, the lower expert index wins a tie), renormalise the selected
 *     probabilities to sum to one. A NaN logit counts as -inf: it is never
 *     chosen ahead of a finite logit and, when chosen, weighs exp(-inf) = 0.
 *     If every logit of a token is -inf or NaN they are all equal, so the k
 *     lowest indices are chosen with weight 1/k each.
 *  R5 SiLU(g) = g * sigma(g), sigma(g) = 1 / (1 + exp(-g)).
 *  R6 int3-g64 two-plane rows ([PR418] "fmt 5", the 24-byte-per-64-group
 *     layout whose lanes stride 16-value low-plane words and whose
 *     high-plane word is pre-shifted to bit 0): a row is K/64 groups of 24
 *     bytes; bytes 0..15 of a group are the low plane, 2 bits per element
 *     (element e in bits 2(e%4), 2(e%4)+1 of byte e/4: 16 elements to a
 *     little-endian 32-bit word), bytes 16..23 the high plane, 1 bit per
 *     element (element e in bit e%8 of byte 16 + e/8). code = low | high << 2
 *     and the value is code - 4 (offset binary, as int4's nibble - 8); one
 *     fp32 scale per group, row-major [rows][K/64]. The pages print no byte
 *     of this layout; this is the plainest reading of the words they name.
 *
 * Every accumulation is in double. No blocking, fusion or reordering beyond
 * the definitions: parallel loops only split independent outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ threads */

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------ a1: nibble decode [PR418] */

/* Offset-binary nibble of element k of a packed row (reading R1). */
static inline int orc_nibble(const uint8_t *row, int64_t k) {
    return (row[k >> 1] >> ((k & 1) * 4)) & 0xF;
}

/* vals[k] = nibble(k) - 8, in [-8, 7]. */
void orc_unpack_int4(const uint8_t *bytes, int64_t n_vals, int8_t *vals) {
    for (int64_t k = 0; k < n_vals; ++k) vals[k] = (int8_t)(orc_nibble(bytes, k) - 8);
}

/* Inverse of orc_unpack_int4 for vals in [-8, 7]; n_vals must be even.
 * Returns -1 (and writes nothing further) on an out-of-range value. */
int orc_pack_int4(const int8_t *vals, int64_t n_vals, uint8_t *bytes) {
    if (n_vals & 1) return -1;
    for (int64_t j = 0; j < n_vals / 2; ++j) {
        int lo = vals[2 * j], hi = vals[2 * j + 1];
        if (lo < -8 || lo > 7 || hi < -8 || hi > 7) return -1;
        bytes[j] = (uint8_t)(((lo + 8) & 0xF) | (((hi + 8) & 0xF) << 4));
    }
    return 0;
}

/* Dequantized element (i, k): (nibble - 8) * s[i][k / gs], exact in double. */
static inline double orc_deq(const uint8_t *wq, const float *s, int K, int gs, int64_t i,
                             int64_t k) {
    const uint8_t *row = wq + i * (int64_t)(K / 2);
    return (double)(orc_nibble(row, k) - 8) * (double)s[i * (int64_t)(K / gs) + k / gs];
}

/* W[N][K] = explicitly dequantized matrix (input to form (ii)). */
void orc_dequant_int4(const uint8_t *wq, const float *s, int N, int K, int gs, double *W) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t k = 0; k < K; ++k) W[i * K + k] = orc_deq(wq, s, K, gs, i, k);
}

/* ------------------------------- a2: int4 grouped-scale GEMV [PR418 fmt 4] */

/* Form (i), as the pages describe it: for every group, the partial dot of the
 * decoded nibbles with x, then multiplied by that group's scale.
 *   y[t][i] = sum_g s[i][g] * sum_{k in g} (nibble(i,k) - 8) * x[t][k]   */
void orc_qmv_int4_gs(const uint8_t *wq, const float *s, int N, int K, int gs, const float *x,
                     int S, double *y) {
    int G = K / gs;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < S; ++t)
        for (int64_t i = 0; i < N; ++i) {
            const uint8_t *row = wq + i * (int64_t)(K / 2);
            const float *xt = x + t * (int64_t)K;
            double acc = 0.0;
            for (int g = 0; g < G; ++g) {
                double part = 0.0;
                for (int64_t k = (int64_t)g * gs; k < (int64_t)(g + 1) * gs; ++k)
                    part += (double)(orc_nibble(row, k) - 8) * (double)xt[k];
                acc += (double)s[i * G + g] * part;
            }
            y[t * N + i] = acc;
        }
}

/* Normalising denominator of the tolerance: den[t][i] = sum_k |deq(i,k) * x[t][k]|. */
void orc_qmv_int4_gs_absden(const uint8_t *wq, const float *s, int N, int K, int gs,
                            const float *x, int S, double *den) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < S; ++t)
        for (int64_t i = 0; i < N; ++i) {
            double a = 0.0;
            for (int64_t k = 0; k < K; ++k)
                a += fabs(orc_deq(wq, s, K, gs, i, k) * (double)x[t * (int64_t)K + k]);
            den[t * N + i] = a;
        }
}

/* Form (ii): plain matvec over an explicitly dequantized fp64 matrix. */
void orc_matvec_f64(const double *W, int N, int K, const float *x, int S, double *y) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < S; ++t)
        for (int64_t i = 0; i < N; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += W[i * K + k] * (double)x[t * (int64_t)K + k];
            y[t * N + i] = acc;
        }
}

/* --------------------------- f2: int3-g64 two-plane GEMV [PR418 fmt 5, R6] */

/* 3-bit code (0..7) of element k of a packed row (reading R6). */
static inline int orc_code3(const uint8_t *row, int64_t k) {
    const uint8_t *g = row + (k / 64) * 24;
    const int e = (int)(k % 64);
    const int lo = (g[e / 4] >> (2 * (e % 4))) & 3;
    const int hi = (g[16 + e / 8] >> (e % 8)) & 1;
    return lo | (hi << 2);
}

/* vals[k] = code(k) - 4, in [-4, 3]; n_vals a multiple of 64 (one row). */
void orc_unpack_int3(const uint8_t *bytes, int64_t n_vals, int8_t *vals) {
    for (int64_t k = 0; k < n_vals; ++k) vals[k] = (int8_t)(orc_code3(bytes, k) - 4);
}

/* Inverse of orc_unpack_int3 for vals in [-4, 3]; n_vals a multiple of 64.
 * Returns -1 on a bad count or value. */
int orc_pack_int3(const int8_t *vals, int64_t n_vals, uint8_t *bytes) {
    if (n_vals % 64) return -1;
    memset(bytes, 0, (size_t)(n_vals / 64) * 24);
    for (int64_t k = 0; k < n_vals; ++k) {
        const int v = vals[k];
        if (v < -4 || v > 3) return -1;
        const int c = v + 4, e = (int)(k % 64);
        uint8_t *g = bytes + (k / 64) * 24;
        g[e / 4] |= (uint8_t)((c & 3) << (2 * (e % 4)));
        g[16 + e / 8] |= (uint8_t)(((c >> 2) & 1) << (e % 8));
    }
    return 0;
}

/* y[t][i] = sum_g s[i][g] * sum_{k in g} (code(i,k) - 4) * x[t][k] (form (i),
 * as for int4), and den[t][i] = sum_k |(code - 4) * s * x|. */
void orc_qmv_int3_gs(const uint8_t *wq, const float *s, int N, int K, const float *x, int S,
                     double *y, double *den) {
    const int G = K / 64;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < S; ++t)
        for (int64_t i = 0; i < N; ++i) {
            const uint8_t *row = wq + i * (int64_t)G * 24;
            const float *xt = x + t * (int64_t)K;
            double acc = 0.0, a = 0.0;
            for (int g = 0; g < G; ++g) {
                double part = 0.0;
                const double sc = (double)s[i * G + g];
                for (int64_t k = (int64_t)g * 64; k < (int64_t)(g + 1) * 64; ++k) {
                    const double v = (double)(orc_code3(row, k) - 4);
                    part += v * (double)xt[k];
                    a += fabs(v * sc * (double)xt[k]);
                }
                acc += sc * part;
            }
            y[t * N + i] = acc;
            den[t * N + i] = a;
        }
}

/* ------------------------------------ a3: int8 per-row-scale GEMV [PR418] */

/* y[t][i] = r[i] * sum_k w[i][k] * x[t][k]; den[t][i] = sum_k |r[i] w[i][k] x[t][k]|. */
void orc_qmv_int8_row(const int8_t *w, const float *r, int N, int K, const float *x, int S,
                      double *y, double *den) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < S; ++t)
        for (int64_t i = 0; i < N; ++i) {
            double acc = 0.0, a = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (double)w[i * (int64_t)K + k] * (double)x[t * (int64_t)K + k];
                acc += p;
                a += fabs(p);
            }
            y[t * N + i] = (double)r[i] * acc;
            if (den) den[t * N + i] = fabs((double)r[i]) * a;
        }
}

/* ------------------------------------------------- a4: top-k routing (R4) */

/* The value routing compares: the logit, except that NaN counts as -inf. */
static inline double orc_route_val(float v) { return v != v ? -INFINITY : (double)v; }

/* ids[t][j], j = 0..k-1, in descending logit order; w[t][j] the selected
 * softmax probabilities renormalised over the k selected experts.
 * Returns 0, or -1 on bad sizes. */
int orc_route_topk(const float *logits, int T, int E, int k, int32_t *ids, double *w) {
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    char *taken = (char *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    if (!taken || !p) { free(taken); free(p); return -1; }
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (int64_t)t * E;
        /* softmax over all experts, in double; with every logit at -inf they
         * are all equal, and so are their probabilities */
        double m = orc_route_val(l[0]);
        for (int e = 1; e < E; ++e) if (orc_route_val(l[e]) > m) m = orc_route_val(l[e]);
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = (m == -INFINITY) ? 1.0 : exp(orc_route_val(l[e]) - m);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= z;
        /* selection on the fp32 logits; a strict '>' keeps the lower index on ties */
        memset(taken, 0, (size_t)E);
        double psum = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || orc_route_val(l[e]) > orc_route_val(l[best])) best = e;
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
            psum += p[best];
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = p[ids[(int64_t)t * k + j]] / psum;
    }
    free(taken);
    free(p);
    return 0;
}

/* ---------------------------------------------- a5: token -> expert lists */

/* Inverts ids[T*k] (pair p = t*k + slot) into per-expert lists.
 *   offsets[E+1]: exclusive prefix sum of the per-expert counts;
 *   list[T*k]:    pair ids, grouped by expert, ascending pair id inside a group;
 *   uexp[E]:      the experts with at least one pair, ascending; *n_used of them.
 * Returns 0, or -1 if an id is out of range. */
int orc_group(const int32_t *ids, int T, int k, int E, int32_t *offsets, int32_t *list,
              int32_t *uexp, int32_t *n_used) {
    int64_t P = (int64_t)T * k;
    for (int64_t p = 0; p < P; ++p) if (ids[p] < 0 || ids[p] >= E) return -1;
    int32_t *fill = (int32_t *)calloc((size_t)E + 1, sizeof(int32_t));
    if (!fill) return -1;
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int64_t p = 0; p < P; ++p) offsets[ids[p] + 1] += 1;
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t p = 0; p < P; ++p) list[fill[ids[p]]++] = (int32_t)p;
    int u = 0;
    for (int e = 0; e < E; ++e) if (offsets[e + 1] > offsets[e]) uexp[u++] = e;
    *n_used = u;
    free(fill);
    return 0;
}

/* ------------------------------- a6 + a7: expert FFN [PR418 gate_up, expert group] */

/* One dot product of a packed int4-gs row with a double vector, form (i). */
static double orc_row_dot(const uint8_t *row, const float *srow, int K, int gs,
                          const double *v, double *absden) {
    double acc = 0.0, a = 0.0;
    for (int g = 0; g < K / gs; ++g) {
        double part = 0.0;
        for (int64_t k = (int64_t)g * gs; k < (int64_t)(g + 1) * gs; ++k) {
            double q = (double)(orc_nibble(row, k) - 8);
            part += q * v[k];
            a += fabs(q * (double)srow[g] * v[k]);
        }
        acc += (double)srow[g] * part;
    }
    if (absden) *absden = a;
    return acc;
}

/* For every token t < T and slot j < k, with e = ids[t*k + j] an index into
 * the weight arrays and wt = w[t*k + j]:
 *   g  = gate_e x_t  (rows 0..I-1 of the stacked tensor, reading R3)
 *   u  = up_e   x_t  (rows I..2I-1)
 *   h  = SiLU(g) * u                                   (reading R5)
 *   out[t][i] = sum_j wt * sum_c down_e[i][c] * h[c]    (weighted combine)
 * Weights: gu_q [n][2I][H/2], gu_s [n][2I][H/gs], dn_q [n][H][I/2], dn_s [n][H][I/gs].
 * x is given as double (fp32 and bf16 inputs widen exactly).
 * Optional outputs (NULL to skip):
 *   h[T*k][I]    the hidden activations;
 *   hden[T*k][I] |SiLU'(g) u| * sum|gate x| + |SiLU(g)| * sum|up x|, the
 *                first-order bound on h's error per unit relative error of
 *                the two dot products;
 *   den[T][H]    sum_j |wt| * sum_c |down_e[i][c] * h[c]|.                  */
void orc_moe_ffn(const uint8_t *gu_q, const float *gu_s, const uint8_t *dn_q, const float *dn_s,
                 int H, int I, int gs, const double *x, int T, const int32_t *ids,
                 const float *w, int k, double *h, double *hden, double *out, double *den) {
    int64_t P = (int64_t)T * k;
    double *hh = (double *)malloc(sizeof(double) * (size_t)(P * I));
    if (!hh) return;
    const int64_t gq_e = (int64_t)2 * I * (H / 2), gs_e = (int64_t)2 * I * (H / gs);
    const int64_t dq_e = (int64_t)H * (I / 2), ds_e = (int64_t)H * (I / gs);

#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t p = 0; p < P; ++p)
        for (int64_t c = 0; c < I; ++c) {
            int64_t e = ids[p];
            const double *xt = x + (p / k) * (int64_t)H;
            const uint8_t *grow = gu_q + e * gq_e + c * (H / 2);
            const uint8_t *urow = gu_q + e * gq_e + (I + c) * (H / 2);
            const float *gsr = gu_s + e * gs_e + c * (H / gs);
            const float *usr = gu_s + e * gs_e + (I + c) * (H / gs);
            double dg, du;
            double g = orc_row_dot(grow, gsr, H, gs, xt, &dg);
            double u = orc_row_dot(urow, usr, H, gs, xt, &du);
            double sg = 1.0 / (1.0 + exp(-g));
            double silu = g * sg;
            hh[p * I + c] = silu * u;
            if (hden) {
                double dsilu = sg * (1.0 + g * (1.0 - sg));
                hden[p * I + c] = fabs(dsilu * u) * dg + fabs(silu) * du;
            }
        }
    if (h) memcpy(h, hh, sizeof(double) * (size_t)(P * I));

#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t i = 0; i < H; ++i) {
            double o = 0.0, a = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t p = t * k + j;
                int64_t e = ids[p];
                double ad;
                double y = orc_row_dot(dn_q + e * dq_e + i * (I / 2), dn_s + e * ds_e + i * (I / gs),
                                       I, gs, hh + p * I, &ad);
                o += (double)w[p] * y;
                a += fabs((double)w[p]) * ad;
            }
            out[t * H + i] = o;
            if (den) den[t * H + i] = a;
        }
    free(hh);
}
