/*
 * CPU oracle for the sparse Mixture-of-Experts layer with int4 experts.
 *
 * TEST INFRASTRUCTURE ONLY.  This file defines what the GPU path must
 * compute, in plain loops that a reader can check against the method's
 * description by eye.  It shares no code with the CUDA library; only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark call it.
 *
 * Sources (pages on Lily, Perplexity's engine for Qwen3.6-35B-A3B):
 *   [MoE]    "Lily: Perplexity's Custom Inference Engine for Apple Silicon",
 *            section "The architecture that forces the issue: MoE plus Gated
 *            DeltaNet": a router scores 256 experts and picks 8; a shared
 *            expert runs on every token; expert loads are uneven.
 *   [DEQ]    same page, section "The measured wins": 4-bit checkpoint,
 *            unpacked on chip inside the matmul.
 *   [FUSE]   "Inside Lily: How Perplexity's Rust and Metal Engine ...",
 *            list "Fused Prefill" / "Unified Command Buffers": 4-bit weights
 *            rebuilt tile by tile inside grouped GEMMs; routing histograms and
 *            block maps kept on the GPU.
 *   [GEMV]   first page, section "Why Apple Silicon isn't just a smaller
 *            datacenter GPU": prefill is GEMM work, batch-1 decode is GEMV.
 * The pages give no formulas.  Where they are silent this file takes the
 * plainest reading (each one is listed where it is used):
 *   - int4 asymmetric, groups of G consecutive K elements, bf16 scale and
 *     bias, w = s*q + b with unsigned q in 0..15 (MLX-style affine format);
 *   - router logits l = x . Wr^T (+ per-expert bias), fp32;
 *   - top-k on the logits, ties broken towards the lower expert index, slot j
 *     holds the j-th largest; weights = softmax over all E logits,
 *     renormalised over the k picked ones;
 *   - expert = SwiGLU MLP: h = silu(x Wg^T) * (x Wu^T), o = h Wd^T;
 *   - y = sum_j w_j o_{e_j} + o_shared (shared expert weight 1, no gate);
 *   - the steps either side of the layer (a pre-norm decoder block of the
 *     model family; the pages name the model but not its norm): residual
 *     add h = a + r, x = RMSNorm(h) * w as the layer's input, and the
 *     residual add out = h + y after it (oracle_residual_rmsnorm,
 *     oracle_residual_out).
 *
 * Precision: quantisation and the router run in fp32 (they decide integers
 * that the GPU must reproduce bit for bit: codes and expert indices);
 * dequantisation, the experts, softmax weights and the combine run in fp64.
 * Build without -ffast-math and with -ffp-contract=off so that every fp32
 * operation is one IEEE operation in the written order.
 *
 * Packed layout: the code of element k of a row lives in 32-bit word k/8 of
 * that row, in nibble n = p/2 + 4*(p%2) with p = k%8 (bits 4n .. 4n+3): the
 * word's even elements fill nibbles 0-3, its odd ones nibbles 4-7.  Scale and
 * bias are bf16 bit patterns, one per (row, group), row-major [rows][K/G].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 */

/* Round an fp32 value to bf16, round-to-nearest-even (NaN kept quiet). */
static uint16_t bf16_from_float(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

static float float_from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void oracle_bf16_round(const float *in, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_from_float(in[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops from now on (the CPU-baseline timing runs the
 * oracle on all host cores and on one); returns the previous count.  The
 * per-element arithmetic does not depend on it. */
int oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n > 0)
        omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}

/* ------------------------------------------------------- int4 quantiser */

/* Nibble of element p (0..7) inside its word: even elements in nibbles 0-3,
 * odd ones in nibbles 4-7 (element 2j in nibble j, 2j + 1 in nibble j + 4). */
static int nibble_of(int32_t p)
{
    return p / 2 + 4 * (p % 2);
}

static int get_code(const uint32_t *row_words, int32_t k)
{
    return (int)((row_words[k / 8] >> (4 * nibble_of(k % 8))) & 0xFu);
}

/*
 * Quantise w[rows][K] (fp32) to int4 codes with one bf16 scale and bias per
 * group of G consecutive elements along K.  Per group, in fp32:
 *   mn, mx  = minimum and maximum, found by a left-to-right scan with strict
 *             comparisons (the first of equal values wins);
 *   s       = bf16_rne((mx - mn) / 15),  b = bf16_rne(mn);
 *   q       = clamp(rint_even((w - b) / s), 0, 15) using the bf16-rounded s
 *             and b, and q = 0 for every element when s == 0.
 * [DEQ] fixes only "4-bit"; the asymmetric group format is the reading above.
 */
void oracle_quantize(const float *w, int64_t rows, int32_t K, int32_t G,
                     uint32_t *q, uint16_t *scale, uint16_t *bias)
{
    const int32_t ngroups = K / G;
    const int32_t nwords = K / 8;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint32_t *qrow = q + r * nwords;
        for (int32_t i = 0; i < nwords; ++i)
            qrow[i] = 0u;
        for (int32_t g = 0; g < ngroups; ++g) {
            const float *v = w + r * K + (int64_t)g * G;
            float mn = v[0], mx = v[0];
            for (int32_t i = 1; i < G; ++i) {
                if (v[i] < mn) mn = v[i];
                if (v[i] > mx) mx = v[i];
            }
            float range = mx - mn;
            float s_exact = range / 15.0f;
            uint16_t s_bits = bf16_from_float(s_exact);
            uint16_t b_bits = bf16_from_float(mn);
            scale[r * ngroups + g] = s_bits;
            bias[r * ngroups + g] = b_bits;
            float s = float_from_bf16(s_bits);
            float b = float_from_bf16(b_bits);
            for (int32_t i = 0; i < G; ++i) {
                int code = 0;
                if (s != 0.0f) {
                    float t = (v[i] - b) / s;
                    float rq = nearbyintf(t); /* default mode: nearest, ties to even */
                    if (rq < 0.0f) code = 0;
                    else if (rq > 15.0f) code = 15;
                    else code = (int)rq;
                }
                int32_t k = g * G + i;
                qrow[k / 8] |= (uint32_t)code << (4 * nibble_of(k % 8));
            }
        }
    }
}

/* w = s * q + b, evaluated in fp64 (exact for bf16 s, b and q <= 15). */
static double dequant_one(const uint32_t *q, const uint16_t *scale, const uint16_t *bias,
                          int64_t row, int32_t K, int32_t G, int32_t k)
{
    const uint32_t *qrow = q + row * (K / 8);
    int code = get_code(qrow, k);
    double s = (double)float_from_bf16(scale[row * (K / G) + k / G]);
    double b = (double)float_from_bf16(bias[row * (K / G) + k / G]);
    return s * (double)code + b;
}

void oracle_dequant(const uint32_t *q, const uint16_t *scale, const uint16_t *bias,
                    int64_t rows, int32_t K, int32_t G, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int32_t k = 0; k < K; ++k)
            out[r * K + k] = dequant_one(q, scale, bias, r, K, G, k);
}

/* ---------------------------------------------------------------- router */

/*
 * l[t][e] = sum_h x[t][h] * Wr[e][h] (+ bias[e]), accumulated in fp32 in
 * increasing h ([MoE]: the router gives every expert a score).  x is bf16
 * (widened exactly), Wr and bias are fp32.
 */
void oracle_router_logits(const uint16_t *x, int32_t T, int32_t H, const float *Wr,
                          const float *router_bias, int32_t E, float *logits)
{
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            float acc = 0.0f;
            for (int32_t h = 0; h < H; ++h) {
                float prod = float_from_bf16(x[(int64_t)t * H + h]) * Wr[(int64_t)e * H + h];
                acc = acc + prod;
            }
            if (router_bias)
                acc = acc + router_bias[e];
            logits[(int64_t)t * E + e] = acc;
        }
    }
}

/* ----------------------------------------------------------- top-k, weights */

typedef struct {
    float logit;
    int32_t expert;
} scored;

/* larger logit first; equal logits: lower expert index first */
static int by_logit_then_index(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->logit > b->logit) return -1;
    if (a->logit < b->logit) return 1;
    return (a->expert > b->expert) - (a->expert < b->expert);
}

/*
 * Full sort of one token's E logits, keep the first k ([MoE]: "picks 8").
 * Weights: p = softmax over all E (fp64, max subtracted), then
 * w_j = p_{e_j} / sum over the picked p (renorm), or w_j = p_{e_j} (no
 * renormalisation: the routing variant whose picked weights sum below 1).
 */
static void topk_one(const float *l, int32_t E, int32_t k, int32_t renorm, int32_t *idx, double *w)
{
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)E);
    for (int32_t e = 0; e < E; ++e) {
        s[e].logit = l[e];
        s[e].expert = e;
    }
    qsort(s, (size_t)E, sizeof(scored), by_logit_then_index);
    double mx = (double)s[0].logit;
    double total = 0.0;
    for (int32_t e = 0; e < E; ++e)
        total += exp((double)l[e] - mx);
    double picked = 0.0;
    for (int32_t j = 0; j < k; ++j) {
        idx[j] = s[j].expert;
        picked += exp((double)s[j].logit - mx) / total;
    }
    for (int32_t j = 0; j < k; ++j)
        w[j] = renorm ? (exp((double)s[j].logit - mx) / total) / picked : exp((double)s[j].logit - mx) / total;
    free(s);
}

void oracle_topk_opt(const float *logits, int32_t T, int32_t E, int32_t k, int32_t renorm, int32_t *idx,
                     double *w)
{
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; ++t)
        topk_one(logits + (int64_t)t * E, E, k, renorm, idx + (int64_t)t * k, w + (int64_t)t * k);
}

void oracle_topk(const float *logits, int32_t T, int32_t E, int32_t k, int32_t *idx, double *w)
{
    oracle_topk_opt(logits, T, E, k, 1, idx, w);
}

/*
 * Shared-expert gate of the routing variant with a gated shared expert: one
 * more router-like score per token, l = sum_h x[t][h] * g[h] (fp32, in
 * increasing h, as the router logits), weight = 1 / (1 + exp(-l)) in fp64.
 */
void oracle_shared_gate(const uint16_t *x, int32_t T, int32_t H, const float *gate, double *w)
{
    float *l = (float *)malloc(sizeof(float) * (size_t)T);
    oracle_router_logits(x, T, H, gate, NULL, 1, l);
    for (int32_t t = 0; t < T; ++t)
        w[t] = 1.0 / (1.0 + exp(-(double)l[t]));
    free(l);
}

/* ------------------------------------------- histogram, scan, permutation */

/*
 * Group g < E holds the (token, slot) pairs routed to expert g; when
 * has_shared, group E holds every token once (the shared expert).
 *   counts[g]   rows of group g (histogram; [FUSE] "routing histograms")
 *   offsets[g]  exclusive prefix sum of counts, offsets[G] = total rows
 *   perm[r]     for routed row r < T*k: t*k + j, rows ordered by (expert asc,
 *               token asc) (a counting sort that is stable in the token)
 *   inv_perm    inverse of perm
 *   tiles       each group cut into blocks of at most BN consecutive rows,
 *               groups in order ([FUSE] "block maps"): (group, first row, rows)
 * Returns the number of tiles, or -1 if max_tiles is too small.
 */
int32_t oracle_route(const int32_t *idx, int32_t T, int32_t k, int32_t E, int32_t has_shared,
                     int32_t BN, int32_t *counts, int32_t *offsets, int32_t *perm,
                     int32_t *inv_perm, int32_t *tile_group, int32_t *tile_row,
                     int32_t *tile_rows, int32_t max_tiles)
{
    const int32_t ngroups = E + (has_shared ? 1 : 0);
    if (E < 1 || k < 1 || T < 0 || BN < 1)
        return -1;
    for (int32_t g = 0; g < ngroups; ++g)
        counts[g] = 0;
    for (int64_t i = 0; i < (int64_t)T * k; ++i)
        counts[idx[i]] += 1;
    if (has_shared)
        counts[E] = T;
    offsets[0] = 0;
    for (int32_t g = 0; g < ngroups; ++g)
        offsets[g + 1] = offsets[g] + counts[g];

    int32_t *fill = (int32_t *)calloc((size_t)ngroups, sizeof(int32_t));
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = idx[(int64_t)t * k + j];
            int32_t r = offsets[e] + fill[e];
            fill[e] += 1;
            perm[r] = t * k + j;
            inv_perm[t * k + j] = r;
        }
    }
    free(fill);

    int32_t n = 0;
    for (int32_t g = 0; g < ngroups; ++g) {
        for (int32_t r0 = 0; r0 < counts[g]; r0 += BN) {
            if (n >= max_tiles)
                return -1;
            tile_group[n] = g;
            tile_row[n] = offsets[g] + r0;
            tile_rows[n] = counts[g] - r0 < BN ? counts[g] - r0 : BN;
            n += 1;
        }
    }
    return n;
}

/* ---------------------------------------------------------------- experts */

typedef struct {
    int32_t H, I, G;
    const uint32_t *qg, *qu, *qd;
    const uint16_t *sg, *bg, *su, *bu, *sd, *bd;
} expert_weights;

typedef void (*expert_fn)(const void *ctx, int32_t e, const double *xv, double *out);

/*
 * One SwiGLU expert on one token vector ([MoE], [FUSE]): gate and up
 * matrices [I][H], down matrix [H][I], all int4 with groups along their K.
 *   g_i = sum_h x_h Wg[i][h],  u_i = sum_h x_h Wu[i][h]
 *   h_i = g_i / (1 + exp(-g_i)) * u_i
 *   o_f = sum_i h_i Wd[f][i]
 */
static void swiglu_expert(const void *ctx, int32_t e, const double *xv, double *out)
{
    const expert_weights *W = (const expert_weights *)ctx;
    const int32_t H = W->H, I = W->I, G = W->G;
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)I);
    for (int32_t i = 0; i < I; ++i) {
        int64_t row = (int64_t)e * I + i;
        double gsum = 0.0, usum = 0.0;
        for (int32_t h = 0; h < H; ++h) {
            gsum += xv[h] * dequant_one(W->qg, W->sg, W->bg, row, H, G, h);
            usum += xv[h] * dequant_one(W->qu, W->su, W->bu, row, H, G, h);
        }
        hbuf[i] = gsum / (1.0 + exp(-gsum)) * usum;
    }
    for (int32_t f = 0; f < H; ++f) {
        int64_t row = (int64_t)e * H + f;
        double osum = 0.0;
        for (int32_t i = 0; i < I; ++i)
            osum += hbuf[i] * dequant_one(W->qd, W->sd, W->bd, row, I, G, i);
        out[f] = osum;
    }
    free(hbuf);
}

/*
 * Dispatch and combine for the listed tokens:
 *   y_t = sum_j w_{t,j} * expert(e_{t,j}, x_t) + c_t * shared(x_t)   (fp64)
 * with c_t = 1, or the shared gate's weight of token n when shared_w is
 * given.  The expert is a callable so that the tests can plug in an identity
 * expert.
 */
static void dispatch_combine(const uint16_t *x, int32_t H, int32_t k, int32_t E,
                             int32_t has_shared, const int32_t *idx, const double *w,
                             const int32_t *tokens, int32_t n_tokens, const double *shared_w,
                             expert_fn fn, const void *ctx, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t n = 0; n < n_tokens; ++n) {
        int32_t t = tokens[n];
        double *xv = (double *)malloc(sizeof(double) * (size_t)H);
        double *o = (double *)malloc(sizeof(double) * (size_t)H);
        double *yt = y + (int64_t)n * H;
        for (int32_t h = 0; h < H; ++h) {
            xv[h] = (double)float_from_bf16(x[(int64_t)t * H + h]);
            yt[h] = 0.0;
        }
        for (int32_t j = 0; j < k; ++j) {
            fn(ctx, idx[(int64_t)n * k + j], xv, o);
            for (int32_t h = 0; h < H; ++h)
                yt[h] += w[(int64_t)n * k + j] * o[h];
        }
        if (has_shared) {
            const double c = shared_w ? shared_w[n] : 1.0;
            fn(ctx, E, xv, o);
            for (int32_t h = 0; h < H; ++h)
                yt[h] += c * o[h];
        }
        free(xv);
        free(o);
    }
}

/*
 * Whole layer for the listed tokens (tokens == NULL: all T tokens, in order):
 * router logits, top-k and weights, experts, combine.  Outputs are per listed
 * token: logits [n][E] fp32, idx [n][k], w [n][k] fp64, y [n][H] fp64, and,
 * when shared_w is not NULL, the shared expert's weight [n] (1, or the gate's).
 * Routing variants: renorm = 0 keeps the picked softmax probabilities as they
 * are; shared_gate ([H] fp32, or NULL) gates the shared expert per token.
 */
void oracle_moe_layer_opt(const uint16_t *x, int32_t T, int32_t H, int32_t I, int32_t E,
                          int32_t k, int32_t G, int32_t has_shared, int32_t renorm,
                          const float *Wr, const float *router_bias, const float *shared_gate,
                          const uint32_t *qg, const uint16_t *sg, const uint16_t *bg,
                          const uint32_t *qu, const uint16_t *su, const uint16_t *bu,
                          const uint32_t *qd, const uint16_t *sd, const uint16_t *bd,
                          const int32_t *tokens, int32_t n_tokens,
                          float *logits, int32_t *idx, double *w, double *y, double *shared_w)
{
    int32_t *all = NULL;
    if (!tokens) {
        all = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
        for (int32_t t = 0; t < T; ++t)
            all[t] = t;
        tokens = all;
        n_tokens = T;
    }
    /* gather the listed tokens so that the router sees only those rows */
    uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_tokens * H);
    for (int32_t n = 0; n < n_tokens; ++n)
        memcpy(xs + (int64_t)n * H, x + (int64_t)tokens[n] * H, sizeof(uint16_t) * (size_t)H);
    oracle_router_logits(xs, n_tokens, H, Wr, router_bias, E, logits);
    oracle_topk_opt(logits, n_tokens, E, k, renorm, idx, w);
    double *cw = NULL;
    if (shared_gate) {
        cw = (double *)malloc(sizeof(double) * (size_t)n_tokens);
        oracle_shared_gate(xs, n_tokens, H, shared_gate, cw);
    }
    if (shared_w)
        for (int32_t n = 0; n < n_tokens; ++n)
            shared_w[n] = cw ? cw[n] : 1.0;

    int32_t *seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_tokens);
    for (int32_t n = 0; n < n_tokens; ++n)
        seq[n] = n;
    expert_weights W = {H, I, G, qg, qu, qd, sg, bg, su, bu, sd, bd};
    dispatch_combine(xs, H, k, E, has_shared, idx, w, seq, n_tokens, cw, swiglu_expert, &W, y);
    free(cw);
    free(seq);
    free(xs);
    free(all);
}

void oracle_moe_layer(const uint16_t *x, int32_t T, int32_t H, int32_t I, int32_t E,
                      int32_t k, int32_t G, int32_t has_shared,
                      const float *Wr, const float *router_bias,
                      const uint32_t *qg, const uint16_t *sg, const uint16_t *bg,
                      const uint32_t *qu, const uint16_t *su, const uint16_t *bu,
                      const uint32_t *qd, const uint16_t *sd, const uint16_t *bd,
                      const int32_t *tokens, int32_t n_tokens,
                      float *logits, int32_t *idx, double *w, double *y)
{
    oracle_moe_layer_opt(x, T, H, I, E, k, G, has_shared, 1, Wr, router_bias, NULL, qg, sg, bg, qu, su, bu,
                         qd, sd, bd, tokens, n_tokens, logits, idx, w, y, NULL);
}

/* Experts only, with routing given (the single-expert dense pin, and the
 * rows that the tests evaluate under the routing the GPU chose): shared_w
 * [T] is the shared expert's weight per token, or NULL for 1. */
void oracle_experts_given_routing(const uint16_t *x, int32_t T, int32_t H, int32_t I,
                                  int32_t E, int32_t k, int32_t G, int32_t has_shared,
                                  const uint32_t *qg, const uint16_t *sg, const uint16_t *bg,
                                  const uint32_t *qu, const uint16_t *su, const uint16_t *bu,
                                  const uint32_t *qd, const uint16_t *sd, const uint16_t *bd,
                                  const int32_t *idx, const double *w, const double *shared_w, double *y)
{
    int32_t *seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    for (int32_t t = 0; t < T; ++t)
        seq[t] = t;
    expert_weights W = {H, I, G, qg, qu, qd, sg, bg, su, bu, sd, bd};
    dispatch_combine(x, H, k, E, has_shared, idx, w, seq, T, shared_w, swiglu_expert, &W, y);
    free(seq);
}

static void identity_expert(const void *ctx, int32_t e, const double *xv, double *out)
{
    const int32_t *dims = (const int32_t *)ctx; /* dims[0] = H, dims[1] = E */
    for (int32_t h = 0; h < dims[0]; ++h)
        out[h] = (e == dims[1]) ? 0.0 : xv[h];
}

/* Dispatch/combine with every routed expert the identity and the shared one zero. */
void oracle_dispatch_combine_identity(const uint16_t *x, int32_t T, int32_t H, int32_t E,
                                      int32_t k, int32_t has_shared, const int32_t *idx,
                                      const double *w, double *y)
{
    int32_t *seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)T);
    for (int32_t t = 0; t < T; ++t)
        seq[t] = t;
    int32_t dims[2] = {H, E};
    dispatch_combine(x, H, k, E, has_shared, idx, w, seq, T, NULL, identity_expert, dims, y);
    free(seq);
}

/* ------------------------------------------- steps either side of the layer */

/* Round a double to bf16 in one step (round to nearest, ties to even): the
 * significand is brought to 8 bits with nearbyint (default rounding mode),
 * which a float then holds exactly.  Normal range only (no subnormals here). */
static uint16_t bf16_from_double(double v)
{
    if (v == 0.0 || !isfinite(v))
        return bf16_from_float((float)v);
    int e;
    const double m = frexp(v, &e);                 /* |m| in [0.5, 1) */
    const double r = nearbyint(ldexp(m, 8));       /* 8 significant bits */
    return bf16_from_float((float)ldexp(r, e - 8)); /* exact in float and bf16 */
}

/* Residual add and RMS norm before the layer, per token t (reading: the MoE
 * sub-layer of a pre-norm decoder block; the pages name the model, not its
 * norm):
 *   h[t]   = bf16(fp32(a[t] + r[t]))                      (the residual stream)
 *   x[t]   = bf16(h[t] / sqrt(mean_k h[t][k]^2 + eps) * w) (fp64 statistics)
 * a, r, h, x: bf16 bit patterns [T][H]; w: [H] fp32. */
void oracle_residual_rmsnorm(const uint16_t *a, const uint16_t *r, int32_t T, int32_t H, const float *w,
                             double eps, uint16_t *h, uint16_t *x)
{
    for (int32_t t = 0; t < T; ++t) {
        const int64_t o = (int64_t)t * H;
        double ss = 0.0;
        for (int32_t k = 0; k < H; ++k) {
            const float s = float_from_bf16(a[o + k]) + float_from_bf16(r[o + k]);
            h[o + k] = bf16_from_float(s);
            const double hv = (double)float_from_bf16(h[o + k]);
            ss += hv * hv;
        }
        const double inv = 1.0 / sqrt(ss / (double)H + eps);
        for (int32_t k = 0; k < H; ++k)
            x[o + k] = bf16_from_double((double)float_from_bf16(h[o + k]) * inv * (double)w[k]);
    }
}

/* The residual add after the layer: out[t] = bf16(h[t] + y[t]), y the
 * layer's output in fp64 (rounded once). */
void oracle_residual_out(const uint16_t *h, const double *y, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bf16_from_double((double)float_from_bf16(h[i]) + y[i]);
}

/* ------------------------------------- GQA decode attention (second workload) */

/*
 * One new token's attention over a cache of L positions, with query heads
 * sharing key-value heads ([MoE] page, section "The architecture that forces
 * the issue": full-attention layers use grouped-query attention, 16 query
 * heads sharing 2 key-value heads; same page, section "How this compares to
 * what else is happening on Apple Silicon": GQA packing loads each shared KV
 * row once instead of once per query head).  Readings where the pages are
 * silent: query head h uses key-value head h / (Hq / Hkv) (consecutive query
 * heads share one), scores are scaled by `scale` (1 / sqrt(D) in the tests
 * and benchmark), the softmax runs over all L cached positions (the new
 * token's own key and value are already in the cache).  For each head h:
 *   s_t    = scale * sum_d q[h][d] k[g][t][d]          (fp64)
 *   p_t    = exp(s_t - max_t s_t) / sum_t exp(s_t - max_t s_t)
 *   o[h][d] = sum_t p_t v[g][t][d]
 * q: bf16 bits [Hq][D]; k, v: bf16 bits [Hkv][L_cap][D], positions 0..L-1
 * used; o: fp64 [Hq][D].
 */
void oracle_gqa_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int32_t Hq, int32_t Hkv,
                          int32_t D, int32_t L, int32_t L_cap, double scale, double *o)
{
    const int32_t group = Hq / Hkv;
#pragma omp parallel for schedule(static)
    for (int32_t h = 0; h < Hq; ++h) {
        const int32_t g = h / group;
        const uint16_t *kh = k + (int64_t)g * L_cap * D;
        const uint16_t *vh = v + (int64_t)g * L_cap * D;
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        double mx = -INFINITY;
        for (int32_t t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d)
                acc += (double)float_from_bf16(q[(int64_t)h * D + d]) *
                       (double)float_from_bf16(kh[(int64_t)t * D + d]);
            s[t] = scale * acc;
            if (s[t] > mx)
                mx = s[t];
        }
        double sum = 0.0;
        for (int32_t t = 0; t < L; ++t) {
            s[t] = exp(s[t] - mx);
            sum += s[t];
        }
        for (int32_t d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int32_t t = 0; t < L; ++t)
                acc += s[t] * (double)float_from_bf16(vh[(int64_t)t * D + d]);
            o[(int64_t)h * D + d] = acc / sum;
        }
        free(s);
    }
}
