/*
 * Plain CPU oracle for one Beam-style sparse MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition the GPU library is checked against.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Sources (web pages describing Reflection's Beam-1.0-501B-A23B model):
 *  [P1-MoE]  "Reflection Beam 1.0: 501B open MoE model, 1M context, Apache 2.0"
 *            (agentlenshq.com), section "Mixture of Experts: 256 experts,
 *            8 routed per token": sigmoid scores over all experts, 8 groups of
 *            32, groups ranked by the sum of their top-2 scores, the best 4
 *            groups kept, top-8 experts chosen inside them, no shared expert,
 *            expert outputs combined with the normalised router weights and
 *            scaled by 2.5; each expert is a SwiGLU MLP of intermediate 2560.
 *  [P1-FP32] same page, section "Residual stream", last paragraph: the router
 *            and the SwiGLU product are computed in FP32.
 *  [P1-ARCH] same page, section "Architecture: hybrid attention, grouped
 *            experts, constant-scale residual stream", first paragraph: 52
 *            decoder layers of hidden size 5120, the first 3 with a dense
 *            SwiGLU MLP, the other 49 with the MoE block.
 *  [P1-RES]  same page, section "Residual stream: a constant scale with
 *            depth-dependent weights": the input embedding is step 1; at step
 *            k the sublayer output is added with weight 1/sqrt(k) and the
 *            stream kept with weight sqrt((k-1)/k); every sublayer is also
 *            normalised before and after, and normalisations run in FP32.
 *  [P4-MoE]  "Beam 501B open model" (aixai.ru), section "256 experts per
 *            layer": the same routing restated.
 *  [P5-MoE]  "Reflection 501B-parameter Beam model" (dothoosh.com), section
 *            "Architecture and memory efficiency": the same routing restated;
 *            FP32 pins restated in the section on residual-stream design.
 *
 * Readings taken where the pages are silent:
 *  - router logits: l[t,e] = sum_h x[t,h]*Wr[h,e], FP32 fused multiply-add in
 *    ascending h, starting from +0.0f.
 *  - sigmoid: s = 1/(1+E) in FP32 where E is exp(-l) rounded to FP32 (computed
 *    through the double-precision exp and one rounding).
 *  - group score: sum of the top min(2, group size) scores of the group (FP32).
 *  - ties: lower group index / lower expert index wins.
 *  - selected-slot order: score descending, expert index ascending.
 *  - weights: S = FP32 sum of the selected scores in slot order,
 *    w_k = (s_k / S) * scale, FP32 divide then FP32 multiply.
 *  - expert: g = x.Wg[e]^T, u = x.Wu[e]^T accumulated in FP64 and rounded to
 *    FP32; h = silu(g)*u in FP32 (the pinned product); y = h.Wd[e]^T in FP64.
 *  - combine: out = bf16_rne(float(sum_k w_k*y_k)), FP64 sum in ascending k.
 *  - permuted order: rows grouped by expert (ascending), tokens ascending
 *    inside an expert.
 *
 * NVFP4 variant (the pages: "most parameters in 4 bits, some kept in BF16",
 * [P1-HW] = "Reflection Beam 1.0", section "Hardware requirements: NVFP4 is
 * the most practical serving path", and [P5-MoE]; they give no recipe, so the
 * whole recipe is a reading): E2M1 values with one E4M3 scale per 16
 * consecutive elements of a row and one FP32 scale per matrix,
 *   gs = amax|W| / (6*448)                     (1 if the matrix is all zero)
 *   sf = e4m3( (amax16 / 6) / gs )             round to nearest even, saturate
 *   q  = e2m1( v / (sf*gs) )                   0 when sf == 0
 *   dequantised value = q * sf * gs.
 * Activations (x before the gate/up GEMM, h before the down GEMM) use the
 * same block recipe with gs = 1.  The router stays FP32 on the bf16 x.
 *
 * Everything here is written for clarity, not speed: no blocking, no fusion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- helpers */

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE round-to-nearest-even from FP32 to bfloat16 (NaN kept quiet). */
static uint16_t float_to_bf16_bits_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* FP32 sigmoid as read from [P1-MoE]/[P1-FP32]: 1/(1+E), E = fp32(exp(-l)). */
static float sigmoid_f32(float l)
{
    float e = (float)exp(-(double)l);
    float den = 1.0f + e;
    return 1.0f / den;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------ router step */

/*
 * Router logits and sigmoid scores, [P1-MoE] + [P1-FP32].
 *   x      [T,H] bf16 bits      wr [H,E] fp32 (row-major, hidden-major)
 *   logits [T,E] fp32 or NULL   scores [T,E] fp32
 */
void oracle_router_scores(const uint16_t *x, const float *wr, int64_t T, int H,
                          int E, float *logits, float *scores)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        float *acc = (float *)malloc(sizeof(float) * (size_t)E);
        for (int e = 0; e < E; ++e)
            acc[e] = 0.0f;
        /* every acc[e] sees the terms h = 0, 1, ..., H-1 in that order */
        for (int h = 0; h < H; ++h) {
            float xv = bf16_bits_to_float(x[t * H + h]);
            const float *wrow = wr + (int64_t)h * E;
            for (int e = 0; e < E; ++e)
                acc[e] = fmaf(xv, wrow[e], acc[e]);
        }
        for (int e = 0; e < E; ++e) {
            if (logits)
                logits[t * E + e] = acc[e];
            scores[t * E + e] = sigmoid_f32(acc[e]);
        }
        free(acc);
    }
}

/* --------------------------------------------------------- selection step */

/* "a ranks before b" for (value descending, index ascending). */
static int ranks_before(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

/*
 * Group-limited top-k on given FP32 scores, [P1-MoE], [P4-MoE], [P5-MoE].
 *   scores [T,E]; ids [T,top_k] int32; w [T,top_k] fp32.
 * Returns 0, or -1 on an invalid configuration or a non-finite score.
 */
int oracle_select(const float *scores, int64_t T, int E, int G, int topk_groups,
                  int top_k, float scale, int32_t *ids, float *w)
{
    if (E <= 0 || G <= 0 || E % G != 0 || topk_groups <= 0 || topk_groups > G ||
        top_k <= 0 || top_k > topk_groups * (E / G))
        return -1;
    const int gsize = E / G;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < T; ++t) {
        const float *s = scores + t * E;
        float *gscore = (float *)malloc(sizeof(float) * (size_t)G);
        char *gkept = (char *)calloc((size_t)G, 1);
        char *taken = (char *)calloc((size_t)E, 1);
        for (int e = 0; e < E; ++e)
            if (!isfinite(s[e]))
                bad = 1;

        /* 1. group score = sum of the group's two largest scores */
        for (int g = 0; g < G; ++g) {
            const float *sg = s + g * gsize;
            int i1 = 0;
            for (int j = 1; j < gsize; ++j)
                if (ranks_before(sg[j], j, sg[i1], i1))
                    i1 = j;
            if (gsize == 1) {
                gscore[g] = sg[i1];
                continue;
            }
            int i2 = -1;
            for (int j = 0; j < gsize; ++j) {
                if (j == i1)
                    continue;
                if (i2 < 0 || ranks_before(sg[j], j, sg[i2], i2))
                    i2 = j;
            }
            gscore[g] = sg[i1] + sg[i2];
        }

        /* 2. keep the topk_groups best groups */
        for (int r = 0; r < topk_groups; ++r) {
            int best = -1;
            for (int g = 0; g < G; ++g) {
                if (gkept[g])
                    continue;
                if (best < 0 || ranks_before(gscore[g], g, gscore[best], best))
                    best = g;
            }
            gkept[best] = 1;
        }

        /* 3. top_k experts among the kept groups, slot order = rank order */
        for (int k = 0; k < top_k; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (!gkept[e / gsize] || taken[e])
                    continue;
                if (best < 0 || ranks_before(s[e], e, s[best], best))
                    best = e;
            }
            taken[best] = 1;
            ids[t * top_k + k] = best;
        }

        /* 4. normalise the selected scores to sum 1, then scale */
        float S = 0.0f;
        for (int k = 0; k < top_k; ++k)
            S = S + s[ids[t * top_k + k]];
        for (int k = 0; k < top_k; ++k) {
            float q = s[ids[t * top_k + k]] / S;
            w[t * top_k + k] = q * scale;
        }
        free(gscore);
        free(gkept);
        free(taken);
    }
    return bad ? -1 : 0;
}

/* ---------------------------------------------------------- dispatch step */

/*
 * Expert histogram, exclusive offsets and the permutation that groups the
 * (token, slot) pairs by expert, tokens ascending inside an expert.
 *   ids [T,K] -> counts [E], offsets [E+1], row_of [T,K], row_src [T*K]
 */
int oracle_dispatch(const int32_t *ids, int64_t T, int K, int E, int32_t *counts,
                    int32_t *offsets, int32_t *row_of, int32_t *row_src)
{
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < T * K; ++i) {
        if (ids[i] < 0 || ids[i] >= E)
            return -1;
        counts[ids[i]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int e = ids[t * K + k];
            int32_t row = offsets[e] + cursor[e];
            cursor[e] += 1;
            row_of[t * K + k] = row;
            row_src[row] = (int32_t)t;
        }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------ expert step */

/*
 * One SwiGLU expert on one token, [P1-MoE] (SwiGLU MLP, intermediate I) and
 * [P1-FP32] (the SwiGLU product in FP32).
 *   xrow [H] bf16 bits; wg, wu [I,H] bf16 bits; wd [H,I] bf16 bits
 *   hbuf [I] fp32 scratch; y [H] fp64 out
 */
static void expert_swiglu(const uint16_t *xrow, const uint16_t *wg,
                          const uint16_t *wu, const uint16_t *wd, int H, int I,
                          float *hbuf, double *y)
{
    for (int i = 0; i < I; ++i) {
        double gd = 0.0, ud = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = (double)bf16_bits_to_float(xrow[h]);
            gd += xv * (double)bf16_bits_to_float(wg[(int64_t)i * H + h]);
            ud += xv * (double)bf16_bits_to_float(wu[(int64_t)i * H + h]);
        }
        float g = (float)gd, u = (float)ud;
        float silu = g * sigmoid_f32(g);
        hbuf[i] = silu * u;
    }
    for (int j = 0; j < H; ++j) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += (double)hbuf[i] * (double)bf16_bits_to_float(wd[(int64_t)j * I + i]);
        y[j] = acc;
    }
}

/* exported for the single-expert pin: y = SwiGLU expert applied to one row */
void oracle_expert_row(const uint16_t *xrow, const uint16_t *wg,
                       const uint16_t *wu, const uint16_t *wd, int H, int I,
                       double *y)
{
    float *hbuf = (float *)malloc(sizeof(float) * (size_t)I);
    expert_swiglu(xrow, wg, wu, wd, H, I, hbuf, y);
    free(hbuf);
}

/* ----------------------------------------------------------- whole layer */

/*
 * The router's scores for one token: computed from x and wr (the router
 * step), or, when the caller gives scores_in [T,E], that token's given row.
 * The given-scores form is the layer from the selection step on, applied to
 * FP32 scores produced elsewhere (the pages fix the selection, weights,
 * experts and combine as functions of the FP32 scores).
 */
static void token_scores(const uint16_t *xrow, const float *wr, const float *scores_in,
                         int64_t t, int H, int E, float *scores)
{
    if (scores_in)
        memcpy(scores, scores_in + t * E, sizeof(float) * (size_t)E);
    else
        oracle_router_scores(xrow, wr, 1, H, E, NULL, scores);
}

/*
 * The layer forward for a list of tokens (all tokens when tokens == NULL):
 * router -> group-limited top-k -> experts -> weighted combine.
 *   x [T,H] bf16; wr [H,E] fp32; wg, wu [E,I,H] bf16; wd [E,H,I] bf16
 *   out [n,H] bf16 bits (row r is token tokens[r]);
 *   ids_out [n,top_k], w_out [n,top_k] may be NULL;
 *   scores_in [T,E] fp32 or NULL: the router's scores, used instead of the
 *   router step when given (wr is then not read);
 *   o_out [n,H] fp32 or NULL: the FP32 combine before the bf16 rounding of
 *   out (the input of the fused block's post-norm).
 */
int oracle_forward(const uint16_t *x, const float *wr, const uint16_t *wg,
                   const uint16_t *wu, const uint16_t *wd, int64_t T, int H,
                   int I, int E, int G, int topk_groups, int top_k, float scale,
                   const int64_t *tokens, int64_t n_tokens, uint16_t *out,
                   int32_t *ids_out, float *w_out, const float *scores_in, float *o_out)
{
    if (E % G != 0 || top_k > topk_groups * (E / G))
        return -1;
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        const uint16_t *xrow = x + t * H;
        float *scores = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
        float *w = (float *)malloc(sizeof(float) * (size_t)top_k);
        float *hbuf = (float *)malloc(sizeof(float) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *acc = (double *)calloc((size_t)H, sizeof(double));

        token_scores(xrow, wr, scores_in, t, H, E, scores);
        if (oracle_select(scores, 1, E, G, topk_groups, top_k, scale, ids, w) != 0)
            bad = 1;
        for (int k = 0; k < top_k && !bad; ++k) {
            const int64_t e = ids[k];
            expert_swiglu(xrow, wg + e * I * H, wu + e * I * H, wd + e * H * I, H,
                          I, hbuf, y);
            for (int j = 0; j < H; ++j)
                acc[j] += (double)w[k] * y[j];
        }
        {
            for (int j = 0; j < H; ++j) {
                if (o_out)
                    o_out[r * H + j] = (float)acc[j];
                out[r * H + j] = float_to_bf16_bits_rne((float)acc[j]);
            }
        }
        if (ids_out)
            memcpy(ids_out + r * top_k, ids, sizeof(int32_t) * (size_t)top_k);
        if (w_out)
            memcpy(w_out + r * top_k, w, sizeof(float) * (size_t)top_k);
        free(scores);
        free(ids);
        free(w);
        free(hbuf);
        free(y);
        free(acc);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------ dense layer */

/*
 * The dense SwiGLU MLP of Beam's first three decoder layers ([P1-ARCH]: the
 * first 3 of the 52 layers use a dense SwiGLU MLP, the other 49 the MoE
 * block), with the SwiGLU product in FP32 ([P1-FP32]).  The pages give no
 * intermediate size for it; I is the caller's.
 *   x [T,H] bf16; wg, wu [I,H] bf16; wd [H,I] bf16; out [n,H] bf16 bits
 *   (row r is token tokens[r], all tokens when tokens == NULL)
 */
int oracle_dense_forward(const uint16_t *x, const uint16_t *wg, const uint16_t *wu,
                         const uint16_t *wd, int64_t T, int H, int I,
                         const int64_t *tokens, int64_t n_tokens, uint16_t *out)
{
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        float *hbuf = (float *)malloc(sizeof(float) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        expert_swiglu(x + t * H, wg, wu, wd, H, I, hbuf, y);
        for (int j = 0; j < H; ++j)
            out[r * H + j] = float_to_bf16_bits_rne((float)y[j]);
        free(hbuf);
        free(y);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------ fused MoE block */

/*
 * RMS normalisation of one row ([P1-RES]: sublayers are normalised before
 * and after, in FP32; the pages name RMSNorm for queries and keys and no
 * other norm, so the reading is RMSNorm with a learned per-channel gain).
 * The sum of squares is accumulated in FP64 and rounded to FP32 once as a
 * mean; r = 1 / sqrt(mean + eps) in FP32; v[h] * r * gamma[h] in FP32.
 */
static float rms_inv(const float *v, int n, float eps)
{
    double ss = 0.0;
    for (int h = 0; h < n; ++h)
        ss += (double)v[h] * (double)v[h];
    const float mean = (float)(ss / (double)n);
    return 1.0f / sqrtf(mean + eps);
}

/*
 * One MoE sublayer of the decoder with its norms and residual ([P1-RES]):
 *   x  = bf16( rmsnorm(s) * gamma_pre )        the layer's bf16 input
 *   o  = MoE(x) in FP32 (combine before the output rounding)
 *   z  = rmsnorm(o) * gamma_post               FP32
 *   s' = bf16( a*s + b*z ),  a = sqrt((k-1)/k), b = 1/sqrt(k) (FP32)
 *   s  [T,H] bf16 bits (the residual stream at step k-1); out [n,H] bf16
 *   bits (row r is token tokens[r], all tokens when tokens == NULL);
 *   scores_in [T,E] fp32 or NULL: the router's scores of the pre-normed x,
 *   used instead of the router step when given.
 */
int oracle_block_forward(const uint16_t *s, int step, const float *gamma_pre,
                         const float *gamma_post, float eps, const float *wr,
                         const uint16_t *wg, const uint16_t *wu, const uint16_t *wd,
                         int64_t T, int H, int I, int E, int G, int topk_groups,
                         int top_k, float scale, const int64_t *tokens, int64_t n_tokens,
                         uint16_t *out, const float *scores_in)
{
    if (step < 1 || E % G != 0 || top_k > topk_groups * (E / G))
        return -1;
    const float a = (float)sqrt((double)(step - 1) / (double)step);
    const float b = (float)(1.0 / sqrt((double)step));
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        float *sv = (float *)malloc(sizeof(float) * (size_t)H);
        uint16_t *xb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)H);
        float *o = (float *)malloc(sizeof(float) * (size_t)H);
        float *scores = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
        float *w = (float *)malloc(sizeof(float) * (size_t)top_k);
        float *hbuf = (float *)malloc(sizeof(float) * (size_t)I);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *acc = (double *)calloc((size_t)H, sizeof(double));

        for (int h = 0; h < H; ++h)
            sv[h] = bf16_bits_to_float(s[t * H + h]);
        const float rp = rms_inv(sv, H, eps);
        for (int h = 0; h < H; ++h) {
            const float v = sv[h] * rp;
            xb[h] = float_to_bf16_bits_rne(v * gamma_pre[h]);
        }
        token_scores(xb, wr, scores_in, t, H, E, scores);
        if (oracle_select(scores, 1, E, G, topk_groups, top_k, scale, ids, w) != 0)
            bad = 1;
        for (int k = 0; k < top_k && !bad; ++k) {
            const int64_t e = ids[k];
            expert_swiglu(xb, wg + e * I * H, wu + e * I * H, wd + e * H * I, H, I, hbuf, y);
            for (int j = 0; j < H; ++j)
                acc[j] += (double)w[k] * y[j];
        }
        for (int j = 0; j < H; ++j)
            o[j] = (float)acc[j];
        const float rq = rms_inv(o, H, eps);
        for (int j = 0; j < H; ++j) {
            const float z = (o[j] * rq) * gamma_post[j];
            out[r * H + j] = float_to_bf16_bits_rne(a * sv[j] + b * z);
        }
        free(sv);
        free(xb);
        free(o);
        free(scores);
        free(ids);
        free(w);
        free(hbuf);
        free(y);
        free(acc);
    }
    return bad ? -1 : 0;
}

/*
 * The fused block's post-norm and residual update on a given FP32 layer
 * combine ([P1-RES]): for row r (token t = tokens[r], or r when tokens is
 * NULL), out[r] = bf16( a*s[t] + b*(rmsnorm(o[r]) * gamma_post) ), with a, b,
 * the norm and the roundings exactly as in oracle_block_forward.  With o the
 * o_out of a layer oracle applied to the pre-normed stream, this is the block
 * for any expert format.
 */
int oracle_block_tail(const uint16_t *s, int step, const float *gamma_post, float eps,
                      const float *o, int64_t T, int H, const int64_t *tokens, int64_t n_tokens,
                      uint16_t *out)
{
    if (step < 1)
        return -1;
    const float a = (float)sqrt((double)(step - 1) / (double)step);
    const float b = (float)(1.0 / sqrt((double)step));
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        const float *orow = o + r * H;
        const float rq = rms_inv(orow, H, eps);
        for (int j = 0; j < H; ++j) {
            const float sv = bf16_bits_to_float(s[t * H + j]);
            const float z = (orow[j] * rq) * gamma_post[j];
            out[r * H + j] = float_to_bf16_bits_rne(a * sv + b * z);
        }
    }
    return bad ? -1 : 0;
}

/* the pre-norm alone, for its pins: x = bf16(rmsnorm(s) * gamma) */
void oracle_rmsnorm_bf16(const uint16_t *s, const float *gamma, float eps, int64_t T, int H,
                         uint16_t *x)
{
    float *sv = (float *)malloc(sizeof(float) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h)
            sv[h] = bf16_bits_to_float(s[t * H + h]);
        const float rp = rms_inv(sv, H, eps);
        for (int h = 0; h < H; ++h) {
            const float v = sv[h] * rp;
            x[t * H + h] = float_to_bf16_bits_rne(v * gamma[h]);
        }
    }
    free(sv);
}

/* ------------------------------------------------------------------ NVFP4 */

/* magnitudes of the E2M1 codes 0..7 (bit 3 is the sign) */
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float oracle_e2m1_value(int code)
{
    const float m = kE2M1[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest E2M1 code; a tie goes to the code whose mantissa bit (bit 0) is 0;
   magnitudes beyond 6 take 6; the sign is kept (so -0.1 gives -0). */
int oracle_e2m1_code(float v)
{
    const double a = fabs((double)v);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        const double d = fabs(a - (double)kE2M1[c]);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            bd = d;
            best = c;
        }
    }
    return best | (signbit(v) ? 8 : 0);
}

/* value of an E4M3 code (4 exponent bits, bias 7, 3 mantissa bits; no
   infinities; 0x7F / 0xFF are NaN and never produced here) */
float oracle_e4m3_value(int code)
{
    const int e = (code >> 3) & 15, m = code & 7;
    const float mag = (e == 0) ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return (code & 0x80) ? -mag : mag;
}

/* Nearest non-negative finite E4M3 code for v >= 0 (ties to an even
   mantissa; values beyond 448 take 448). */
int oracle_e4m3_code(float v)
{
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs((double)v - (double)oracle_e4m3_value(c));
        if (d < bd || (d == bd && (c & 1) == 0)) {
            bd = d;
            best = c;
        }
    }
    return best;
}

/* Quantise one row of n (multiple of 16) floats with global scale g:
   codes[n] (one E2M1 code per byte), sf[n/16] (E4M3 codes). */
static void quantize_row(const float *v, int64_t n, float g, uint8_t *codes, uint8_t *sf)
{
    for (int64_t b = 0; b < n / 16; ++b) {
        const float *blk = v + b * 16;
        float bmax = 0.0f;
        for (int i = 0; i < 16; ++i)
            if (fabsf(blk[i]) > bmax)
                bmax = fabsf(blk[i]);
        const float want = (bmax / 6.0f) / g;
        const int sc = oracle_e4m3_code(want);
        sf[b] = (uint8_t)sc;
        const float sfv = oracle_e4m3_value(sc);
        const float den = sfv * g;
        for (int i = 0; i < 16; ++i)
            codes[b * 16 + i] = (sfv == 0.0f) ? 0 : (uint8_t)oracle_e2m1_code(blk[i] / den);
    }
}

/*
 * NVFP4 quantisation of n_mat bf16 matrices [rows, cols] (cols % 16 == 0):
 *   codes [n_mat, rows, cols] one E2M1 code per byte
 *   sf    [n_mat, rows, cols/16] E4M3 codes
 *   gs    [n_mat] FP32 global scales
 */
int oracle_quantize_nvfp4(const uint16_t *w, int64_t n_mat, int64_t rows, int64_t cols,
                          uint8_t *codes, uint8_t *sf, float *gs)
{
    if (cols % 16 != 0)
        return -1;
    for (int64_t mat = 0; mat < n_mat; ++mat) {
        const uint16_t *wm = w + mat * rows * cols;
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * cols; ++i) {
            const float a = fabsf(bf16_bits_to_float(wm[i]));
            if (a > amax)
                amax = a;
        }
        const float g = (amax > 0.0f) ? amax / (6.0f * 448.0f) : 1.0f;
        gs[mat] = g;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            float *row = (float *)malloc(sizeof(float) * (size_t)cols);
            for (int64_t c = 0; c < cols; ++c)
                row[c] = bf16_bits_to_float(wm[r * cols + c]);
            quantize_row(row, cols, g, codes + (mat * rows + r) * cols,
                         sf + (mat * rows + r) * (cols / 16));
            free(row);
        }
    }
    return 0;
}

/* Quantise-then-dequantise a row in place with global scale 1 (activations). */
static void fake_quant_row(float *v, int64_t n)
{
    uint8_t *codes = (uint8_t *)malloc((size_t)n);
    uint8_t *sf = (uint8_t *)malloc((size_t)(n / 16));
    quantize_row(v, n, 1.0f, codes, sf);
    for (int64_t i = 0; i < n; ++i)
        v[i] = oracle_e2m1_value(codes[i]) * oracle_e4m3_value(sf[i / 16]);
    free(codes);
    free(sf);
}

/* exported for the pins: quantise-dequantise rows [n_rows, n] with gs = 1 */
void oracle_fake_quant_rows(float *v, int64_t n_rows, int64_t n)
{
    for (int64_t r = 0; r < n_rows; ++r)
        fake_quant_row(v + r * n, n);
}

static double deq(const uint8_t *codes, const uint8_t *sf, float g, int64_t row, int64_t cols,
                  int64_t c)
{
    return (double)oracle_e2m1_value(codes[row * cols + c]) *
           (double)oracle_e4m3_value(sf[row * (cols / 16) + c / 16]) * (double)g;
}

/*
 * The layer with NVFP4 experts and NVFP4 activations (see the header note):
 * router and selection exactly as oracle_forward; per selected expert,
 *   g, u = xq . deq(Wg)^T, xq . deq(Wu)^T   (FP64 sums, rounded to FP32)
 *   h    = fakequant( silu(g) * u )          (FP32 product, then gs = 1 blocks)
 *   y    = h . deq(Wd)^T                     (FP64)
 * where xq = fakequant(x).  Weight arrays are the outputs of
 * oracle_quantize_nvfp4: codes [E,I,H] / [E,H,I], sf [.., /16], gs [E].
 * scores_in [T,E] fp32 or NULL: given router scores, and o_out [n,H] fp32 or
 * NULL: the FP32 combine, both as in oracle_forward.
 */
int oracle_forward_nvfp4(const uint16_t *x, const float *wr, const uint8_t *gc, const uint8_t *gsf,
                         const float *ggs, const uint8_t *uc, const uint8_t *usf,
                         const float *ugs, const uint8_t *dc, const uint8_t *dsf,
                         const float *dgs, int64_t T, int H, int I, int E, int G,
                         int topk_groups, int top_k, float scale, const int64_t *tokens,
                         int64_t n_tokens, uint16_t *out, int32_t *ids_out, float *w_out,
                         const float *scores_in, float *o_out)
{
    if (E % G != 0 || top_k > topk_groups * (E / G) || H % 16 || I % 16)
        return -1;
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        const uint16_t *xrow = x + t * H;
        float *scores = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
        float *w = (float *)malloc(sizeof(float) * (size_t)top_k);
        float *xq = (float *)malloc(sizeof(float) * (size_t)H);
        float *hq = (float *)malloc(sizeof(float) * (size_t)I);
        double *acc = (double *)calloc((size_t)H, sizeof(double));

        token_scores(xrow, wr, scores_in, t, H, E, scores);
        if (oracle_select(scores, 1, E, G, topk_groups, top_k, scale, ids, w) != 0)
            bad = 1;
        for (int h = 0; h < H; ++h)
            xq[h] = bf16_bits_to_float(xrow[h]);
        fake_quant_row(xq, H);
        for (int k = 0; k < top_k && !bad; ++k) {
            const int64_t e = ids[k];
            for (int i = 0; i < I; ++i) {
                double gd = 0.0, ud = 0.0;
                const int64_t row = e * I + i;
                for (int h = 0; h < H; ++h) {
                    gd += (double)xq[h] * deq(gc, gsf, ggs[e], row, H, h);
                    ud += (double)xq[h] * deq(uc, usf, ugs[e], row, H, h);
                }
                const float g = (float)gd, u = (float)ud;
                hq[i] = (g * sigmoid_f32(g)) * u;
            }
            fake_quant_row(hq, I);
            for (int j = 0; j < H; ++j) {
                double yd = 0.0;
                const int64_t row = e * H + j;
                for (int i = 0; i < I; ++i)
                    yd += (double)hq[i] * deq(dc, dsf, dgs[e], row, I, i);
                acc[j] += (double)w[k] * yd;
            }
        }
        {
            for (int j = 0; j < H; ++j) {
                if (o_out)
                    o_out[r * H + j] = (float)acc[j];
                out[r * H + j] = float_to_bf16_bits_rne((float)acc[j]);
            }
        }
        if (ids_out)
            memcpy(ids_out + r * top_k, ids, sizeof(int32_t) * (size_t)top_k);
        if (w_out)
            memcpy(w_out + r * top_k, w, sizeof(float) * (size_t)top_k);
        free(scores);
        free(ids);
        free(w);
        free(xq);
        free(hq);
        free(acc);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ MXFP8 */

/*
 * MXFP8 expert weights and activations: E4M3 values with one power-of-two
 * (UE8M0) scale per 32 consecutive elements of a row.  The pages only say an
 * FP8 checkpoint exists ([P1-MoE] checkpoints paragraph; [P5] checkpoint
 * list); the recipe is a reading: the OCP microscaling rule, shared exponent
 * E = floor(log2(amax32)) - 8 (8 = the largest E4M3 exponent), clamped to
 * [-127, 127], E = -127 for an all-zero block; q = e4m3_rn_satfinite(v / 2^E);
 * the scale byte is E + 127.  Dequantised value: e4m3(q) * 2^E.
 */
int oracle_mx_shared_exp(float amax)
{
    if (!(amax > 0.0f))
        return -127;
    int ex;
    frexpf(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
    int e = ex - 1 - 8;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return e;
}

/* the finite non-negative E4M3 values, codes 0..126, ascending */
static double kE4M3Pos[127];

static void e4m3_table_init(void)
{
    for (int c = 0; c < 127; ++c)
        kE4M3Pos[c] = (double)oracle_e4m3_value(c);
}

/* signed E4M3 code: the sign bit and the nearest magnitude, as
 * oracle_e4m3_code (ties to the even code, saturating at 448) but found by
 * bisection of the ascending value table; call e4m3_table_init() first */
static int e4m3_code_signed(float v)
{
    const double a = fabs((double)v);
    int c;
    if (a >= kE4M3Pos[126]) {
        c = 126;
    } else {
        int lo = 0, hi = 126; /* largest c with value(c) <= a */
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (kE4M3Pos[mid] <= a)
                lo = mid;
            else
                hi = mid - 1;
        }
        c = lo;
        const double d0 = a - kE4M3Pos[c], d1 = kE4M3Pos[c + 1] - a;
        if (d1 < d0 || (d1 == d0 && ((c + 1) & 1) == 0))
            c = c + 1;
    }
    return (signbit(v) ? 0x80 : 0) | c;
}

static void mx_quantize_row(const float *v, int64_t n, uint8_t *codes, uint8_t *sf)
{
    for (int64_t b = 0; b < n / 32; ++b) {
        const float *blk = v + b * 32;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i)
            if (fabsf(blk[i]) > amax)
                amax = fabsf(blk[i]);
        const int e = oracle_mx_shared_exp(amax);
        sf[b] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; ++i)
            codes[b * 32 + i] = (uint8_t)e4m3_code_signed(ldexpf(blk[i], -e));
    }
}

static double mx_value(uint8_t code, uint8_t sfb)
{
    return ldexp((double)oracle_e4m3_value(code), (int)sfb - 127);
}

/* w [n_mat, rows, cols] bf16 -> codes [n_mat, rows, cols] E4M3 bytes, sf
 * [n_mat, rows, cols/32] UE8M0 bytes (plain row-major layout) */
int oracle_quantize_mxfp8(const uint16_t *w, int64_t n_mat, int64_t rows, int64_t cols,
                          uint8_t *codes, uint8_t *sf)
{
    if (cols % 32 != 0)
        return -1;
    e4m3_table_init();
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n_mat * rows; ++r) {
        float *row = (float *)malloc(sizeof(float) * (size_t)cols);
        for (int64_t c = 0; c < cols; ++c)
            row[c] = bf16_bits_to_float(w[r * cols + c]);
        mx_quantize_row(row, cols, codes + r * cols, sf + r * (cols / 32));
        free(row);
    }
    return 0;
}

/* in place: one row's values <- their MXFP8 values (table already built) */
static void mx_fake_quant_row(float *row, int64_t n)
{
    uint8_t *codes = (uint8_t *)malloc((size_t)n);
    uint8_t *sf = (uint8_t *)malloc((size_t)(n / 32));
    mx_quantize_row(row, n, codes, sf);
    for (int64_t i = 0; i < n; ++i)
        row[i] = (float)mx_value(codes[i], sf[i / 32]);
    free(codes);
    free(sf);
}

/* in place: v[i] <- its MXFP8 value (the activations' quantisation) */
void oracle_fake_quant_mxfp8_rows(float *v, int64_t n_rows, int64_t n)
{
    e4m3_table_init();
    uint8_t *codes = (uint8_t *)malloc((size_t)n);
    uint8_t *sf = (uint8_t *)malloc((size_t)(n / 32));
    for (int64_t r = 0; r < n_rows; ++r) {
        float *row = v + r * n;
        mx_quantize_row(row, n, codes, sf);
        for (int64_t i = 0; i < n; ++i)
            row[i] = (float)mx_value(codes[i], sf[i / 32]);
    }
    free(codes);
    free(sf);
}

/*
 * The layer forward with MXFP8 experts: routing as oracle_forward (FP32 on
 * the bf16 x); x and h quantised to MXFP8 as above; FP64 dot products of
 * the dequantised values; h = silu(g)*u in FP32 from g, u rounded to FP32.
 * scores_in [T,E] fp32 or NULL: given router scores, and o_out [n,H] fp32 or
 * NULL: the FP32 combine, both as in oracle_forward.
 */
int oracle_forward_mxfp8(const uint16_t *x, const float *wr, const uint8_t *gc, const uint8_t *gsf,
                         const uint8_t *uc, const uint8_t *usf, const uint8_t *dc,
                         const uint8_t *dsf, int64_t T, int H, int I, int E, int G,
                         int topk_groups, int top_k, float scale, const int64_t *tokens,
                         int64_t n_tokens, uint16_t *out, int32_t *ids_out, float *w_out,
                         const float *scores_in, float *o_out)
{
    if (E % G != 0 || top_k > topk_groups * (E / G) || H % 32 || I % 32)
        return -1;
    e4m3_table_init();
    const int64_t n = tokens ? n_tokens : T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t r = 0; r < n; ++r) {
        const int64_t t = tokens ? tokens[r] : r;
        if (t < 0 || t >= T) {
            bad = 1;
            continue;
        }
        const uint16_t *xrow = x + t * H;
        float *scores = (float *)malloc(sizeof(float) * (size_t)E);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)top_k);
        float *w = (float *)malloc(sizeof(float) * (size_t)top_k);
        float *xq = (float *)malloc(sizeof(float) * (size_t)H);
        float *hq = (float *)malloc(sizeof(float) * (size_t)I);
        double *acc = (double *)calloc((size_t)H, sizeof(double));

        token_scores(xrow, wr, scores_in, t, H, E, scores);
        if (oracle_select(scores, 1, E, G, topk_groups, top_k, scale, ids, w) != 0)
            bad = 1;
        for (int h = 0; h < H; ++h)
            xq[h] = bf16_bits_to_float(xrow[h]);
        mx_fake_quant_row(xq, H);
        for (int k = 0; k < top_k && !bad; ++k) {
            const int64_t e = ids[k];
            for (int i = 0; i < I; ++i) {
                double gd = 0.0, ud = 0.0;
                const int64_t row = e * I + i;
                for (int h = 0; h < H; ++h) {
                    gd += (double)xq[h] * mx_value(gc[row * H + h], gsf[row * (H / 32) + h / 32]);
                    ud += (double)xq[h] * mx_value(uc[row * H + h], usf[row * (H / 32) + h / 32]);
                }
                const float g = (float)gd, u = (float)ud;
                hq[i] = (g * sigmoid_f32(g)) * u;
            }
            mx_fake_quant_row(hq, I);
            for (int j = 0; j < H; ++j) {
                double yd = 0.0;
                const int64_t row = e * H + j;
                for (int i = 0; i < I; ++i)
                    yd += (double)hq[i] * mx_value(dc[row * I + i], dsf[row * (I / 32) + i / 32]);
                acc[j] += (double)w[k] * yd;
            }
        }
        {
            for (int j = 0; j < H; ++j) {
                if (o_out)
                    o_out[r * H + j] = (float)acc[j];
                out[r * H + j] = float_to_bf16_bits_rne((float)acc[j]);
            }
        }
        if (ids_out)
            memcpy(ids_out + r * top_k, ids, sizeof(int32_t) * (size_t)top_k);
        if (w_out)
            memcpy(w_out + r * top_k, w, sizeof(float) * (size_t)top_k);
        free(scores);
        free(ids);
        free(w);
        free(xq);
        free(hq);
        free(acc);
    }
    return bad ? -1 : 0;
}

