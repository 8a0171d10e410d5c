/*
 * moe_ref.c -- plain, slow CPU oracle of the sparse MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_ref.h).  Written for a reader checking it
 * against the pages by eye: no blocking, no fusion, no reordering beyond what
 * each step states.  Build with -ffp-contract=off so that every fp32 multiply
 * and add rounds on its own, on every host.
 */
#include "moe_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GS 64 /* int4 group size: one fp32 scale per 64 weights ("colibri 开发演进实录" §2.1, int4-gs64) */

static int check_config(const moe_ref_config *c)
{
    if (!c) return -1;
    if (c->hidden <= 0 || c->hidden % GS) return -2;
    if (c->n_experts <= 0 || c->top_k <= 0 || c->top_k > c->n_experts) return -2;
    if (c->d_ff <= 0 || c->d_ff % GS) return -2;
    if (c->n_shared < 0 || c->n_shared > 1) return -2;
    if (c->n_shared && (c->d_ff_shared <= 0 || c->d_ff_shared % GS)) return -2;
    return 0;
}

int moe_ref_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * Router ["MoE 路由与专家流式加载" §1.1 sigmoid routing (noaux_tc), §1.2 top-k
 * selection and adaptive top-p, norm_topk_prob, routed_scaling_factor].
 *
 *   logit[e]  = x . W_router[e]                 (fp32, sequential over h)
 *   sig[e]    = 1 / (1 + exp(-logit[e]))        (sigmoidf)
 *   choice[e] = sig[e] + bias[e]                (bias steers the choice only)
 *   K rounds of argmax over choice[] among the experts not yet chosen; the
 *   gate of a chosen expert is its unbiased sig.  Equal choices: the lowest
 *   expert index wins (strict '>' while scanning e upwards).
 *   top-p (0 < p < 1): sort the K gates descending (stable), accumulate and
 *   stop at the first m whose running sum reaches p * total; that expert is
 *   kept.  keff = m.
 *   norm: w_i = g_i / sum_{j<keff} g_j; then w_i *= routed_scaling_factor.
 * With all K = E experts, bias 0, norm on and scale 1 the weights reduce to
 * sig / sum(sig) over all experts ["colibrì 深度拆解" §3.4].
 * ------------------------------------------------------------------------ */
static float sigmoid32(float v)
{
    return 1.0f / (1.0f + expf(-v));
}

/* One token through the router; scratch arrays of E and K entries. */
static void route_token(const moe_ref_config *c, const float *xt, const float *w_router,
                        const float *bias, int32_t *ids, float *w, int32_t *keff, float *logits,
                        float *sig, float *choice, unsigned char *taken, int32_t *sel, float *g)
{
    const int H = c->hidden, E = c->n_experts, K = c->top_k;
    const int topp_on = c->top_p > 0.0f && c->top_p < 1.0f;
    for (int e = 0; e < E; ++e) {
        const float *we = w_router + (size_t)e * H;
        float acc = 0.0f;
        for (int h = 0; h < H; ++h) acc += xt[h] * we[h];
        if (logits) logits[e] = acc;
        sig[e] = sigmoid32(acc);
        choice[e] = sig[e] + bias[e];
    }

    /* iterated argmax, excluding the experts already chosen */
    memset(taken, 0, (size_t)E);
    for (int k = 0; k < K; ++k) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || choice[e] > choice[best]) best = e;
        }
        taken[best] = 1;
        sel[k] = best;
        g[k] = sig[best];
    }

    int m = K;
    if (topp_on) {
        /* stable insertion sort by gate, descending */
        for (int i = 1; i < K; ++i) {
            float gv = g[i];
            int32_t sv = sel[i];
            int j = i;
            while (j > 0 && g[j - 1] < gv) {
                g[j] = g[j - 1];
                sel[j] = sel[j - 1];
                --j;
            }
            g[j] = gv;
            sel[j] = sv;
        }
        float tot = 0.0f;
        for (int i = 0; i < K; ++i) tot += g[i];
        const float thr = c->top_p * tot;
        float cum = 0.0f;
        for (int i = 0; i < K; ++i) {
            cum += g[i];
            if (cum >= thr) { m = i + 1; break; }
        }
    }

    float s = 0.0f;
    for (int i = 0; i < m; ++i) s += g[i];
    for (int i = 0; i < K; ++i) {
        if (i < m) {
            float v = c->norm_topk_prob ? g[i] / s : g[i];
            w[i] = v * c->routed_scaling_factor;
            ids[i] = sel[i];
        } else {
            w[i] = 0.0f;
            ids[i] = -1;
        }
    }
    *keff = m;
}

int moe_ref_route(const moe_ref_config *c, const float *x, const float *w_router,
                  const float *bias, int T, int32_t *ids, float *w, int32_t *keff,
                  float *logits)
{
    int rc = check_config(c);
    if (rc) return rc;
    if (T < 0 || (T > 0 && (!x || !w_router || !bias || !ids || !w || !keff))) return -1;
    const int H = c->hidden, E = c->n_experts, K = c->top_k;
    int err = 0;
#pragma omp parallel reduction(| : err)
    {
        float *sig = (float *)malloc(sizeof(float) * E);
        float *choice = (float *)malloc(sizeof(float) * E);
        unsigned char *taken = (unsigned char *)malloc(E);
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * K);
        float *g = (float *)malloc(sizeof(float) * K);
        if (!sig || !choice || !taken || !sel || !g) {
            err = 1;
        } else {
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t)
                route_token(c, x + (size_t)t * H, w_router, bias, ids + (size_t)t * K,
                            w + (size_t)t * K, keff + t, logits ? logits + (size_t)t * E : NULL,
                            sig, choice, taken, sel, g);
        }
        free(sig); free(choice); free(taken); free(sel); free(g);
    }
    return err ? -3 : 0;
}

/* ------------------------------------------------------------------------
 * Batch-union ["MoE 路由与专家流式加载" §1.3]: the experts chosen by all
 * positions of the batch are deduplicated so each is read once and applied to
 * every position routed to it.  Grouping by counting sort, O(N + E)
 * ["Colibri 是什么" §3.3]: count per expert, exclusive prefix sum, then place
 * pairs in ascending (token, slot) order, which keeps each list stable.
 * ------------------------------------------------------------------------ */
int moe_ref_permute(const moe_ref_config *c, const int32_t *ids, const int32_t *keff,
                    int T, int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *slot,
                    int32_t *uniq, int32_t *n_uniq)
{
    int rc = check_config(c);
    if (rc) return rc;
    const int E = c->n_experts, K = c->top_k;
    if (T < 0 || !counts || !offsets || !uniq || !n_uniq) return -1;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int t = 0; t < T; ++t) {
        if (keff[t] < 0 || keff[t] > K) return -2;
        for (int i = 0; i < keff[t]; ++i) {
            int e = ids[(size_t)t * K + i];
            if (e < 0 || e >= E) return -2;
            counts[e] += 1;
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * E);
    if (!fill) return -3;
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < keff[t]; ++i) {
            int e = ids[(size_t)t * K + i];
            int p = fill[e]++;
            tok[p] = t;
            slot[p] = t * K + i;
        }
    }
    free(fill);

    int n = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0) uniq[n++] = e;
    *n_uniq = n;
    return 0;
}

/* ------------------------------------------------------------------------
 * Activation quantisation: the pages say only that the activation vector is
 * quantised to int8 once per layer for the integer dot
 * ["colibri 开发演进实录" §2.2]; the scheme below is the plain reading:
 * symmetric, per row, scale amax/127, round to nearest even, clamp to +-127.
 * All in fp32, the precision of the kernel it is compared with.
 * ------------------------------------------------------------------------ */
void moe_ref_quant_row(const float *v, int n, int8_t *q, float *scale)
{
    moe_ref_quant_row_pre(v, n, q, scale, NULL);
}

void moe_ref_quant_row_pre(const float *v, int n, int8_t *q, float *scale, float *pre)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int i = 0; i < n; ++i) {
            q[i] = 0;
            if (pre) pre[i] = 0.0f;
        }
        *scale = 0.0f;
        return;
    }
    const float inv = 127.0f / amax;
    for (int i = 0; i < n; ++i) {
        const float p = v[i] * inv;   /* the value the code rounds */
        if (pre) pre[i] = p;
        float r = rintf(p);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    *scale = amax / 127.0f;
}

/* ------------------------------------------------------------------------
 * int4 x int8 group dot ["colibri 开发演进实录" §2.1 int4-gs64, §2.2 K1/K1b]:
 * nibbles are stored unsigned with zero point 8, so the signed weight is
 * (u - 8); element k sits in byte k/2, low nibble for even k
 * ["colibrì 深度拆解" §5.2 pack order].  The sum over one 64-group is exact in
 * int32 (|sum| <= 64 * 8 * 127).
 * ------------------------------------------------------------------------ */
static int nibble_at(const uint8_t *row, int k)
{
    uint8_t b = row[k >> 1];
    return (k & 1) ? (b >> 4) : (b & 0x0F);
}

int32_t moe_ref_group_dot(const uint8_t *row, const int8_t *q, int g)
{
    int32_t acc = 0;
    for (int k = g * GS; k < (g + 1) * GS; ++k) acc += (nibble_at(row, k) - 8) * (int32_t)q[k];
    return acc;
}

/* One matrix row against a quantised vector of length n:
 * act_scale * sum_g row_scale[g] * A[g], fp64. */
static double row_dot(const uint8_t *row, const float *row_scales, const int8_t *q, int n,
                      float act_scale, int32_t *acc_out)
{
    double s = 0.0;
    for (int g = 0; g < n / GS; ++g) {
        int32_t a = moe_ref_group_dot(row, q, g);
        if (acc_out) acc_out[g] = a;
        s += (double)row_scales[g] * (double)a;
    }
    return (double)act_scale * s;
}

/* ------------------------------------------------------------------------
 * Expert FFN for one (expert, token) ["MoE 路由与专家流式加载" §1.3: gate, up,
 * SiLU, down, four matrix products on the integer-dot path]:
 *   gate = Wg . x,  up = Wu . x,  h = silu(gate) * up = gate / (1 + e^-gate) * up
 *   h is quantised per row like x (decision in fp32), then y = Wd . h.
 * ------------------------------------------------------------------------ */
int moe_ref_expert_apply(int H, int F, const uint8_t *w_gate, const float *s_gate,
                         const uint8_t *w_up, const float *s_up, const uint8_t *w_down,
                         const float *s_down, const int8_t *xq, float sx, double *y,
                         int32_t *acc_gate, int32_t *acc_up, int32_t *acc_down,
                         int8_t *hq_out, float *hs_out, const int8_t *hq_in,
                         const float *hs_in, float *hpre_out)
{
    if (H <= 0 || F <= 0 || H % GS || F % GS) return -2;
    const int GH = H / GS, GF = F / GS;
    float *h32 = (float *)malloc(sizeof(float) * F);
    int8_t *hq = (int8_t *)malloc((size_t)F);
    if (!h32 || !hq) { free(h32); free(hq); return -3; }

    for (int r = 0; r < F; ++r) {
        double gate = row_dot(w_gate + (size_t)r * (H / 2), s_gate + (size_t)r * GH, xq, H, sx,
                              acc_gate ? acc_gate + (size_t)r * GH : NULL);
        double up = row_dot(w_up + (size_t)r * (H / 2), s_up + (size_t)r * GH, xq, H, sx,
                            acc_up ? acc_up + (size_t)r * GH : NULL);
        double h = gate / (1.0 + exp(-gate)) * up;
        h32[r] = (float)h;
    }

    float hs;
    if (hq_in) {
        memcpy(hq, hq_in, (size_t)F);
        hs = *hs_in;
        if (hpre_out) memset(hpre_out, 0, sizeof(float) * (size_t)F);
    } else {
        moe_ref_quant_row_pre(h32, F, hq, &hs, hpre_out);
    }
    if (hq_out) memcpy(hq_out, hq, (size_t)F);
    if (hs_out) *hs_out = hs;

    for (int r = 0; r < H; ++r)
        y[r] = row_dot(w_down + (size_t)r * (F / 2), s_down + (size_t)r * GF, hq, F, hs,
                       acc_down ? acc_down + (size_t)r * GF : NULL);
    free(h32);
    free(hq);
    return 0;
}

static int quantise_tokens(const float *x, int T, int H, int8_t **xq, float **sx)
{
    *xq = (int8_t *)malloc((size_t)T * H + 1);
    *sx = (float *)malloc(sizeof(float) * (size_t)T + 4);
    if (!*xq || !*sx) { free(*xq); free(*sx); return -3; }
    for (int t = 0; t < T; ++t) moe_ref_quant_row(x + (size_t)t * H, H, *xq + (size_t)t * H, *sx + t);
    return 0;
}

int moe_ref_expert_ffn(const moe_ref_config *c, const float *x, int T,
                       const moe_ref_weights *rw, const int32_t *offsets,
                       const int32_t *tok, double *y_pairs, int32_t *acc_gate,
                       int32_t *acc_up, int32_t *acc_down, int8_t *hq_out, float *hs_out,
                       const int8_t *hq_in, const float *hs_in, float *hpre_out)
{
    int rc = check_config(c);
    if (rc) return rc;
    const int H = c->hidden, F = c->d_ff, E = c->n_experts;
    const int GH = H / GS, GF = F / GS;
    const int P = offsets[E];
    int8_t *xq; float *sx;
    if ((rc = quantise_tokens(x, T, H, &xq, &sx))) return rc;

    /* expert of every pair */
    int32_t *pe = (int32_t *)malloc(sizeof(int32_t) * ((size_t)P + 1));
    if (!pe) { free(xq); free(sx); return -3; }
    for (int e = 0; e < E; ++e)
        for (int p = offsets[e]; p < offsets[e + 1]; ++p) pe[p] = e;

    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int p = 0; p < P; ++p) {
        const int e = pe[p], t = tok[p];
        const size_t up_off = (size_t)e * F * (H / 2), ups = (size_t)e * F * GH;
        const size_t dn_off = (size_t)e * H * (F / 2), dns = (size_t)e * H * GF;
        err |= moe_ref_expert_apply(
            H, F, rw->w_gate + up_off, rw->s_gate + ups, rw->w_up + up_off, rw->s_up + ups,
            rw->w_down + dn_off, rw->s_down + dns, xq + (size_t)t * H, sx[t],
            y_pairs + (size_t)p * H,
            acc_gate ? acc_gate + (size_t)p * F * GH : NULL,
            acc_up ? acc_up + (size_t)p * F * GH : NULL,
            acc_down ? acc_down + (size_t)p * H * GF : NULL,
            hq_out ? hq_out + (size_t)p * F : NULL, hs_out ? hs_out + p : NULL,
            hq_in ? hq_in + (size_t)p * F : NULL, hs_in ? hs_in + p : NULL,
            hpre_out ? hpre_out + (size_t)p * F : NULL) != 0;
    }
    free(pe); free(xq); free(sx);
    return err ? -3 : 0;
}

/* Shared expert ["MoE 路由与专家流式加载" §1.4]: every token, weight 1. */
int moe_ref_shared_ffn(const moe_ref_config *c, const float *x, int T,
                       const moe_ref_weights *sw, double *ys)
{
    int rc = check_config(c);
    if (rc) return rc;
    if (!c->n_shared) return -1;
    const int H = c->hidden, F = c->d_ff_shared;
    int8_t *xq; float *sx;
    if ((rc = quantise_tokens(x, T, H, &xq, &sx))) return rc;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int t = 0; t < T; ++t)
        err |= moe_ref_expert_apply(H, F, sw->w_gate, sw->s_gate, sw->w_up, sw->s_up, sw->w_down,
                                    sw->s_down, xq + (size_t)t * H, sx[t], ys + (size_t)t * H,
                                    NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL) != 0;
    free(xq); free(sx);
    return err ? -3 : 0;
}

/* Combine ["MoE 路由与专家流式加载" §1.3, §1.4]: gated sum of the token's
 * kept experts, in slot order, plus the shared expert. */
int moe_ref_combine(const moe_ref_config *c, const double *y_pairs, const int32_t *slot,
                    const int32_t *offsets, const float *w, const int32_t *keff, int T,
                    const double *ys, double *y)
{
    int rc = check_config(c);
    if (rc) return rc;
    const int H = c->hidden, K = c->top_k, E = c->n_experts;
    const int P = offsets[E];
    int32_t *pair_of = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * K + 1));
    if (!pair_of) return -3;
    for (int i = 0; i < T * K; ++i) pair_of[i] = -1;
    for (int p = 0; p < P; ++p) pair_of[slot[p]] = p;
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int i = 0; i < keff[t]; ++i) {
                int p = pair_of[t * K + i];
                acc += (double)w[(size_t)t * K + i] * y_pairs[(size_t)p * H + h];
            }
            if (ys) acc += ys[(size_t)t * H + h];
            y[(size_t)t * H + h] = acc;
        }
    }
    free(pair_of);
    return 0;
}

int moe_ref_layer_forward(const moe_ref_config *c, const float *x, int T,
                          const float *w_router, const float *bias,
                          const moe_ref_weights *routed, const moe_ref_weights *shared,
                          double *y, int32_t *ids_out, float *w_out, int32_t *keff_out)
{
    int rc = check_config(c);
    if (rc) return rc;
    const int H = c->hidden, E = c->n_experts, K = c->top_k;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * K + 1));
    float *w = (float *)malloc(sizeof(float) * ((size_t)T * K + 1));
    int32_t *keff = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T + 1));
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * E);
    int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (E + 1));
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * K + 1));
    int32_t *slot = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * K + 1));
    int32_t *uniq = (int32_t *)malloc(sizeof(int32_t) * E);
    double *y_pairs = (double *)malloc(sizeof(double) * ((size_t)T * K * H + 1));
    double *ys = (c->n_shared && shared) ? (double *)malloc(sizeof(double) * ((size_t)T * H + 1)) : NULL;
    int32_t n_uniq = 0;
    rc = -3;
    if (!ids || !w || !keff || !counts || !offsets || !tok || !slot || !uniq || !y_pairs ||
        (c->n_shared && shared && !ys))
        goto done;
    if ((rc = moe_ref_route(c, x, w_router, bias, T, ids, w, keff, NULL))) goto done;
    if ((rc = moe_ref_permute(c, ids, keff, T, counts, offsets, tok, slot, uniq, &n_uniq))) goto done;
    if ((rc = moe_ref_expert_ffn(c, x, T, routed, offsets, tok, y_pairs, NULL, NULL, NULL, NULL,
                                 NULL, NULL, NULL, NULL)))
        goto done;
    if (ys && (rc = moe_ref_shared_ffn(c, x, T, shared, ys))) goto done;
    rc = moe_ref_combine(c, y_pairs, slot, offsets, w, keff, T, ys, y);
    if (!rc) {
        if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)T * K);
        if (w_out) memcpy(w_out, w, sizeof(float) * (size_t)T * K);
        if (keff_out) memcpy(keff_out, keff, sizeof(int32_t) * (size_t)T);
    }
done:
    free(ids); free(w); free(keff); free(counts); free(offsets); free(tok); free(slot);
    free(uniq); free(y_pairs); free(ys);
    return rc;
}

/* ------------------------------------------------------------------------
 * Router look-ahead ["MoE 路由与专家流式加载" §5, la_predict]: a layer's
 * top-K is predicted from the residual state of an earlier point by the real
 * routing pipeline -- RMSNorm with the layer's norm weight, then its router
 * (sigmoid, bias for the choice, top-K; §1.1, §1.2).
 *
 *   rms      = sqrt(mean_h x[h]^2 + eps)
 *   out[h]   = x[h] / rms * g[h]
 * The mean of squares, the root and the products run in fp64; the result is
 * rounded to fp32, the router's input precision.  A row whose mean of squares
 * plus eps is 0 (all zeros with eps = 0) normalises to zeros.
 *
 * The pages' measure of the predictor is its recall of the true top-8 (71.6%):
 * per token, hits = the number of experts kept by both the prediction and the
 * true routing; recall = sum(hits) / sum(true keff).
 * ------------------------------------------------------------------------ */
int moe_ref_rmsnorm(const float *x, const float *g, float eps, int T, int H, float *out)
{
    if (T < 0 || H <= 0 || !(eps >= 0.0f)) return -1;
    if (T > 0 && (!x || !g || !out)) return -1;
    for (int t = 0; t < T; ++t) {
        const float *xt = x + (size_t)t * H;
        double ss = 0.0;
        for (int h = 0; h < H; ++h) ss += (double)xt[h] * (double)xt[h];
        const double ms = ss / (double)H + (double)eps;
        const double inv = ms > 0.0 ? 1.0 / sqrt(ms) : 0.0;
        for (int h = 0; h < H; ++h)
            out[(size_t)t * H + h] = (float)((double)xt[h] * inv * (double)g[h]);
    }
    return 0;
}

int moe_ref_route_lookahead(const moe_ref_config *c, const float *x, const float *norm_w,
                            float eps, const float *w_router, const float *bias, int T,
                            int32_t *ids, float *w, int32_t *keff, float *logits)
{
    int rc = check_config(c);
    if (rc) return rc;
    if (T < 0 || (T > 0 && (!x || !norm_w || !w_router || !bias || !ids || !w || !keff))) return -1;
    if (T == 0) return 0;
    const int H = c->hidden;
    float *xn = (float *)malloc(sizeof(float) * (size_t)T * H);
    if (!xn) return -3;
    rc = moe_ref_rmsnorm(x, norm_w, eps, T, H, xn);
    if (!rc) rc = moe_ref_route(c, xn, w_router, bias, T, ids, w, keff, logits);
    free(xn);
    return rc;
}

int moe_ref_topk_hits(int T, int K, const int32_t *ids_pred, const int32_t *keff_pred,
                      const int32_t *ids_true, const int32_t *keff_true, int32_t *hits)
{
    if (T < 0 || K <= 0) return -1;
    if (T > 0 && (!ids_pred || !keff_pred || !ids_true || !keff_true || !hits)) return -1;
    for (int t = 0; t < T; ++t) {
        const int kp = keff_pred[t] < 0 ? 0 : (keff_pred[t] > K ? K : keff_pred[t]);
        const int kt = keff_true[t] < 0 ? 0 : (keff_true[t] > K ? K : keff_true[t]);
        int n = 0;
        for (int i = 0; i < kp; ++i) {
            const int32_t e = ids_pred[(size_t)t * K + i];
            for (int j = 0; j < kt; ++j)
                if (ids_true[(size_t)t * K + j] == e) {
                    ++n;
                    break;
                }
        }
        hits[t] = n;
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Offline weight quantiser: fp32 -> int4-gs64 (the container format the pages
 * recommend, "colibri 开发演进实录" §2.1 int4-gs64; the conversion tool is
 * `coli convert`, ibid. §9).  The scale rule is not stated; the reading
 * taken is the symmetric absmax one of the activations, per 64-weight group:
 *   amax  = max |w|   over the group
 *   scale = amax / 7                  (fp32)
 *   u     = clamp(rint(w * (7 / amax)), -7, 7) + 8   (round half to even, fp32)
 * so the group's largest magnitude lands on +-7 and value = scale * (u - 8);
 * an all-zero group gets scale 0 and codes 8.  Packing as the layer reads it:
 * byte j of a row holds element 2j in the low nibble and 2j+1 in the high.
 *   w [rows][K] fp32, K a multiple of 64 -> packed [rows][K/2] u8,
 *   scales [rows][K/64] fp32.
 * ------------------------------------------------------------------------ */
int moe_ref_quantize_int4(const float *w, int rows, int K, uint8_t *packed, float *scales)
{
    if (rows < 0 || K <= 0 || K % GS) return -2;
    if (rows > 0 && (!w || !packed || !scales)) return -1;
    const int G = K / GS;
    for (int r = 0; r < rows; ++r) {
        for (int g = 0; g < G; ++g) {
            const float *v = w + (size_t)r * K + (size_t)g * GS;
            float amax = 0.0f;
            for (int k = 0; k < GS; ++k) {
                const float a = fabsf(v[k]);
                if (a > amax) amax = a;
            }
            const float inv = amax > 0.0f ? 7.0f / amax : 0.0f;
            scales[(size_t)r * G + g] = amax / 7.0f;
            uint8_t *out = packed + (size_t)r * (K / 2) + (size_t)g * (GS / 2);
            for (int j = 0; j < GS / 2; ++j) {
                int u[2];
                for (int h = 0; h < 2; ++h) {
                    const float p = v[2 * j + h] * inv;
                    float q = rintf(p);
                    if (q > 7.0f) q = 7.0f;
                    if (q < -7.0f) q = -7.0f;
                    u[h] = (int)q + 8;
                }
                out[j] = (uint8_t)(u[0] | (u[1] << 4));
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Offline fp32 -> int3-g64 weight quantiser (fmt=5 of "colibri 开发演进实录"
 * §8.3: 3-bit weights with one scale per 64-weight group).  The pages give the
 * container, not the rule or the bit packing; the readings taken follow the
 * int4-gs64 quantiser above with three bits:
 *   amax  = max |w|   over the group
 *   scale = amax / 3                  (fp32)
 *   u     = clamp(rint(w * (3 / amax)), -3, 3) + 4   (round half to even, fp32)
 * so value = scale * (u - 4) and u = 0 is unused; an all-zero group gets scale 0
 * and codes 4.  Packing: a group is 24 bytes holding a 192-bit little-endian bit
 * string, weight k of the group in bits 3k .. 3k+2 (bit b in byte b / 8, bit
 * b % 8 of that byte, least significant first).
 *   w [rows][K] fp32, K a multiple of 64 -> packed [rows][3K/8] u8,
 *   scales [rows][K/64] fp32.
 * ------------------------------------------------------------------------ */
#define I3_GROUP_BYTES 24 /* 64 weights x 3 bits */

static void put_bits3(uint8_t *grp, int k, int u)
{
    for (int j = 0; j < 3; ++j) {
        const int b = 3 * k + j;
        if ((u >> j) & 1) grp[b >> 3] |= (uint8_t)(1u << (b & 7));
    }
}

static int get_bits3(const uint8_t *grp, int k)
{
    int u = 0;
    for (int j = 0; j < 3; ++j) {
        const int b = 3 * k + j;
        u |= ((grp[b >> 3] >> (b & 7)) & 1) << j;
    }
    return u;
}

int moe_ref_quantize_int3(const float *w, int rows, int K, uint8_t *packed, float *scales)
{
    if (rows < 0 || K <= 0 || K % GS) return -2;
    if (rows > 0 && (!w || !packed || !scales)) return -1;
    const int G = K / GS;
    for (int r = 0; r < rows; ++r) {
        for (int g = 0; g < G; ++g) {
            const float *v = w + (size_t)r * K + (size_t)g * GS;
            float amax = 0.0f;
            for (int k = 0; k < GS; ++k) {
                const float a = fabsf(v[k]);
                if (a > amax) amax = a;
            }
            const float inv = amax > 0.0f ? 3.0f / amax : 0.0f;
            scales[(size_t)r * G + g] = amax / 3.0f;
            uint8_t *grp = packed + ((size_t)r * G + g) * I3_GROUP_BYTES;
            memset(grp, 0, I3_GROUP_BYTES);
            for (int k = 0; k < GS; ++k) {
                const float p = v[k] * inv;
                float q = rintf(p);
                if (q > 3.0f) q = 3.0f;
                if (q < -3.0f) q = -3.0f;
                put_bits3(grp, k, (int)q + 4);
            }
        }
    }
    return 0;
}

/* The values an int3-g64 matrix stands for: out[r][k] = scale(r, k/64) * (u - 4). */
int moe_ref_dequant_int3(const uint8_t *packed, const float *scales, int rows, int K, float *out)
{
    if (rows < 0 || K <= 0 || K % GS) return -2;
    if (rows > 0 && (!packed || !scales || !out)) return -1;
    const int G = K / GS;
    for (int r = 0; r < rows; ++r)
        for (int g = 0; g < G; ++g) {
            const uint8_t *grp = packed + ((size_t)r * G + g) * I3_GROUP_BYTES;
            const float s = scales[(size_t)r * G + g];
            for (int k = 0; k < GS; ++k)
                out[(size_t)r * K + (size_t)g * GS + k] = s * (float)(get_bits3(grp, k) - 4);
        }
    return 0;
}
