/*
 * moe_ref.h -- plain, slow CPU oracle of the sparse MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library; the two meet only through the seeded
 * input generator.
 *
 * What it computes, step by step, and where each step is stated:
 *   router    sigmoid scores, noaux_tc selection bias that steers the choice
 *             only, iterated-argmax top-k, adaptive top-p, norm_topk_prob,
 *             routed_scaling_factor
 *             ["MoE 路由与专家流式加载" §1.1, §1.2; "colibrì 深度拆解" §3.4]
 *   permute   batch-union of the selected experts; per-expert token lists by
 *             a stable counting sort
 *             ["MoE 路由与专家流式加载" §1.3; "Colibri 是什么" §3.3]
 *   quant     per-row symmetric int8 activation quantisation, done once per
 *             layer ["colibri 开发演进实录" §2.2, layer-level hoist]
 *   ffn       gate/up/SiLU/down on int4 gs64 weights (unsigned nibble, zero
 *             point 8) against int8 activations: int32 dot per 64-group, then
 *             the group scale ["colibri 开发演进实录" §2.1, §2.2 (K1, K1b);
 *             "MoE 路由与专家流式加载" §1.3]
 *   shared    always-on shared expert added to the output
 *             ["MoE 路由与专家流式加载" §1.4]
 *   quantise  offline fp32 -> int4-gs64 weights, symmetric absmax per group
 *             ["colibri 开发演进实录" §2.1], and the int3-g64 variant (fmt=5,
 *             ibid. §8.3)
 *   lookahead RMSNorm then the router, predicting a later layer's top-K from
 *             a residual state, and the recall of such a prediction
 *             ["MoE 路由与专家流式加载" §5]
 *
 * Precision: the router runs in fp32 because the pages' router is float
 * (`sigmoidf`, float32 router gate); the expert FFN combination of group
 * results, SiLU, down projection and combine run in fp64.  Every decision that
 * floating point makes about an integer (an int8 code, an argmax, the top-p
 * cut) is taken in fp32, the precision of the kernel it is compared with.
 *
 * Layouts (host memory, row major):
 *   x [T][H] fp32; w_router [E][H] fp32; bias [E] fp32
 *   w_gate, w_up [E][F][H/2] u8 and s_gate, s_up [E][F][H/64] fp32
 *   w_down [E][H][F/2] u8 and s_down [E][H][F/64] fp32
 *   byte j of a row: low nibble = element 2j, high nibble = element 2j+1;
 *   code u in 0..15 means (u - 8) * scale of its 64-element group.
 * All functions return 0 on success and a negative value on bad arguments.
 */
#ifndef MOE_REF_H
#define MOE_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t hidden;           /* H, multiple of 64 */
    int32_t n_experts;        /* E */
    int32_t top_k;            /* K <= E */
    int32_t d_ff;             /* F, multiple of 64 */
    int32_t n_shared;         /* 0 or 1 */
    int32_t d_ff_shared;      /* Fs, multiple of 64 when n_shared */
    int32_t norm_topk_prob;   /* 0 or 1 */
    float routed_scaling_factor;
    float top_p;              /* in (0,1): adaptive top-p; otherwise off */
} moe_ref_config;

typedef struct {
    const uint8_t *w_gate; const float *s_gate;
    const uint8_t *w_up;   const float *s_up;
    const uint8_t *w_down; const float *s_down;
} moe_ref_weights;

/* Router.  ids [T][K]: kept experts first (selection order, or descending
 * gate when top-p is on), -1 for slots >= keff.  w [T][K]: applied weights,
 * 0 for slots >= keff.  keff [T].  logits [T][E] (nullable): fp32 logits. */
int moe_ref_route(const moe_ref_config *c, const float *x, const float *w_router,
                  const float *bias, int T, int32_t *ids, float *w, int32_t *keff,
                  float *logits);

/* Batch-union.  counts [E], offsets [E+1], tok/slot [sum keff] (ascending
 * token within each expert, slot = t*K + i), uniq [E] (ascending id), n_uniq. */
int moe_ref_permute(const moe_ref_config *c, const int32_t *ids, const int32_t *keff,
                    int T, int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *slot,
                    int32_t *uniq, int32_t *n_uniq);

/* Per-row symmetric int8 quantisation of n fp32 values: q [n], *scale. */
void moe_ref_quant_row(const float *v, int n, int8_t *q, float *scale);
/* The same, also writing pre [n] (nullable): the fp32 value v * (127 / amax) that each
 * code rounds, so a test can tell how close a code lies to a rounding boundary. */
void moe_ref_quant_row_pre(const float *v, int n, int8_t *q, float *scale, float *pre);

/* int32 dot of one 64-group: sum_k (u_k - 8) * q_k for elements 64g..64g+63
 * of a packed row. */
int32_t moe_ref_group_dot(const uint8_t *row, const int8_t *q, int g);

/* One expert applied to one token (gate/up, SiLU*up, h quantisation, down).
 * Pointers are that expert's own matrices ([F][H/2] ...).  xq [H], sx: the
 * token's quantised activations.  y [H] fp64 output.
 * Optional (nullable) probes: acc_gate/acc_up [F][H/64], acc_down [H][F/64]
 * int32 group accumulators; hq_out [F], hs_out: the quantised h.
 * hq_in/hs_in (nullable): run the down projection on this quantised h
 * instead of the one computed here.  hpre_out [F] (nullable): the pre-rounding
 * value of each h code (see moe_ref_quant_row_pre; zeros when hq_in is given). */
int moe_ref_expert_apply(int H, int F, const uint8_t *w_gate, const float *s_gate,
                         const uint8_t *w_up, const float *s_up, const uint8_t *w_down,
                         const float *s_down, const int8_t *xq, float sx, double *y,
                         int32_t *acc_gate, int32_t *acc_up, int32_t *acc_down,
                         int8_t *hq_out, float *hs_out, const int8_t *hq_in,
                         const float *hs_in, float *hpre_out);

/* Routed expert FFN over a permutation: pair p (permuted order) is token
 * tok[p] through expert e with offsets[e] <= p < offsets[e+1].
 * y_pairs [P][H] fp64.  Probes as in moe_ref_expert_apply, indexed by pair:
 * acc_gate/acc_up [P][F][H/64], acc_down [P][H][F/64], hq_out [P][F],
 * hs_out [P], hq_in [P][F], hs_in [P], hpre_out [P][F].  Parallel over pairs
 * (OpenMP). */
int moe_ref_expert_ffn(const moe_ref_config *c, const float *x, int T,
                       const moe_ref_weights *routed, const int32_t *offsets,
                       const int32_t *tok, double *y_pairs, int32_t *acc_gate,
                       int32_t *acc_up, int32_t *acc_down, int8_t *hq_out, float *hs_out,
                       const int8_t *hq_in, const float *hs_in, float *hpre_out);

/* Shared expert over every token: ys [T][H] fp64 (weight 1). */
int moe_ref_shared_ffn(const moe_ref_config *c, const float *x, int T,
                       const moe_ref_weights *shared, double *ys);

/* Combine: y[t] = sum_{i<keff[t]} w[t][i] * y_pairs[pair(t,i)] + ys[t]
 * (ys nullable), summed in slot order, then the shared term.  y [T][H]. */
int moe_ref_combine(const moe_ref_config *c, const double *y_pairs, const int32_t *slot,
                    const int32_t *offsets, const float *w, const int32_t *keff, int T,
                    const double *ys, double *y);

/* Whole layer: route, permute, quantise, routed FFN, shared FFN, combine.
 * y [T][H] fp64.  ids/w/keff (nullable) receive the routing. */
int moe_ref_layer_forward(const moe_ref_config *c, const float *x, int T,
                          const float *w_router, const float *bias,
                          const moe_ref_weights *routed, const moe_ref_weights *shared,
                          double *y, int32_t *ids, float *w, int32_t *keff);

/* Number of OpenMP threads the parallel loops use (1 without OpenMP). */
int moe_ref_threads(void);

/* Router look-ahead ["MoE 路由与专家流式加载" §5, la_predict]: RMSNorm of the
 * residual state x [T][H] with norm_w [H] and eps, then moe_ref_route on the
 * result.  moe_ref_rmsnorm alone writes out [T][H].  moe_ref_topk_hits writes,
 * per token, how many experts the predicted kept set (ids_pred [T][K], first
 * keff_pred[t]) shares with the true one. */
int moe_ref_rmsnorm(const float *x, const float *g, float eps, int T, int H, float *out);
int moe_ref_route_lookahead(const moe_ref_config *c, const float *x, const float *norm_w,
                            float eps, const float *w_router, const float *bias, int T,
                            int32_t *ids, float *w, int32_t *keff, float *logits);
int moe_ref_topk_hits(int T, int K, const int32_t *ids_pred, const int32_t *keff_pred,
                      const int32_t *ids_true, const int32_t *keff_true, int32_t *hits);

/* Offline fp32 -> int4-gs64 weight quantiser ("colibri 开发演进实录" §2.1):
 * per 64-weight group, scale = amax / 7 and u = clamp(rint(w * 7 / amax), -7, 7)
 * + 8 (fp32, round half to even); w [rows][K] -> packed [rows][K/2] (element
 * 2j low nibble) and scales [rows][K/64].  Returns -2 unless K % 64 == 0. */
int moe_ref_quantize_int4(const float *w, int rows, int K, uint8_t *packed, float *scales);

/* Offline fp32 -> int3-g64 weight quantiser (fmt=5, "colibri 开发演进实录" §8.3):
 * per 64-weight group, scale = amax / 3 and u = clamp(rint(w * 3 / amax), -3, 3) + 4
 * (fp32, round half to even); each group packs into 24 bytes, weight k in bits
 * 3k .. 3k+2 of the group's little-endian bit string.  w [rows][K] -> packed
 * [rows][3K/8], scales [rows][K/64].  moe_ref_dequant_int3 writes the values the
 * codes stand for, scale * (u - 4).  Both return -2 unless K % 64 == 0. */
int moe_ref_quantize_int3(const float *w, int rows, int K, uint8_t *packed, float *scales);
int moe_ref_dequant_int3(const uint8_t *packed, const float *scales, int rows, int K, float *out);

#ifdef __cplusplus
}
#endif
#endif
