// router_select.cuh -- expert selection of one token by one warp ["MoE 路由与专家流式加载"
// §1.1, §1.2]: sigmoid scores, the selection bias that only steers the choice (noaux_tc), K
// rounds of iterated argmax over the unchosen experts (ties to the lower id), optional
// adaptive top-p over the kept gates, norm_topk_prob and routed_scaling_factor.
//
// Every decision is taken in fp32 with IEEE operations (__fdiv_rn, __fadd_rn, __fmul_rn):
// given the same logits the warp reproduces the host oracle's choices and weights exactly.
#pragma once

#include "device_util.cuh"
#include "moe_internal.cuh"

namespace moe {

struct SelectParams {
    int E, K, norm;
    float scale, top_p;
    const float *bias;
};

inline SelectParams select_params(const moe_config &c, const float *bias)
{
    SelectParams p;
    p.E = c.n_experts;
    p.K = c.top_k;
    p.norm = c.norm_topk_prob;
    p.scale = c.routed_scaling_factor;
    p.top_p = c.top_p;
    p.bias = bias;
    return p;
}

struct Cand {
    float v;   // choice = sig + bias
    float g;   // sig (the applied gate)
    int e;     // expert id, INT_MAX = none
};

__device__ __forceinline__ bool cand_better(const Cand &a, const Cand &b)
{
    // a beats b: any candidate beats none; larger choice wins; equal choice -> lower id
    if (b.e == 0x7fffffff) return a.e != 0x7fffffff;
    if (a.e == 0x7fffffff) return false;
    return a.v > b.v || (a.v == b.v && a.e < b.e);
}

// One warp; logit(e) returns token t's router logit of expert e.  sel / g are this warp's
// kMaxTopK-entry shared-memory scratch.  Writes ids/w of the token (K entries: the kept ones
// in order, then -1 / 0) and keff[t]; also the ids to sm_ids[0..K) and keff to *sm_keff
// when those are non-null.
template <typename LogitFn>
__device__ void select_token(const SelectParams &p, LogitFn logit, int t, int *sel, float *g,
                             int32_t *__restrict__ ids, float *__restrict__ w,
                             int32_t *__restrict__ keff, int *sm_ids = nullptr,
                             int *sm_keff = nullptr)
{
    constexpr int kPerLane = kMaxExperts / 32;
    const int lane = threadIdx.x & 31;
    const int E = p.E, K = p.K;

    float sig[kPerLane], ch[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int e = lane + 32 * j;
        sig[j] = 0.0f;
        ch[j] = 0.0f;
        if (e < E) {
            const float l = logit(e);
            sig[j] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
            ch[j] = __fadd_rn(sig[j], p.bias[e]);
        }
    }

    unsigned taken = 0;
    for (int k = 0; k < K; ++k) {
        Cand best{0.0f, 0.0f, 0x7fffffff};
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u)) {
                const Cand c{ch[j], sig[j], e};
                if (cand_better(c, best)) best = c;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Cand o;
            o.v = __shfl_xor_sync(0xffffffffu, best.v, off);
            o.g = __shfl_xor_sync(0xffffffffu, best.g, off);
            o.e = __shfl_xor_sync(0xffffffffu, best.e, off);
            if (cand_better(o, best)) best = o;
        }
        if ((best.e & 31) == lane) taken |= 1u << (best.e >> 5);
        if (lane == 0) {
            sel[k] = best.e;
            g[k] = best.g;
        }
    }
    __syncwarp();

    if (lane == 0) {
        int m = K;
        if (p.top_p > 0.0f && p.top_p < 1.0f) {
            // stable insertion sort of the kept gates, descending
            for (int i = 1; i < K; ++i) {
                const float gv = g[i];
                const int sv = sel[i];
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
            for (int i = 0; i < K; ++i) tot = __fadd_rn(tot, g[i]);
            const float thr = __fmul_rn(p.top_p, tot);
            float cum = 0.0f;
            for (int i = 0; i < K; ++i) {
                cum = __fadd_rn(cum, g[i]);
                if (cum >= thr) {
                    m = i + 1;
                    break;
                }
            }
        }
        float ssum = 0.0f;
        for (int i = 0; i < m; ++i) ssum = __fadd_rn(ssum, g[i]);
        for (int i = 0; i < K; ++i) {
            const size_t o = (size_t)t * K + i;
            const int id = i < m ? sel[i] : -1;
            w[o] = i < m ? __fmul_rn(p.norm ? __fdiv_rn(g[i], ssum) : g[i], p.scale) : 0.0f;
            ids[o] = id;
            if (sm_ids) sm_ids[i] = id;
        }
        keff[t] = m;
        if (sm_keff) *sm_keff = m;
    }
    __syncwarp();
}

}  // namespace moe
