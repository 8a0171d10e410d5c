// router_select.cuh -- expert selection of one token by one warp ["MoE 路由与专家流式加载"
// §1.1, §1.2]: sigmoid scores, the selection bias that only steers the choice (noaux_tc), K
// rounds of iterated argmax over the unchosen experts (ties to the lower id), optional
// adaptive top-p over the kept gates, norm_topk_prob and routed_scaling_factor.
//
// Every decision is taken in fp32 with IEEE operations (__frcp_rn, __fdiv_rn, __fadd_rn,
// __fmul_rn): given the same logits the warp reproduces the host oracle's choices and
// weights exactly.
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

// Order-preserving map of an fp32 value (not NaN) to uint32, so that comparing keys as
// unsigned integers compares the values.  -0 is first turned into +0 (x + 0 in round to
// nearest), so values that compare equal as fp32 get equal keys.  Every key is above 0,
// which marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float v)
{
    const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp; logit(e) returns token t's router logit of expert e.  Writes ids/w of the token
// (K entries: the kept ones in order, then -1 / 0) and keff[t]; also the ids to sm_ids[0..K)
// and keff to *sm_keff when those are non-null.
//
// Each of the K rounds takes, over the experts not chosen yet, the largest choice value
// (ties to the lower id): every lane finds its best candidate among its experts
// e = lane + 32j, one warp max-reduction finds the best value and one min-reduction the
// lowest id holding it.  After the rounds lane k holds the k-th choice; top-p, the sums
// (sequential, in the oracle's order) and the divisions then run on those lanes.
//
// PL is the experts each lane holds (E <= 32 * PL); select_token below picks it from E.
// select_from_scores takes over once the lane holds its experts' gates and choice keys.
template <int PL>
__device__ void select_from_scores(const SelectParams &p, const float (&sig)[PL],
                                   uint32_t (&key)[PL], int t, int32_t *__restrict__ ids,
                                   float *__restrict__ w, int32_t *__restrict__ keff,
                                   int *sm_ids, int *sm_keff);

// The sigmoid gate of a logit, 1 / (1 + e^-l) rounded once (the correctly rounded
// reciprocal is the correctly rounded quotient 1 / d), and its choice key.
__device__ __forceinline__ void score_expert(float l, float bias, float &sig, uint32_t &key)
{
    sig = __frcp_rn(__fadd_rn(1.0f, expf(-l)));
    key = order_key(__fadd_rn(sig, bias));
}

template <int PL, typename LogitFn>
__device__ void select_token_pl(const SelectParams &p, LogitFn logit, int t,
                                int32_t *__restrict__ ids, float *__restrict__ w,
                                int32_t *__restrict__ keff, int *sm_ids, int *sm_keff)
{
    constexpr int kPerLane = PL;
    const int lane = threadIdx.x & 31;
    const int E = p.E;

    // every logit and bias of this lane is loaded before any of them is used, so the loads
    // overlap instead of queueing behind each other's arithmetic
    float lv[kPerLane], bv[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int e = lane + 32 * j;
        lv[j] = 0.0f;
        bv[j] = 0.0f;
        if (e < E) {
            lv[j] = logit(e);
            bv[j] = p.bias[e];
        }
    }
    float sig[kPerLane];
    uint32_t key[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int e = lane + 32 * j;
        sig[j] = 0.0f;
        key[j] = 0u;
        if (e < E) score_expert(lv[j], bv[j], sig[j], key[j]);
    }
    select_from_scores<PL>(p, sig, key, t, ids, w, keff, sm_ids, sm_keff);
}

// The same selection from gates and keys already in shared memory (sig_s[e], key_s[e] for the
// token's E experts, from score_expert).
template <int PL>
__device__ void select_token_staged_pl(const SelectParams &p, const float *sig_s,
                                       const uint32_t *key_s, int t, int32_t *__restrict__ ids,
                                       float *__restrict__ w, int32_t *__restrict__ keff,
                                       int *sm_ids, int *sm_keff)
{
    const int lane = threadIdx.x & 31;
    float sig[PL];
    uint32_t key[PL];
#pragma unroll
    for (int j = 0; j < PL; ++j) {
        const int e = lane + 32 * j;
        sig[j] = e < p.E ? sig_s[e] : 0.0f;
        key[j] = e < p.E ? key_s[e] : 0u;
    }
    select_from_scores<PL>(p, sig, key, t, ids, w, keff, sm_ids, sm_keff);
}

template <int PL>
__device__ void select_from_scores(const SelectParams &p, const float (&sig)[PL],
                                   uint32_t (&key)[PL], int t, int32_t *__restrict__ ids,
                                   float *__restrict__ w, int32_t *__restrict__ keff,
                                   int *sm_ids, int *sm_keff)
{
    constexpr int kPerLane = PL;
    constexpr unsigned kAll = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int K = p.K;
    int my_id = -1;       // lane k < K: the k-th chosen expert
    float my_g = 0.0f;    // and its gate (the unbiased sigmoid)
    for (int k = 0; k < K; ++k) {
        uint32_t bk = 0u;
        int bj = 0;
        float bg = 0.0f;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            if (key[j] > bk) {   // strict: the lower id of this lane wins a tie
                bk = key[j];
                bj = j;
                bg = sig[j];
            }
        }
        const uint32_t wk = __reduce_max_sync(kAll, bk);
        const uint32_t mine = (bk == wk && bk != 0u) ? (uint32_t)(lane + 32 * bj) : 0xffffffffu;
        const uint32_t we = __reduce_min_sync(kAll, mine);
        const float wg = __shfl_sync(kAll, bg, (int)(we & 31u));
        if (mine == we) {
#pragma unroll
            for (int j = 0; j < kPerLane; ++j)
                if (j == bj) key[j] = 0u;
        }
        if (lane == k) {
            my_id = (int)we;
            my_g = wg;
        }
    }

    int m = K;
    if (p.top_p > 0.0f && p.top_p < 1.0f) {
        // stable sort of the K choices by gate, descending: lane i's rank
        int rank = 0;
        for (int j = 0; j < K; ++j) {
            const float gj = __shfl_sync(kAll, my_g, j);
            rank += (gj > my_g || (gj == my_g && j < lane)) ? 1 : 0;
        }
        int src = 0;
        for (int j = 0; j < K; ++j) src = __shfl_sync(kAll, rank, j) == lane ? j : src;
        my_g = __shfl_sync(kAll, my_g, src);
        my_id = __shfl_sync(kAll, my_id, src);
        // sequential sums, in every lane alike
        float tot = 0.0f;
        for (int i = 0; i < K; ++i) tot = __fadd_rn(tot, __shfl_sync(kAll, my_g, i));
        const float thr = __fmul_rn(p.top_p, tot);
        float cum = 0.0f;
        for (int i = 0; i < K; ++i) {
            cum = __fadd_rn(cum, __shfl_sync(kAll, my_g, i));
            if (cum >= thr) {
                m = i + 1;
                break;
            }
        }
    }
    float ssum = 0.0f;
    for (int i = 0; i < m; ++i) ssum = __fadd_rn(ssum, __shfl_sync(kAll, my_g, i));
    if (lane < K) {
        const size_t o = (size_t)t * K + lane;
        const int id = lane < m ? my_id : -1;
        w[o] = lane < m ? __fmul_rn(p.norm ? __fdiv_rn(my_g, ssum) : my_g, p.scale) : 0.0f;
        ids[o] = id;
        if (sm_ids) sm_ids[lane] = id;
    }
    if (lane == 0) {
        keff[t] = m;
        if (sm_keff) *sm_keff = m;
    }
    __syncwarp();
}

template <typename LogitFn>
__device__ __forceinline__ void select_token(const SelectParams &p, LogitFn logit, int t,
                                             int32_t *__restrict__ ids, float *__restrict__ w,
                                             int32_t *__restrict__ keff, int *sm_ids = nullptr,
                                             int *sm_keff = nullptr)
{
    static_assert(kMaxExperts <= 32 * 16, "one warp holds at most 16 experts per lane");
    if (p.E <= 32 * 4) select_token_pl<4>(p, logit, t, ids, w, keff, sm_ids, sm_keff);
    else if (p.E <= 32 * 8) select_token_pl<8>(p, logit, t, ids, w, keff, sm_ids, sm_keff);
    else select_token_pl<16>(p, logit, t, ids, w, keff, sm_ids, sm_keff);
}

__device__ __forceinline__ void select_token_staged(const SelectParams &p, const float *sig_s,
                                                    const uint32_t *key_s, int t, int32_t *ids,
                                                    float *w, int32_t *keff, int *sm_ids,
                                                    int *sm_keff)
{
    if (p.E <= 32 * 4) select_token_staged_pl<4>(p, sig_s, key_s, t, ids, w, keff, sm_ids, sm_keff);
    else if (p.E <= 32 * 8) select_token_staged_pl<8>(p, sig_s, key_s, t, ids, w, keff, sm_ids, sm_keff);
    else select_token_staged_pl<16>(p, sig_s, key_s, t, ids, w, keff, sm_ids, sm_keff);
}

}  // namespace moe
