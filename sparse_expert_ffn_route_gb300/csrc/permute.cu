// permute.cu -- batch-union of the selected experts ["MoE 路由与专家流式加载" §1.3] by a
// stable counting sort ["Colibri 是什么" §3.3], and the tile plan of the grouped expert FFN.
//
// permute_kernel: one CTA of 1024 threads.
//   1. histogram of the kept (token, slot) pairs per expert (shared-memory atomics: counts
//      do not depend on their order);
//   2. exclusive scan -> offsets; unique experts in ascending id;
//   3. stable scatter: pairs are taken 1024 at a time in ascending pair index p = t*K + i;
//      a pair's place is offset[e] + pairs of e in earlier chunks + pairs of e in earlier
//      warps of this chunk + its rank among the lanes of its warp with the same expert
//      (__match_any_sync).  No atomic decides an order, so the lists are deterministic and
//      ascending in token.
// plan_kernel (and the tail of permute_kernel when asked): slot table and tile prefix sums
// of the FFN kernels.
#include "device_util.cuh"
#include "moe_internal.cuh"
#include "ffn_tiles.cuh"

namespace moe {

namespace {

struct PlanParams {
    int T, n_shared, include_routed;
    int rowbase_routed;   // output row of routed pair 0
    int tc_gu, tc_dn;
    Geo geo_gu[2], geo_dn[2];   // [0] routed, [1] shared
};

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int *total, int *s_warp)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = lane < nw ? s_warp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) s_warp[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == nw - 1) s_warp[32] = wi;
    }
    __syncthreads();
    const int res = s_warp[wid] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return res;
}

// Slot table + tile prefixes.  Reads offsets/uniq/n_uniq from global memory (written by
// this CTA or by an earlier kernel).  Must be called by every thread of a block of at least
// kMaxSlots threads... or any size: slots are strided.
__device__ void build_plan(const PlanParams &pp, const int32_t *offsets, const int32_t *uniq,
                           const int32_t *n_uniq, FfnPlan *plan, int *s_warp)
{
    const int ns = pp.n_shared;
    const int nu = pp.include_routed ? *n_uniq : 0;
    const int nslots = ns + nu;
    int base_gu = 0, base_dn = 0;
    for (int s0 = 0; s0 < nslots; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        int gu = 0, dn = 0;
        if (s < nslots) {
            int e, ntok, tokbase, rowbase, sh;
            if (s < ns) {
                e = -1; ntok = pp.T; tokbase = 0; rowbase = 0; sh = 1;
            } else {
                e = uniq[s - ns];
                tokbase = offsets[e];
                ntok = offsets[e + 1] - tokbase;
                rowbase = pp.rowbase_routed + tokbase;
                sh = 0;
            }
            plan->expert[s] = e;
            plan->ntok[s] = ntok;
            plan->tokbase[s] = tokbase;
            plan->rowbase[s] = rowbase;
            gu = tasks_of(pp.geo_gu[sh], ntok, pp.tc_gu);
            dn = tasks_of(pp.geo_dn[sh], ntok, pp.tc_dn);
        }
        int tot_gu, tot_dn;
        const int ex_gu = block_exclusive_scan(gu, &tot_gu, s_warp);
        const int ex_dn = block_exclusive_scan(dn, &tot_dn, s_warp);
        if (s < nslots) {
            plan->gu_prefix[s] = base_gu + ex_gu;
            plan->dn_prefix[s] = base_dn + ex_dn;
        }
        base_gu += tot_gu;
        base_dn += tot_dn;
    }
    if (threadIdx.x == 0) {
        plan->n_slots = nslots;
        plan->gu_prefix[nslots] = base_gu;
        plan->dn_prefix[nslots] = base_dn;
        plan->gu_tiles = base_gu;
        plan->dn_tiles = base_dn;
    }
}

__global__ void __launch_bounds__(1024) permute_kernel(
    const int32_t *__restrict__ ids, const int32_t *__restrict__ keff, int T, int K, int E,
    int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ tok,
    int32_t *__restrict__ slot, int32_t *__restrict__ uniq, int32_t *__restrict__ n_uniq,
    int32_t *__restrict__ err)
{
    __shared__ int s_cnt[kMaxExperts];
    __shared__ int s_off[kMaxExperts];
    __shared__ int s_base[kMaxExperts];
    __shared__ int s_tot[kMaxExperts];
    __shared__ unsigned short s_wt[32][kMaxExperts];
    __shared__ int s_warp[33];

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const long long P = (long long)T * K;

    for (int e = tid; e < E; e += blockDim.x) {
        s_cnt[e] = 0;
        s_base[e] = 0;
    }
    for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&s_wt[0][0])[i] = 0;
    __syncthreads();

    int bad = 0;
    for (long long p = tid; p < P; p += blockDim.x) {
        const int t = (int)(p / K), i = (int)(p - (long long)t * K);
        int k = keff[t];
        if (k < 0 || k > K) {
            if (i == 0) bad |= kErrBadKeff;
            k = max(0, min(K, k));
        }
        if (i < k) {
            const int e = ids[p];
            if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
            else bad |= kErrBadExpertId;
        }
    }
    if (bad) atomicOr(err, bad);
    __syncthreads();

    // exclusive scan of counts; unique experts
    {
        const int v = tid < E ? s_cnt[tid] : 0;
        int total, nu;
        const int ex = block_exclusive_scan(v, &total, s_warp);
        const int f = (tid < E && v > 0) ? 1 : 0;
        const int exf = block_exclusive_scan(f, &nu, s_warp);
        if (tid < E) {
            s_off[tid] = ex;
            offsets[tid] = ex;
            counts[tid] = v;
            if (f) uniq[exf] = tid;
        }
        if (tid == 0) {
            offsets[E] = total;
            *n_uniq = nu;
        }
    }
    __syncthreads();

    // stable scatter, 1024 pairs at a time
    for (long long c0 = 0; c0 < P; c0 += blockDim.x) {
        const long long p = c0 + tid;
        int e = -1, t = 0;
        if (p < P) {
            t = (int)(p / K);
            const int i = (int)(p - (long long)t * K);
            const int k = max(0, min(K, keff[t]));
            if (i < k) {
                const int id = ids[p];
                if (id >= 0 && id < E) e = id;
            }
        }
        const unsigned m = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(m & lanemask_lt());
        if (e >= 0 && rank == 0) s_wt[wid][e] = (unsigned short)__popc(m);
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) {
            int run = 0;
#pragma unroll 8
            for (int w = 0; w < 32; ++w) {
                const int v = s_wt[w][x];
                s_wt[w][x] = (unsigned short)run;
                run += v;
            }
            s_tot[x] = run;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = s_off[e] + s_base[e] + s_wt[wid][e] + rank;
            tok[pos] = t;
            slot[pos] = (int)p;
        }
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) {
            s_base[x] += s_tot[x];
#pragma unroll 8
            for (int w = 0; w < 32; ++w) s_wt[w][x] = 0;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams pp, const int32_t *offsets,
                                                    const int32_t *uniq, const int32_t *n_uniq,
                                                    FfnPlan *plan)
{
    __shared__ int s_warp[33];
    build_plan(pp, offsets, uniq, n_uniq, plan, s_warp);
}

}  // namespace

cudaError_t launch_permute(const moe_config &c, const int32_t *ids, const int32_t *keff, int T,
                           int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *slot,
                           int32_t *uniq, int32_t *n_uniq, int32_t *err, cudaStream_t st)
{
    permute_kernel<<<1, 1024, 0, st>>>(ids, keff, T, c.top_k, c.n_experts, counts, offsets, tok,
                                       slot, uniq, n_uniq, err);
    return cudaGetLastError();
}

cudaError_t launch_plan(const FfnArgs &a, const int32_t *uniq, const int32_t *n_uniq,
                        FfnPlan *plan, cudaStream_t st)
{
    PlanParams pp;
    pp.T = a.T;
    pp.n_shared = a.n_shared;
    pp.include_routed = a.include_routed;
    pp.rowbase_routed = a.routed_rowbase;
    pp.tc_gu = a.tc_gu;
    pp.tc_dn = a.tc_dn;
    for (int i = 0; i < 2; ++i) {
        pp.geo_gu[i] = a.geo_gu[i];
        pp.geo_dn[i] = a.geo_dn[i];
    }
    plan_kernel<<<1, 1024, 0, st>>>(pp, a.offsets, uniq, n_uniq, plan);
    return cudaGetLastError();
}

}  // namespace moe
