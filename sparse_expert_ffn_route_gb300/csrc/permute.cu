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
// plan_kernel: slot table and tile prefix sums of the FFN kernels.
// route_tail_kernel: decode-sized batches -- selection from the final router logits
// (router_select.cuh), the batch-union and the plan, all in one CTA of 1024 threads.
#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"
#include "router_select.cuh"

namespace moe {

namespace {

struct PlanParams {
    int T, n_shared, include_routed;
    int rowbase_routed;   // output row of routed pair 0
    int tc_gu, tc_dn;
    Geo geo_gu[2], geo_dn[2];   // [0] routed, [1] shared
};

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024).
template <typename V>
__device__ V block_exclusive_scan(V v, V *total, V *s_warp)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    V incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const V o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        V w = lane < nw ? s_warp[lane] : V(0);
        V wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const V o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < nw) s_warp[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == nw - 1) s_warp[32] = wi;
    }
    __syncthreads();
    const V res = s_warp[wid] + incl - v;
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
    __shared__ long long s_warp64[33];
    const int ns = pp.n_shared;
    const int nu = pp.include_routed ? *n_uniq : 0;
    const int nslots = ns + nu;
    int base_gu = 0, base_dn = 0;
    long long cbase_gu = 0, cbase_dn = 0;
    for (int s0 = 0; s0 < nslots; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        int gu = 0, dn = 0;
        long long cgu = 0, cdn = 0;
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
            cgu = slot_cost(pp.geo_gu[sh], ntok, pp.tc_gu);
            cdn = slot_cost(pp.geo_dn[sh], ntok, pp.tc_dn);
        }
        int tot_gu, tot_dn;
        const int ex_gu = block_exclusive_scan(gu, &tot_gu, s_warp);
        const int ex_dn = block_exclusive_scan(dn, &tot_dn, s_warp);
        long long ctot_gu, ctot_dn;
        const long long cex_gu = block_exclusive_scan(cgu, &ctot_gu, s_warp64);
        const long long cex_dn = block_exclusive_scan(cdn, &ctot_dn, s_warp64);
        if (s < nslots) {
            plan->gu_prefix[s] = base_gu + ex_gu;
            plan->dn_prefix[s] = base_dn + ex_dn;
            plan->gu_cost[s] = cbase_gu + cex_gu;
            plan->dn_cost[s] = cbase_dn + cex_dn;
        }
        base_gu += tot_gu;
        base_dn += tot_dn;
        cbase_gu += ctot_gu;
        cbase_dn += ctot_dn;
    }
    if (threadIdx.x == 0) {
        plan->n_slots = nslots;
        plan->gu_prefix[nslots] = base_gu;
        plan->dn_prefix[nslots] = base_dn;
        plan->gu_cost[nslots] = cbase_gu;
        plan->dn_cost[nslots] = cbase_dn;
        plan->gu_tiles = base_gu;
        plan->dn_tiles = base_dn;
        plan->next[0] = plan->next[1] = 0;
        plan->done[0] = plan->done[1] = 0;
    }
}

// Shared-memory working set of the batch-union (E <= kMaxExperts).
struct PermuteSmem {
    int *cnt, *off, *base, *tot;   // [kMaxExperts]; off has one more entry: the pair total
    unsigned short *wt;            // [32][kMaxExperts]
    int *uniq, *nu;                // unique experts [kMaxExperts], their count [1]
    int *warp;                     // [33] scan scratch
};

constexpr size_t kPermuteSmemBytes =
    sizeof(int) * (4 * kMaxExperts + 1) + sizeof(unsigned short) * 32 * kMaxExperts +
    sizeof(int) * (kMaxExperts + 1) + sizeof(int) * 33;

__device__ PermuteSmem carve_permute_smem(char *pool)
{
    PermuteSmem m;
    m.wt = reinterpret_cast<unsigned short *>(pool);
    int *p = reinterpret_cast<int *>(pool + sizeof(unsigned short) * 32 * kMaxExperts);
    m.cnt = p; p += kMaxExperts;
    m.off = p; p += kMaxExperts + 1;
    m.base = p; p += kMaxExperts;
    m.tot = p; p += kMaxExperts;
    m.uniq = p; p += kMaxExperts;
    m.nu = p; p += 1;
    m.warp = p;
    return m;
}

// The batch-union by the whole block (blockDim.x == 1024).  ids / keff may point to global
// or shared memory.  Besides the global outputs, sm.off[0..E] (offsets), sm.uniq and *sm.nu
// hold the lists' heads for the caller.
__device__ void permute_block(const int32_t *ids, const int32_t *keff, int T, int K, int E,
                              const PermuteOut &o, const PermuteSmem &sm)
{
    int32_t *__restrict__ counts = o.counts;
    int32_t *__restrict__ offsets = o.offsets;
    int32_t *__restrict__ tok = o.tok;
    int32_t *__restrict__ slot = o.slot;
    int32_t *__restrict__ uniq = o.uniq;
    int32_t *__restrict__ n_uniq = o.n_uniq;
    int32_t *__restrict__ err = o.err;
    int *s_cnt = sm.cnt, *s_off = sm.off, *s_base = sm.base, *s_tot = sm.tot;
    unsigned short(*s_wt)[kMaxExperts] = reinterpret_cast<unsigned short(*)[kMaxExperts]>(sm.wt);

    const int tid = threadIdx.x, wid = tid >> 5;
    const long long P = (long long)T * K;

    for (int e = tid; e < E; e += blockDim.x) {
        s_cnt[e] = 0;
        s_base[e] = 0;
    }
    for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) sm.wt[i] = 0;
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
        const int ex = block_exclusive_scan(v, &total, sm.warp);
        const int f = (tid < E && v > 0) ? 1 : 0;
        const int exf = block_exclusive_scan(f, &nu, sm.warp);
        if (tid < E) {
            s_off[tid] = ex;
            offsets[tid] = ex;
            counts[tid] = v;
            if (f) {
                uniq[exf] = tid;
                sm.uniq[exf] = tid;
            }
        }
        if (tid == 0) {
            s_off[E] = total;
            offsets[E] = total;
            *n_uniq = nu;
            *sm.nu = nu;
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
        if (o.pair_of && p < P) o.pair_of[p] = e >= 0 ? s_off[e] + s_base[e] + s_wt[wid][e] + rank : -1;
        __syncthreads();
        for (int x = tid; x < E; x += blockDim.x) {
            s_base[x] += s_tot[x];
#pragma unroll 8
            for (int w = 0; w < 32; ++w) s_wt[w][x] = 0;
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(1024) permute_kernel(const int32_t *__restrict__ ids,
                                                       const int32_t *__restrict__ keff, int T,
                                                       int K, int E, PermuteOut o)
{
    __shared__ __align__(16) char pool[kPermuteSmemBytes];
    pdl_wait();
    pdl_launch_dependents();
    permute_block(ids, keff, T, K, E, o, carve_permute_smem(pool));
}

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams pp, const int32_t *offsets,
                                                    const int32_t *uniq, const int32_t *n_uniq,
                                                    FfnPlan *plan)
{
    __shared__ int s_warp[33];
    pdl_wait();
    pdl_launch_dependents();
    build_plan(pp, offsets, uniq, n_uniq, plan, s_warp);
}

// Batch-union of at most 1024 pairs by a block of 1024 threads, from the routing in shared
// memory: histogram, one scan of (count, present) packed in an int, a scatter of the pairs
// into their experts' segments in any order, then each pair's final place from its rank
// among the segment's pair indices (pair index p = t*K + i, so ascending p is ascending
// token within an expert).  Fills sm.off[0..E], sm.uniq, *sm.nu besides the global outputs.
__device__ void permute_small_block(const int *s_ids, const int *s_keff, int T, int K, int E,
                                    const PermuteOut &o, const PermuteSmem &sm, int *s_stage,
                                    int *s_fill)
{
    const int tid = threadIdx.x;
    const int P = T * K;
    int e_mine = -1;
    if (o.pair_of && tid < P) o.pair_of[tid] = -1;
    if (tid < P) {
        const int t = tid / K, i = tid - t * K;
        const int k = s_keff[t];
        int bad = 0;
        if (k < 0 || k > K) bad |= (i == 0) ? kErrBadKeff : 0;
        if (i < max(0, min(K, k))) {
            const int e = s_ids[tid];
            if (e >= 0 && e < E) e_mine = e;
            else bad |= kErrBadExpertId;
        }
        if (bad) atomicOr(o.err, bad);
        if (e_mine >= 0) atomicAdd(&sm.cnt[e_mine], 1);
    }
    __syncthreads();
    {
        const int v = tid < E ? sm.cnt[tid] : 0;
        const int packed = v | ((v > 0 ? 1 : 0) << 16);   // counts <= 1024, experts <= 512
        int total;
        const int ex = block_exclusive_scan(packed, &total, sm.warp);
        if (tid < E) {
            const int off = ex & 0xffff;
            sm.off[tid] = off;
            o.offsets[tid] = off;
            o.counts[tid] = v;
            if (v > 0) {
                sm.uniq[ex >> 16] = tid;
                o.uniq[ex >> 16] = tid;
            }
            s_fill[tid] = 0;
        }
        if (tid == 0) {
            sm.off[E] = total & 0xffff;
            o.offsets[E] = total & 0xffff;
            *sm.nu = total >> 16;
            *o.n_uniq = total >> 16;
        }
    }
    __syncthreads();
    if (e_mine >= 0) s_stage[sm.off[e_mine] + atomicAdd(&s_fill[e_mine], 1)] = tid;
    __syncthreads();
    if (tid < sm.off[E]) {
        const int p = s_stage[tid];
        const int e = s_ids[p];
        const int lo = sm.off[e], hi = sm.off[e + 1];
        int rank = 0;
        for (int j = lo; j < hi; ++j) rank += s_stage[j] < p ? 1 : 0;
        o.tok[lo + rank] = p / K;
        o.slot[lo + rank] = p;
        if (o.pair_of) o.pair_of[p] = lo + rank;
    }
}

// Decode-sized batch (T <= kRouteClusterMaxT, so T * K <= 1024 pairs): one warp per token
// selects, then the block permutes and plans.  The routing and the lists' heads stay in
// shared memory between the phases; the global outputs are written alongside.
constexpr size_t kTailSmemBytes = kPermuteSmemBytes + sizeof(int) * (kRouteClusterMaxT * kMaxTopK) +
                                  sizeof(int) * kRouteClusterMaxT + sizeof(int) * (1024 + kMaxExperts);

__global__ void __launch_bounds__(1024) route_tail_kernel(const float *__restrict__ logits, int T,
                                                          SelectParams sp, int32_t *ids, float *w,
                                                          int32_t *keff, int do_permute,
                                                          PermuteOut o, int do_plan,
                                                          PlanParams pp, FfnPlan *plan)
{
    extern __shared__ __align__(16) char tail_pool[];
    const PermuteSmem sm = carve_permute_smem(tail_pool);
    int *s_ids = reinterpret_cast<int *>(tail_pool + kPermuteSmemBytes);
    int *s_keff = s_ids + kRouteClusterMaxT * kMaxTopK;
    int *s_stage = s_keff + kRouteClusterMaxT;
    int *s_fill = s_stage + 1024;
    pdl_wait();
    pdl_launch_dependents();
    const int wid = threadIdx.x >> 5;
    const int E = sp.E, K = sp.K;
    for (int e = threadIdx.x; e < E; e += blockDim.x) sm.cnt[e] = 0;
    for (int t = wid; t < T; t += 32) {
        const float *lrow = logits + (size_t)t * E;
        select_token(sp, [&](int e) { return lrow[e]; }, t, ids, w, keff, s_ids + t * K,
                     s_keff + t);
    }
    if (!do_permute) return;
    __syncthreads();
    permute_small_block(s_ids, s_keff, T, K, E, o, sm, s_stage, s_fill);
    if (!do_plan) return;
    __syncthreads();
    build_plan(pp, sm.off, sm.uniq, sm.nu, plan, sm.warp);
}

PlanParams plan_params(const FfnArgs &a)
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
    return pp;
}

}  // namespace

cudaError_t launch_permute(const moe_config &c, const int32_t *ids, const int32_t *keff, int T,
                           const PermuteOut &o, cudaStream_t st)
{
    return launch_kernel(permute_kernel, dim3(1), dim3(1024), 0, st, 1, ids, keff, T, c.top_k,
                         c.n_experts, o);
}

cudaError_t launch_plan(const FfnArgs &a, const int32_t *uniq, const int32_t *n_uniq,
                        FfnPlan *plan, cudaStream_t st)
{
    return launch_kernel(plan_kernel, dim3(1), dim3(1024), 0, st, 1, plan_params(a), a.offsets,
                         uniq, n_uniq, plan);
}

cudaError_t launch_route_tail(const moe_config &c, const float *logits, const float *bias, int T,
                              int32_t *ids, float *w, int32_t *keff, const PermuteOut *perm,
                              const FfnArgs *plan_args, cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    const PermuteOut o = perm ? *perm : PermuteOut{};
    const PlanParams pp = plan_args ? plan_params(*plan_args) : PlanParams{};
    FfnPlan *plan = plan_args ? const_cast<FfnPlan *>(plan_args->plan) : nullptr;
    return launch_kernel(route_tail_kernel, dim3(1), dim3(1024), kTailSmemBytes, st, 1, logits, T,
                         select_params(c, bias), ids, w, keff, perm ? 1 : 0, o,
                         (perm && plan_args) ? 1 : 0, pp, plan);
}

}  // namespace moe
