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
// (router_select.cuh), the batch-union and the plan, in one CTA (above 32 tokens the
// selection spreads over one CTA per 8 tokens of 1024 threads and the last one goes on
// alone); up to 256 pairs the batch-union ranks the pairs' keys with the whole block, which
// then has only the threads its phases need.
#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"
#include "router_select.cuh"

namespace moe {

namespace {

// What the plan needs of the FFN kernels' task geometry (tasks_of / slot_cost in
// ffn_tiles.cuh): the token chunk of a task, a power of two 2^lg, and the tasks per chunk
// of tokens, [0] routed, [1] shared; so the device forms them with shifts.
struct PlanParams {
    int T, n_shared, include_routed;
    int rowbase_routed;   // output row of routed pair 0
    int lg_gu, lg_dn;
    int per_chunk_gu[2], per_chunk_dn[2];
};

// The four running sums of the plan: gate/up and down tasks, and their costs.
struct PlanSums {
    int gu, dn;
    long long cgu, cdn;
};
__device__ __forceinline__ PlanSums operator+(const PlanSums &a, const PlanSums &b)
{
    return PlanSums{a.gu + b.gu, a.dn + b.dn, a.cgu + b.cgu, a.cdn + b.cdn};
}
__device__ __forceinline__ PlanSums operator-(const PlanSums &a, const PlanSums &b)
{
    return PlanSums{a.gu - b.gu, a.dn - b.dn, a.cgu - b.cgu, a.cdn - b.cdn};
}
__device__ __forceinline__ int shfl_up_v(int v, int off) { return __shfl_up_sync(0xffffffffu, v, off); }
__device__ __forceinline__ PlanSums shfl_up_v(const PlanSums &v, int off)
{
    return PlanSums{__shfl_up_sync(0xffffffffu, v.gu, off), __shfl_up_sync(0xffffffffu, v.dn, off),
                    __shfl_up_sync(0xffffffffu, v.cgu, off),
                    __shfl_up_sync(0xffffffffu, v.cdn, off)};
}

// Inclusive scan over the lanes of a warp.
template <typename V>
__device__ __forceinline__ V warp_inclusive_scan(V v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const V o = shfl_up_v(v, off);
        if (lane >= off) v = v + o;
    }
    return v;
}

// Block-wide exclusive scan of one value per thread (blockDim.x <= 1024).
template <typename V>
__device__ V block_exclusive_scan(V v, V *total, V *s_warp)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    const V incl = warp_inclusive_scan(v);
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const V w = lane < nw ? s_warp[lane] : V{};
        const V wi = warp_inclusive_scan(w);
        if (lane < nw) s_warp[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == nw - 1) s_warp[32] = wi;
    }
    __syncthreads();
    const V res = s_warp[wid] + incl - v;
    *total = s_warp[32];
    __syncthreads();
    return res;
}

// One slot of the plan: its expert (-1 for a shared one), tokens and list heads, written to
// the slot table; returns its task counts and costs.  Slots 0 .. ns-1 are the shared
// experts (every token), then the routed experts in ascending id.
// tasks_of and slot_cost for a chunk of 2^lg tokens and per_chunk tasks per chunk
__device__ __forceinline__ void chunk_tasks(int per_chunk, int lg, int ntok, int &tasks,
                                            long long &cost)
{
    tasks = 0;
    cost = 0;
    if (ntok <= 0) return;
    const int tc = 1 << lg;
    const int nch = (ntok + tc - 1) >> lg, nlast = ntok - ((nch - 1) << lg);
    const int wlast = min(nlast <= 1 ? 1 : 1 << (32 - __clz(nlast - 1)), tc) + 3;   // task_weight
    tasks = per_chunk * nch;
    cost = (long long)per_chunk * ((long long)(nch - 1) * (tc + 3) + wlast);
}

__device__ __forceinline__ PlanSums plan_slot(const PlanParams &pp, int s, int e, int tokbase,
                                              int ntok, FfnPlan *plan)
{
    const int sh = e < 0 ? 1 : 0;
    plan->expert[s] = e;
    plan->ntok[s] = ntok;
    plan->tokbase[s] = tokbase;
    plan->rowbase[s] = sh ? 0 : pp.rowbase_routed + tokbase;
    PlanSums v;
    chunk_tasks(pp.per_chunk_gu[sh], pp.lg_gu, ntok, v.gu, v.cgu);
    chunk_tasks(pp.per_chunk_dn[sh], pp.lg_dn, ntok, v.dn, v.cdn);
    return v;
}

__device__ __forceinline__ void plan_prefix(int s, const PlanSums &ex, FfnPlan *plan)
{
    plan->gu_prefix[s] = ex.gu;
    plan->dn_prefix[s] = ex.dn;
    plan->gu_cost[s] = ex.cgu;
    plan->dn_cost[s] = ex.cdn;
}

// The plan's header and the totals after its last slot; zeroes the task counters.
__device__ __forceinline__ void plan_header(int nslots, const PlanSums &tot, FfnPlan *plan)
{
    plan->n_slots = nslots;
    plan_prefix(nslots, tot, plan);
    plan->gu_tiles = tot.gu;
    plan->dn_tiles = tot.dn;
    plan->next[0] = plan->next[1] = 0;
    plan->done[0] = plan->done[1] = 0;
}

// Slot table + tile prefixes by a whole block.  Reads offsets/uniq/n_uniq from global or
// shared memory (written by this CTA or by an earlier kernel).  Slots are strided over the
// threads; one block scan forms the four prefixes.
__device__ void build_plan(const PlanParams &pp, const int32_t *offsets, const int32_t *uniq,
                           const int32_t *n_uniq, FfnPlan *plan)
{
    __shared__ PlanSums s_ps[33];
    const int ns = pp.n_shared;
    const int nu = pp.include_routed ? *n_uniq : 0;
    const int nslots = ns + nu;
    PlanSums base{};
    for (int s0 = 0; s0 < nslots; s0 += blockDim.x) {
        const int s = s0 + threadIdx.x;
        PlanSums v{};
        if (s < nslots) {
            if (s < ns) {
                v = plan_slot(pp, s, -1, 0, pp.T, plan);
            } else {
                const int e = uniq[s - ns];
                const int tokbase = offsets[e];
                v = plan_slot(pp, s, e, tokbase, offsets[e + 1] - tokbase, plan);
            }
        }
        PlanSums tot;
        const PlanSums ex = block_exclusive_scan(v, &tot, s_ps);
        if (s < nslots) plan_prefix(s, base + ex, plan);
        base = base + tot;
    }
    if (threadIdx.x == 0) plan_header(nslots, base, plan);
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
    pdl_wait();
    pdl_launch_dependents();
    build_plan(pp, offsets, uniq, n_uniq, plan);
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

// Batch-union and plan of a batch of at most 256 pairs by the whole block (at least E + 1,
// n_shared + E and T * K threads), in four block barriers and with short per-thread chains.  A kept pair's
// place is its rank among the kept pairs' keys (expert << 8 | pair index): the lists come
// out in ascending expert id and, within an expert, ascending pair index, i.e. ascending
// token -- the order permute_small_block gives.  Same outputs as permute_small_block
// followed by build_plan.  s_bits (kMaxExperts / 32 words) is zero on entry.
constexpr int kSmallRouteMaxPairs = 256;
constexpr int kPlanByCountMinT = 16;

struct SmallRouteSmem {
    int *key, *sorted;    // [kSmallRouteMaxPairs]
    unsigned *bits;       // [kMaxExperts / 32] experts present
    int *uq, *start, *len;   // [kMaxExperts] unique experts, their list heads and lengths
    PlanSums *ps;         // [32] warp totals of the plan scan
    int *c, *lo;          // [kMaxExperts] per expert: kept pairs, first list entry
};

__device__ void route_small_block(const int *s_ids, const int *s_keff, int T, int K, int E,
                                  const PermuteOut &o, int do_plan, const PlanParams &pp,
                                  FfnPlan *plan, const SmallRouteSmem &sm)
{
    constexpr int kNone = 0x7fffffff;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int P = T * K, P4 = (P + 3) & ~3;
    int *sm_c = sm.c, *sm_lo = sm.lo;   // per expert: kept pairs, first list entry
    const bool by_count = do_plan && T > kPlanByCountMinT;
    // keys of the kept pairs (padded to a multiple of 4 with kNone); experts present as bits
    int key = kNone;
    if (tid < P) {
        const int t = tid / K, i = tid - t * K;
        const int k = s_keff[t];
        int bad = 0;
        if (k < 0 || k > K) bad |= (i == 0) ? kErrBadKeff : 0;
        if (i < max(0, min(K, k))) {
            const int e = s_ids[tid];
            if (e >= 0 && e < E) {
                key = (e << 8) | tid;
                atomicOr(&sm.bits[e >> 5], 1u << (e & 31));
            } else {
                bad |= kErrBadExpertId;
            }
        }
        if (bad) atomicOr(o.err, bad);
        if (o.pair_of && key == kNone) o.pair_of[tid] = -1;
    }
    if (tid < P4) sm.key[tid] = key;
    __syncthreads();
    // a kept pair's place: its rank among the keys
    const bool valid = key != kNone;
    if (valid) {
        const int4 *k4 = reinterpret_cast<const int4 *>(sm.key);
        int rank = 0;
        for (int q = 0; q < P4 / 4; ++q) {
            const int4 v = k4[q];
            rank += (v.x < key ? 1 : 0) + (v.y < key ? 1 : 0) + (v.z < key ? 1 : 0) +
                    (v.w < key ? 1 : 0);
        }
        sm.sorted[rank] = key >> 8;
        o.tok[rank] = tid / K;
        o.slot[rank] = tid;
        if (o.pair_of) o.pair_of[tid] = rank;
    }
    const int nvalid = __syncthreads_count(valid);
    // expert x: offsets[x] (kept pairs of lower experts), counts[x]; a present expert's
    // place among the unique ones is the number of present experts below it
    if (tid <= E) {
        const int x = tid;
        int lo = 0, hi = nvalid;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sm.sorted[mid] < x) lo = mid + 1;
            else hi = mid;
        }
        o.offsets[x] = lo;
        if (x < E) {
            const unsigned word = sm.bits[x >> 5];
            int c = 0;
            if ((word >> (x & 31)) & 1u) {
                int up = lo, top = nvalid;
                while (up < top) {
                    const int mid = (up + top) >> 1;
                    if (sm.sorted[mid] <= x) up = mid + 1;
                    else top = mid;
                }
                c = up - lo;
                int u = __popc(word & ((1u << (x & 31)) - 1u));
                for (int wi = 0; wi < (x >> 5); ++wi) u += __popc(sm.bits[wi]);
                o.uniq[u] = x;
                sm_lo[x] = lo;
                if (!by_count) {
                    sm.uq[u] = x;
                    sm.start[u] = lo;
                    sm.len[u] = c;
                }
            }
            o.counts[x] = c;
            sm_c[x] = c;
        }
    }
    int nu = 0;
    for (int wi = 0; wi < (E + 31) >> 5; ++wi) nu += __popc(sm.bits[wi]);
    if (tid == 0) *o.n_uniq = nu;
    if (!do_plan) return;
    __syncthreads();
    // Above kPlanByCountMinT tokens the plan's routed slots go by descending token count
    // (ties by id): the FFN kernels hand out tasks in slot order, so the longest come first
    // and the shortest close the launch (GLM decode T = 32: gate/up and down each 2.4 µs
    // shorter; at 8 and 16 tokens the ranking costs more than it saves, and the slots stay
    // in ascending id).
    if (by_count && tid < E && ((sm.bits[tid >> 5] >> (tid & 31)) & 1u)) {
        const int x = tid, c = sm_c[x];
        int v = 0;
        for (int wi = 0; wi < (E + 31) >> 5; ++wi) {
            unsigned w = sm.bits[wi];
            while (w) {
                const int y = wi * 32 + __ffs(w) - 1;
                w &= w - 1;
                const int cy = sm_c[y];
                v += (cy > c || (cy == c && y < x)) ? 1 : 0;
            }
        }
        sm.uq[v] = x;
        sm.start[v] = sm_lo[x];
        sm.len[v] = c;
    }
    if (by_count) __syncthreads();
    // plan: slot s by thread s; warp scans, then the warps' totals
    const int ns = pp.n_shared;
    const int nslots = ns + (pp.include_routed ? nu : 0);
    PlanSums v{};
    if (tid < nslots) {
        if (tid < ns) v = plan_slot(pp, tid, -1, 0, pp.T, plan);
        else v = plan_slot(pp, tid, sm.uq[tid - ns], sm.start[tid - ns], sm.len[tid - ns], plan);
    }
    const int nw = (nslots + 31) >> 5;
    PlanSums incl{};
    if (wid < nw) {
        incl = warp_inclusive_scan(v);
        if (lane == 31) sm.ps[wid] = incl;
    }
    __syncthreads();
    if (tid < nslots) {
        PlanSums ex = incl - v;
        for (int w = 0; w < wid; ++w) ex = ex + sm.ps[w];
        plan_prefix(tid, ex, plan);
    }
    if (tid == 0) {
        PlanSums tot{};
        for (int w = 0; w < nw; ++w) tot = tot + sm.ps[w];
        plan_header(nslots, tot, plan);
    }
}

// Decode-sized batch (T <= kRouteClusterMaxT, so T * K <= 1024 pairs): one warp per token
// selects, then the block permutes and plans.  The routing and the lists' heads stay in
// shared memory between the phases; the global outputs are written alongside.
// the routing arrays start on a 16-byte boundary after the batch-union's working set (the
// small path reads keys as int4 and keeps 8-byte sums); every array below is a multiple of
// 16 bytes long, so each starts aligned
constexpr size_t kTailIdsOffset = (kPermuteSmemBytes + 15) & ~size_t(15);
constexpr size_t kTailSmemBytes = kTailIdsOffset + sizeof(int) * (kRouteClusterMaxT * kMaxTopK) +
                                  sizeof(int) * kRouteClusterMaxT + sizeof(int) * (1024 + kMaxExperts) +
                                  sizeof(float) * kMaxExperts;

// Batches of more than kTailOneCtaMaxT tokens select over several CTAs, kTailTokensPerCta
// tokens each (one warp per token: one SM's 32 warps selecting 64 tokens took 12 µs); the
// last CTA to finish, by a ticket in the workspace's first 256 bytes, reads every token's
// choice back and builds the batch-union and the plan.
constexpr int kTailOneCtaMaxT = 32;
constexpr int kTailTokensPerCta = 8;
constexpr int kTailTicketOffset = 24;   // ints into the workspace's first 256 bytes
// room for this many (token, expert) pairs, a key and a gate each, in the batch-union's
// scratch: one CTA scores up to one pair a thread there before the per-token rounds
constexpr int kTailStagedScores = 4096;
static_assert(kTailStagedScores * (sizeof(uint32_t) + sizeof(float)) <=
                  32 * kMaxExperts * sizeof(unsigned short),
              "staged scores fit the batch-union's per-warp count table");

__global__ void __launch_bounds__(1024) route_tail_kernel(const float *__restrict__ logits, int T,
                                                          SelectParams sp, int32_t *ids, float *w,
                                                          int32_t *keff, int do_permute,
                                                          PermuteOut o, int do_plan,
                                                          PlanParams pp, FfnPlan *plan)
{
    extern __shared__ __align__(16) char tail_pool[];
    const PermuteSmem sm = carve_permute_smem(tail_pool);
    int *s_ids = reinterpret_cast<int *>(tail_pool + kTailIdsOffset);
    int *s_keff = s_ids + kRouteClusterMaxT * kMaxTopK;
    int *s_stage = s_keff + kRouteClusterMaxT;
    int *s_fill = s_stage + 1024;
    float *s_bias = reinterpret_cast<float *>(s_fill + kMaxExperts);
    const int wid = threadIdx.x >> 5;
    const int E = sp.E, K = sp.K;
    static_assert((kRouteClusterMaxT * kMaxTopK * sizeof(int)) % 16 == 0 &&
                      (kRouteClusterMaxT * sizeof(int)) % 16 == 0 &&
                      (2 * kSmallRouteMaxPairs + kMaxExperts / 32) * sizeof(int) % 16 == 0 &&
                      (2 * kSmallRouteMaxPairs + kMaxExperts / 32) * sizeof(int) +
                              32 * sizeof(PlanSums) <= 1024 * sizeof(int),
                  "tail shared-memory layout");
    SmallRouteSmem srm;
    srm.key = s_stage;
    srm.sorted = s_stage + kSmallRouteMaxPairs;
    srm.bits = reinterpret_cast<unsigned *>(s_stage + 2 * kSmallRouteMaxPairs);
    srm.ps = reinterpret_cast<PlanSums *>(s_stage + 2 * kSmallRouteMaxPairs + kMaxExperts / 32);
    srm.uq = sm.uniq;
    srm.c = sm.cnt;
    srm.lo = sm.off;
    srm.start = sm.base;
    srm.len = sm.tot;
    // the selection bias is a layer parameter, not an output of the router kernel: it is
    // staged before the dependency wait
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_bias[e] = __ldcg(sp.bias + e);
    if (threadIdx.x < kMaxExperts / 32) srm.bits[threadIdx.x] = 0u;
    __syncthreads();
    sp.bias = s_bias;
    pdl_wait();
    pdl_launch_dependents();
    const int G = (int)gridDim.x;
    const int tb = G > 1 ? (int)blockIdx.x * kTailTokensPerCta : 0;
    const int te = G > 1 ? min(T, tb + kTailTokensPerCta) : T;
    const int nwarps = (int)(blockDim.x >> 5);
    if (G == 1 && T * E <= (int)blockDim.x) {
        // every (token, expert) gate and choice key by the whole block, one pair a thread, into
        // the batch-union's scratch (free until the batch-union below), then each token's
        // rounds by one warp: one warp scoring all of a token's experts ran the long unrolled
        // scoring code alone (GLM decode T = 1: 16.55k -> 16.72k tokens/s; with several pairs
        // a thread, at 8 tokens, it was 0.6% slower)
        uint32_t *s_key = reinterpret_cast<uint32_t *>(tail_pool);
        float *s_sig = reinterpret_cast<float *>(s_key + kTailStagedScores);
        for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
            const int e = i % E;
            score_expert(logits[i], s_bias[e], s_sig[i], s_key[i]);
        }
        __syncthreads();
        for (int t = wid; t < T; t += nwarps)
            select_token_staged(sp, s_sig + t * E, s_key + t * E, t, ids, w, keff, s_ids + t * K,
                                s_keff + t);
    } else {
        for (int t = tb + wid; t < te; t += nwarps) {
            const float *lrow = logits + (size_t)t * E;
            select_token(sp, [&](int e) { return lrow[e]; }, t, ids, w, keff, s_ids + t * K,
                         s_keff + t);
        }
    }
    if (!do_permute) return;
    if (G > 1) {
        __shared__ int s_last;
        __syncthreads();   // this CTA's choices are written
        if (threadIdx.x == 0) {
            __threadfence();
            int32_t *ticket = o.err + kTailTicketOffset;
            s_last = atomicAdd(ticket, 1) == G - 1;
            if (s_last) {
                *ticket = 0;   // back to zero for the next call
                __threadfence();
            }
        }
        __syncthreads();
        if (!s_last) return;
        // every token's choice (the other CTAs' through L2)
        for (int i = threadIdx.x; i < T * K; i += blockDim.x) s_ids[i] = __ldcg(ids + i);
        for (int i = threadIdx.x; i < T; i += blockDim.x) s_keff[i] = __ldcg(keff + i);
    }
    const bool small = T * K <= kSmallRouteMaxPairs && pp.n_shared + E <= (int)blockDim.x;
    if (!small)
        for (int e = threadIdx.x; e < E; e += blockDim.x) sm.cnt[e] = 0;
    __syncthreads();
    if (small) {
        route_small_block(s_ids, s_keff, T, K, E, o, do_plan, pp, plan, srm);
        return;
    }
    permute_small_block(s_ids, s_keff, T, K, E, o, sm, s_stage, s_fill);
    if (!do_plan) return;
    __syncthreads();
    // the plan's routed slots by descending token count (ties by id), as on the small path
    // above kPlanByCountMinT tokens (GLM decode T = 64: 90.9k -> 93.4k tokens/s; A3B T = 64
    // 699k -> 722k)
    const int nu = *sm.nu;
    int *order = sm.base;
    if ((int)threadIdx.x < nu) {
        const int x = sm.uniq[threadIdx.x], c = sm.off[x + 1] - sm.off[x];
        int v = 0;
        for (int u = 0; u < nu; ++u) {
            const int y = sm.uniq[u], cy = sm.off[y + 1] - sm.off[y];
            v += (cy > c || (cy == c && y < x)) ? 1 : 0;
        }
        order[v] = x;
    }
    __syncthreads();
    build_plan(pp, sm.off, order, sm.nu, plan);
}

// Threads of the route tail: 1024, except for one CTA whose pairs take the small path, which
// gets the threads its phases use (a warp per token, a thread per pair, per expert + 1 and
// per plan slot): every block-wide phase is run by all of the block's warps, so a GLM decode
// batch of one token (E = 256) takes 288 threads instead of 1024.
int tail_threads(const moe_config &c, int T, int grid, const PlanParams &pp)
{
    const int P = T * c.top_k, E = c.n_experts;
    if (grid != 1 || P > kSmallRouteMaxPairs) return 1024;
    int need = max(max(E + 1, pp.n_shared + E), max((P + 3) & ~3, 32 * T));
    need = (need + 31) & ~31;
    return need < 1024 ? need : 1024;
}

// log2 of a token chunk; every chunk the FFN paths configure is a power of two
int log2_pow2(int tc)
{
    int lg = 0;
    while ((1 << lg) < tc) ++lg;
    return lg;
}

PlanParams plan_params(const FfnArgs &a)
{
    PlanParams pp;
    pp.T = a.T;
    pp.n_shared = a.n_shared;
    pp.include_routed = a.include_routed;
    pp.rowbase_routed = a.routed_rowbase;
    pp.lg_gu = log2_pow2(a.tc_gu);
    pp.lg_dn = log2_pow2(a.tc_dn);
    for (int i = 0; i < 2; ++i) {
        const Geo &g = a.geo_gu[i], &d = a.geo_dn[i];
        pp.per_chunk_gu[i] = (g.nrows + g.rb - 1) / g.rb * g.S;
        pp.per_chunk_dn[i] = (d.nrows + d.rb - 1) / d.rb * d.S;
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
    const int grid = T > kTailOneCtaMaxT ? (T + kTailTokensPerCta - 1) / kTailTokensPerCta : 1;
    return launch_kernel(route_tail_kernel, dim3(grid), dim3(tail_threads(c, T, grid, pp)),
                         kTailSmemBytes, st, 1, logits, T,
                         select_params(c, bias), ids, w, keff, perm ? 1 : 0, o,
                         (perm && plan_args) ? 1 : 0, pp, plan);
}

}  // namespace moe
