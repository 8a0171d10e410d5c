// ffn_kernels.cuh -- the warp GEMV: grouped int4 x int8 expert FFN for few tokens per expert
// (GEMV-shaped, HBM-bound), run for batches under 3 tokens and for reductions that are not
// multiples of 256 (the row GEMV of ffn_rows.cu takes the rest below the tensor-core
// crossover) ["MoE 路由与专家流式加载" §1.3: gate/up/SiLU/down on the integer-dot path;
// "colibri 开发演进实录" §2.2 K1: unsigned nibbles, dot(u - 8, q) = dot(u, q) - 8 * sum(q);
// K1b: integer dot per 64-group, then the group scale].
//
// Work: tasks (slot, token chunk, input slice, block of rows) numbered by the planner, in
// that order of significance within a slot.  The grid is persistent (one CTA of 8 warps per
// SM); every warp owns a contiguous range of tasks of equal summed cost (task_weight: a
// task of a many-token chunk costs more than a one-token one) and walks it, keeping the int8
// activations of its lanes' chunks in registers for as long as the (expert, token chunk,
// slice) stays the same.
//
// Weight streaming: each lane copies the 16-byte nibble chunks it will multiply (and their
// group scales) with cp.async into its own slots of a per-warp ring of D stages in shared
// memory, D-1 tasks ahead of the one it computes.  A lane only ever reads back what it
// copied itself, so the ring needs no barrier: cp.async.wait_group orders it.  The bytes in
// flight (7/8 of the ring: ~100 KB per SM) are held by shared memory, not registers, which
// leaves the registers to the activations of up to 8 tokens.
//
// In a row, lanes gl (of lpr) own the 16-byte chunks gl, gl+lpr, ... (32 codes each) of the
// task's slice.  Per chunk and token:
//     A = -8 * sum(codes) + sum_{4 words} dp4a(w & 0x0F0F0F0F, even codes)
//                         + (sum_{4 words} dp4a(w & 0xF0F0F0F0, odd codes)) / 16    (int32)
//     acc += scale[row][chunk/2] * A                                                (fp32)
// (the high nibbles stay in place, so their products come out 16x and the division by 16
// is exact).
// then acc is summed over the row's lanes: with a whole warp per row, all V accumulators of
// the task (rows x matrices x tokens) at once by a reduce-scatter (V-1 shuffles in all, lane
// l ends with one total); with fewer lanes per row, each by a shuffle tree.  gate/up tasks
// carry both matrices and end with h = SiLU(sx*gate) * (sx*up); down tasks end with
// y = sh * acc.  When the rows are sliced (decode-route batches of 3 tokens or more), a task
// ends with its slice's partial sums instead: sx*gate and sx*up into per-slice planes that
// the h quantisation adds up in slice order, and sh*acc into the slice's plane of y that the
// combine adds up in slice order.
#pragma once

#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace ffn_impl {

struct Task {
    int slot, sh, e, j0, nt, rowbase, r0, tokbase, s;   // s: slice of the rows' inputs
};

// Walks a contiguous range of tasks: one binary search over the slots' task prefixes at the
// start, then a mixed-radix count (row block, slice, token chunk, slot) with no division.
template <bool GU>
struct Walker {
    Task t;                    // the current task
    int blk, nblk, rb, S, ntok, tc;

    __device__ __forceinline__ void enter(const FfnArgs &a, int s)
    {
        const FfnPlan *plan = a.plan;
        t.slot = s;
        t.e = plan->expert[s];
        t.sh = t.e < 0 ? 1 : 0;
        const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
        rb = g.rb;
        nblk = (g.nrows + g.rb - 1) / g.rb;
        S = g.S;
        ntok = plan->ntok[s];
        t.tokbase = plan->tokbase[s];
        t.rowbase = plan->rowbase[s];
        t.j0 = 0;
        t.s = 0;
        t.r0 = 0;
        blk = 0;
        t.nt = min(tc, ntok);
    }

    __device__ void start(const FfnArgs &a, int task)
    {
        tc = GU ? a.tc_gu : a.tc_dn;
        const int32_t *prefix = GU ? a.plan->gu_prefix : a.plan->dn_prefix;
        int lo = 0, hi = a.plan->n_slots;   // prefix[lo] <= task < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= task) lo = mid;
            else hi = mid;
        }
        enter(a, lo);
        locate(task - prefix[lo]);
    }

    // Task `task` of the shared expert, slot 0, without the plan: every token, list head 0,
    // output rows from 0.  Walking stays inside the slot (next() is only called while
    // another task of the range follows).
    __device__ void start_shared(const FfnArgs &a, int task)
    {
        tc = GU ? a.tc_gu : a.tc_dn;
        t.slot = 0;
        t.e = -1;
        t.sh = 1;
        const Geo &g = GU ? a.geo_gu[1] : a.geo_dn[1];
        rb = g.rb;
        nblk = (g.nrows + g.rb - 1) / g.rb;
        S = g.S;
        ntok = a.T;
        t.tokbase = 0;
        t.rowbase = 0;
        locate(task);
    }

    // the slot's local task index = (chunk * S + slice) * nblk + block
    __device__ __forceinline__ void locate(int local)
    {
        const int cs = local / nblk;
        blk = local - cs * nblk;
        const int ch = cs / S;
        t.s = cs - ch * S;
        t.j0 = ch * tc;
        t.rowbase += t.j0;
        t.r0 = blk * rb;
        t.nt = min(tc, ntok - t.j0);
    }

    // only called while another task of the range follows
    __device__ __forceinline__ void next(const FfnArgs &a)
    {
        t.r0 += rb;
        if (++blk < nblk) return;
        blk = 0;
        t.r0 = 0;
        if (++t.s < S) return;
        t.s = 0;
        t.j0 += tc;
        t.rowbase += tc;
        if (t.j0 < ntok) {
            t.nt = min(tc, ntok - t.j0);
            return;
        }
        int s = t.slot + 1;
        enter(a, s);
        while (ntok == 0 && s + 1 < a.plan->n_slots) enter(a, ++s);
    }
};

// lanes per row: a launch whose lanes own two or more chunks gives every row the whole warp
// (the host configures both matrices so), which makes the chunk offsets compile-time
template <int NC>
__device__ __forceinline__ int lpr_of(const Geo &g)
{
    return NC >= 2 ? 32 : g.lpr;
}


// one lane's ring slots: [stage][u][m][c] x 32 lanes
template <int NC, int RU, int NM>
__device__ __forceinline__ int slot_of(int st, int u, int m, int c, int lane)
{
    return (((st * RU + u) * NM + m) * NC + c) * 32 + lane;
}

// Issue the copies of one task into ring stage `st` (zero-fill outside the rows / slice).
template <int NC, int RU, bool GU>
__device__ __forceinline__ void issue_task(const FfnArgs &a, const Task &t, int st, uint4 *wbuf,
                                           float *sbuf, uint64_t pol)
{
    constexpr int NM = GU ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
    const int lpr = lpr_of<NC>(g), rpw = 32 / lpr;
    const int sub = lane / lpr, gl = lane - sub * lpr;
    const int cb = t.s * g.sch;
    const int sn = min(g.sch, g.kdim / 32 - cb);
    const moe_expert_weights &W = t.sh ? a.shared : a.routed;
    const size_t erow = t.sh ? 0 : (size_t)t.e * g.nrows;
    const uint8_t *wm[2] = {GU ? W.w_gate : W.w_down, W.w_up};
    const float *smat[2] = {GU ? W.s_gate : W.s_down, W.s_up};
#pragma unroll
    for (int u = 0; u < RU; ++u) {
        const int r = t.r0 + u * rpw + sub;
        const bool rv = r < g.nrows;
        const size_t row = erow + (size_t)(rv ? r : 0);
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int li = gl + c * lpr;
                const bool ok = rv && li < sn;
                const int ci = cb + (ok ? li : 0);
                const int k = slot_of<NC, RU, NM>(st, u, m, c, lane);
                cp_async16_hint(wbuf + k, wm[m] + row * g.rowbytes + (size_t)ci * 16, ok, pol);
                cp_async4_hint(sbuf + k, smat[m] + row * g.G + (ci >> 1), ok, pol);
            }
        }
    }
}

template <int NC, int TC, int RU, int N, bool GU, bool PROBE>
__device__ __forceinline__ void run_task(const FfnArgs &a, const Task &t, const Geo &g, int st,
                                         const uint4 *wbuf, const float *sbuf,
                                         const uint32_t (&act)[TC][NC][8], const int (&csum8)[TC][NC],
                                         const float (&ascale)[TC])
{
    constexpr int NM = GU ? 2 : 1;
    constexpr int V = RU * N * NM;        // accumulators of the task
    const int lane = threadIdx.x & 31;
    const int lpr = lpr_of<NC>(g), rpw = 32 / lpr;
    const int sub = lane / lpr, gl = lane - sub * lpr;
    const int cb = t.s * g.sch;
    const int sn = min(g.sch, g.kdim / 32 - cb);

    // acc[o] with o = (u * N + j) * NM + m
    float acc[V];
#pragma unroll
    for (int o = 0; o < V; ++o) acc[o] = 0.0f;
#pragma unroll
    for (int u = 0; u < RU; ++u) {
        const int r = t.r0 + u * rpw + sub;
        const bool rv = r < g.nrows;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int li = gl + c * lpr, ci = cb + li;
                const int k = slot_of<NC, RU, NM>(st, u, m, c, lane);
                const uint4 wq = wbuf[k];
                const float sc = sbuf[k];
                const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
                // low nibbles against the even codes, high nibbles (kept in place, i.e. 16x)
                // against the odd codes: two chains per token, the first starting from the
                // zero-point correction -8 * sum(codes)
                int clo[N], chi[N];
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    clo[j] = csum8[j][c];
                    chi[j] = 0;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t lo = wv[q] & 0x0F0F0F0Fu;
                    const uint32_t hi16 = wv[q] & 0xF0F0F0F0u;
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        clo[j] = dp4a_us(lo, act[j][c][2 * q], clo[j]);
                        chi[j] = dp4a_us(hi16, act[j][c][2 * q + 1], chi[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const int ai = clo[j] + (chi[j] >> 4);   // exact: chi is 16 x an integer
                    float &x = acc[(u * N + j) * NM + m];
                    x = fmaf(sc, (float)ai, x);
                    if (PROBE) {
                        // exact per-64-group accumulators: the two chunks of a group sit in
                        // lanes gl and gl ^ 1 (lpr is even)
                        const int other = __shfl_xor_sync(0xffffffffu, ai, 1);
                        if (rv && li < sn && t.sh == 0 && j < t.nt && (ci & 1) == 0) {
                            const size_t pr = (size_t)(t.rowbase + j - a.routed_rowbase);
                            const size_t o = (pr * g.nrows + r) * g.G + (ci >> 1);
                            int32_t *dst = GU ? (m == 0 ? a.probe.acc_gate : a.probe.acc_up)
                                              : a.probe.acc_down;
                            if (dst) dst[o] = ai + other;
                        }
                    }
                }
            }
        }
    }

    // output o of the task: row t.r0 + u*rpw + sub, token j, matrix m
    auto emit = [&](int o, float v, float partner) {
        const int m = o % NM, j = (o / NM) % N, u = o / (NM * N);
        const int r = t.r0 + u * rpw + sub;
        if (r >= g.nrows || j >= t.nt) return;
        float sx = 0.0f;
#pragma unroll
        for (int jj = 0; jj < N; ++jj)
            if (jj == j) sx = ascale[jj];
        const size_t orow = (size_t)(t.rowbase + j);
        const size_t prow = (size_t)t.s * a.plane_rows + orow;   // row of the slice's plane
        if (GU) {
            if (g.S == 1) {
                if (m == 0) {
                    const float gate = sx * v, up = sx * partner;
                    a.h[orow * a.hstride + r] = gate / (1.0f + expf(-gate)) * up;
                }
            } else {
                (m == 0 ? a.gpart : a.upart)[prow * a.hstride + r] = sx * v;
            }
        } else {
            a.y[prow * a.H + r] = sx * v;
        }
    };

    if (lpr == 32) {
        // one row per u: reduce-scatter all V accumulators, 32 at a time
        constexpr int G32 = V < 32 ? V : 32;
        constexpr int SH = 5 - ilog2(G32);   // lanes sharing one total: 1 << SH
#pragma unroll
        for (int base = 0; base < V; base += G32) {
            ReduceScatter<G32, 16>::run(acc + base, lane);
            const float v = acc[base];
            // gate and up of one (row, token) are neighbours (m is the lowest digit of o)
            const float partner = __shfl_xor_sync(0xffffffffu, v, 1 << SH);
            if ((lane & ((1 << SH) - 1)) == 0) emit(base + (lane >> SH), v, partner);
        }
    } else {
#pragma unroll
        for (int o = 0; o < V; ++o)
            for (int off = lpr >> 1; off > 0; off >>= 1)
                acc[o] += __shfl_xor_sync(0xffffffffu, acc[o], off);
        if (gl == 0) {
#pragma unroll
            for (int o = 0; o < V; o += NM) emit(o, acc[o], acc[o + NM - 1]);
            if (!GU || g.S > 1) {
#pragma unroll
                for (int o = 1; o < V; o += NM)
                    if (NM > 1) emit(o, acc[o], 0.0f);
            }
        }
    }
}

// global index of the task whose cost interval holds cost c (0 <= c < total cost)
template <bool GU>
__device__ int task_at(const FfnArgs &a, long long c)
{
    const FfnPlan *plan = a.plan;
    const int64_t *cost = GU ? plan->gu_cost : plan->dn_cost;
    int lo = 0, hi = plan->n_slots;   // the last slot starting at or before c
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cost[mid] <= c) lo = mid;
        else hi = mid;
    }
    const int sh = plan->expert[lo] < 0 ? 1 : 0;
    const Geo &g = GU ? a.geo_gu[sh] : a.geo_dn[sh];
    return (GU ? plan->gu_prefix : plan->dn_prefix)[lo] +
           task_at_cost(g, plan->ntok[lo], GU ? a.tc_gu : a.tc_dn, c - cost[lo]);
}

template <int NC, int RU, bool GU>
constexpr int ring_slots() { return RU * (GU ? 2 : 1) * NC; }

// stages of the ring: as many as fit about 224 KB of shared memory for the CTA's 8 warps
// (at most 8, at least 2)
template <int NC, int RU, bool GU>
constexpr int ring_depth()
{
    constexpr int per_stage = kFfnWarpsPerCta * ring_slots<NC, RU, GU>() * 32 * 20;
    constexpr int d = 224 * 1024 / per_stage;
    return d < 2 ? 2 : (d > 8 ? 8 : d);
}

template <int NC, int RU, bool GU>
constexpr size_t ring_bytes()
{
    return (size_t)kFfnWarpsPerCta * ring_depth<NC, RU, GU>() * ring_slots<NC, RU, GU>() * 32 *
           (sizeof(uint4) + sizeof(float));
}

template <int NC, int TC, int RU, bool GU, bool PROBE>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(const __grid_constant__ FfnArgs a)
{
    constexpr int D = ring_depth<NC, RU, GU>();
    constexpr int SL = ring_slots<NC, RU, GU>();
    extern __shared__ uint4 ffn_ring[];
    const bool early = GU && a.shared_early && a.n_shared;
    // Down: the plan and the weights are older than the h codes (the planner ran at least
    // three launches back, the h quantisation is the launch just before), so each warp sends
    // its first D-1 tasks' weight copies before the dependency wait and only its reads of the
    // codes wait.
    const bool early_w = !GU;
    if (!early && !early_w) pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    uint4 *wbuf = ffn_ring + (size_t)wid * D * SL * 32;
    float *sbuf = reinterpret_cast<float *>(ffn_ring + (size_t)kFfnWarpsPerCta * D * SL * 32) +
                  (size_t)wid * D * SL * 32;

    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    const QuantRows &src = GU ? a.xq : a.hq;
    // a slot's last token chunk (its chunks come in order) reads the weights for the last
    // time in this launch: evict-first in L2
    const uint64_t pol_last = l2_policy_evict_first(), pol_again = l2_policy_evict_normal();
    uint32_t act[TC][NC][8];
    int csum8[TC][NC];   // -8 x the chunk's code sum
    float ascale[TC];

    // Runs tasks [t_begin, t_end) through this warp's ring; `shared`: the range lies in the
    // shared expert's slot and is walked without the plan; `wait`: the dependency wait comes
    // after the first copies.
    auto run = [&](int t_begin, int t_end, bool shared, bool wait) {
        Walker<GU> cw;   // the task being computed
        if (shared) cw.start_shared(a, t_begin);
        else cw.start(a, t_begin);
        Walker<GU> iw = cw;   // the next task to copy in
        int issued = t_begin;
        auto issue_next = [&](int st) {
            if (issued < t_end) {
                issue_task<NC, RU, GU>(a, iw.t, st, wbuf, sbuf,
                                       iw.ntok <= iw.t.j0 + iw.tc ? pol_last : pol_again);
                if (++issued < t_end) iw.next(a);
            }
            cp_async_commit();   // possibly empty: keeps one group per task
        };
#pragma unroll
        for (int k = 0; k < D - 1; ++k) issue_next(k);
        if (wait) pdl_wait();

        int cur_slot = -1, cur_j0 = -1, cur_s = -1;
        for (int task = t_begin, it = 0; task < t_end; ++task, ++it) {
            issue_next((it + D - 1) % D);
            cp_async_wait<D - 1>();   // this task's copies (group `it`) have landed
            if (task > t_begin) cw.next(a);
            const Task &t = cw.t;
            const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
            // activations of this lane's chunks for the task's tokens (kept across tasks)
            if (t.slot != cur_slot || t.j0 != cur_j0 || t.s != cur_s) {
                cur_slot = t.slot;
                cur_j0 = t.j0;
                cur_s = t.s;
                const int lpr = lpr_of<NC>(g);
                const int gl = lane % lpr, cb = t.s * g.sch, sn = min(g.sch, g.kdim / 32 - cb);
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    int row = 0;
                    ascale[j] = 0.0f;
                    if (j < t.nt) {
                        if (GU) row = t.sh ? t.j0 + j : a.tok[t.tokbase + t.j0 + j];
                        else row = t.rowbase + j;
                        ascale[j] = src.scale[row];
                    }
#pragma unroll
                    for (int c = 0; c < NC; ++c) {
                        const int li = gl + c * lpr, ci = cb + li;
                        if (j < t.nt && li < sn) {
                            const uint4 *p = reinterpret_cast<const uint4 *>(
                                src.q + (size_t)row * src.q_ld + (size_t)ci * 32);
                            const uint4 v0 = p[0], v1 = p[1];
                            act[j][c][0] = v0.x; act[j][c][1] = v0.y; act[j][c][2] = v0.z; act[j][c][3] = v0.w;
                            act[j][c][4] = v1.x; act[j][c][5] = v1.y; act[j][c][6] = v1.z; act[j][c][7] = v1.w;
                            csum8[j][c] = -8 * src.csum[(size_t)row * src.c_ld + ci];
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q) act[j][c][q] = 0;
                            csum8[j][c] = 0;
                        }
                    }
                }
            }

            // the chunk's real token count picks the variant, so padding costs little
            const int st = it % D;
            if (t.nt == 1 || TC == 1)
                run_task<NC, TC, RU, 1, GU, PROBE>(a, t, g, st, wbuf, sbuf, act, csum8, ascale);
            else if (t.nt == 2 || TC == 2)
                run_task<NC, TC, RU, (TC >= 2 ? 2 : 1), GU, PROBE>(a, t, g, st, wbuf, sbuf, act, csum8, ascale);
            else if (t.nt <= 4 || TC == 4)
                run_task<NC, TC, RU, (TC >= 4 ? 4 : 1), GU, PROBE>(a, t, g, st, wbuf, sbuf, act, csum8, ascale);
            else
                run_task<NC, TC, RU, TC, GU, PROBE>(a, t, g, st, wbuf, sbuf, act, csum8, ascale);
        }
        cp_async_wait<0>();
    };

    // Early mode (gate/up of a call whose x codes were written at least two launches back):
    // the shared expert's tasks, a contiguous share per warp, run before the dependency wait.
    long long c0 = 0;   // the routed tasks' share of the cost starts here
    if (early) {
        const int n_sh = tasks_of(a.geo_gu[1], a.T, a.tc_gu);
        const int s_begin = (int)(n_sh * gw / nw), s_end = (int)(n_sh * (gw + 1) / nw);
        if (s_begin < s_end) run(s_begin, s_end, true, false);
        pdl_wait();
        c0 = (GU ? a.plan->gu_cost : a.plan->dn_cost)[1];
    }
    const int n_slots = a.plan->n_slots;
    const long long C = (GU ? a.plan->gu_cost : a.plan->dn_cost)[n_slots];
    // every warp passes the dependency wait once, so that the launch never ends before the
    // work it depends on
    if (C <= c0) {
        if (early_w) pdl_wait();
        return;
    }
    const int t_begin = task_at<GU>(a, c0 + (C - c0) * gw / nw);
    const int t_end = gw + 1 == nw ? (GU ? a.plan->gu_tiles : a.plan->dn_tiles)
                                   : task_at<GU>(a, c0 + (C - c0) * (gw + 1) / nw);
    if (t_begin < t_end) run(t_begin, t_end, false, early_w);
    else if (early_w) pdl_wait();
}

typedef void (*FfnKernel)(const FfnArgs);

// Each (kind, chunks, tokens) combination: the production kernel and its probe-writing twin
// (the same arithmetic, plus stores of the exact per-group accumulators), the rows per task
// and the dynamic shared memory of the ring.
struct Variant {
    FfnKernel k;
    FfnKernel kprobe;
    int ru;
    size_t smem;
};

// Rows per task: about 8 ring slots (16-byte loads) per lane and task, a power of two.
constexpr int ru_for(int nc, int nm)
{
    const int want = 8 / (nm * nc);
    return want >= 8 ? 8 : (want >= 4 ? 4 : (want >= 2 ? 2 : 1));
}

template <bool GU, int NC, int TC>
Variant variant_tc()
{
    constexpr int RU = ru_for(NC, GU ? 2 : 1);
    return {ffn_kernel<NC, TC, RU, GU, false>, ffn_kernel<NC, TC, RU, GU, true>, RU,
            ring_bytes<NC, RU, GU>()};
}

// largest tokens-per-chunk whose activations (8 * tc * nc registers) leave room for the rest
// within the 170 registers a thread of a 12-warp CTA has
constexpr int tc_max(int nc) { return nc <= 1 ? 4 : (nc <= 2 ? 2 : 1); }

template <bool GU, int NC>
Variant variant_nc(int tc)
{
    switch (tc) {
    case 1: return variant_tc<GU, NC, 1>();
    case 2: if constexpr (tc_max(NC) >= 2) return variant_tc<GU, NC, 2>(); else break;
    case 4: if constexpr (tc_max(NC) >= 4) return variant_tc<GU, NC, 4>(); else break;
    }
    return {};
}

}  // namespace ffn_impl

// one translation unit per (kind, chunks-per-lane pair), compiled in parallel; each returns
// the variant for chunk count nc (one of its pair) and tokens per chunk tc
ffn_impl::Variant ffn_variant_gu_12(int nc, int tc);
ffn_impl::Variant ffn_variant_gu_34(int nc, int tc);
ffn_impl::Variant ffn_variant_gu_56(int nc, int tc);
ffn_impl::Variant ffn_variant_gu_78(int nc, int tc);
ffn_impl::Variant ffn_variant_dn_12(int nc, int tc);
ffn_impl::Variant ffn_variant_dn_34(int nc, int tc);
ffn_impl::Variant ffn_variant_dn_56(int nc, int tc);
ffn_impl::Variant ffn_variant_dn_78(int nc, int tc);

}  // namespace moe
