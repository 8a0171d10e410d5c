// ffn_kernels.cuh -- grouped int4 x int8 expert FFN for few tokens per expert (GEMV-shaped,
// HBM-bound) ["MoE 路由与专家流式加载" §1.3: gate/up/SiLU/down on the integer-dot path;
// "colibri 开发演进实录" §2.2 K1: unsigned nibbles, dot(u - 8, q) = dot(u, q) - 8 * sum(q);
// K1b: integer dot per 64-group, then the group scale].
//
// Work: tasks (slot, token chunk, block of rows) numbered by the planner, chunk-major within
// a slot.  The grid is persistent; every warp owns a contiguous range of tasks and walks it,
// so it keeps the int8 activations of its lanes' chunks in registers for as long as the
// (expert, token chunk) stays the same.  The packed nibbles stream from HBM with 16-byte
// read-only loads: a lane issues ru * nc loads per matrix before computing, which with 16
// warps per SM keeps enough bytes in flight to run at the HBM roof.
//
// In a row, lanes gl (of lpr) own the 16-byte chunks gl, gl+lpr, ... (32 codes each).  Per
// chunk and token:
//     A = -8 * sum(codes) + sum_{4 words} dp4a(w & 0x0F0F0F0F, even codes)
//                                       + dp4a((w >> 4) & 0x0F0F0F0F, odd codes)   (int32)
//     acc += scale[row][chunk/2] * A                                                (fp32)
// then acc is summed over the row's lanes with shuffles.  gate/up tasks carry both matrices
// and end with h = SiLU(sx*gate) * (sx*up); down tasks end with y = sh * acc.
#pragma once

#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace ffn_impl {

struct Task {
    int slot, sh, e, j0, nt, rowbase, r0, tokbase;
};

// walks a contiguous range of tasks without a search per task; everything it does not
// change is read from the kernel arguments (constant bank) when needed
template <bool GU>
struct Walker {
    int slot, local, slot_tasks, nblk;

    __device__ __forceinline__ const Geo &geo(const FfnArgs &a, int sh) const
    {
        return GU ? a.geo_gu[sh] : a.geo_dn[sh];
    }

    __device__ void enter(const FfnArgs &a, int s)
    {
        slot = s;
        const int sh = a.plan->expert[s] < 0 ? 1 : 0;
        const Geo &g = geo(a, sh);
        nblk = (g.nrows + g.rb - 1) / g.rb;
        slot_tasks = tasks_of(g, a.plan->ntok[s], GU ? a.tc_gu : a.tc_dn);
    }

    __device__ void start(const FfnArgs &a, int task)
    {
        const int32_t *prefix = GU ? a.plan->gu_prefix : a.plan->dn_prefix;
        int lo = 0, hi = a.plan->n_slots;   // prefix[lo] <= task < prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= task) lo = mid;
            else hi = mid;
        }
        enter(a, lo);
        local = task - prefix[lo];
    }

    __device__ void next(const FfnArgs &a)
    {
        if (++local >= slot_tasks) {
            int s = slot + 1;
            enter(a, s);
            while (slot_tasks == 0 && s + 1 < a.plan->n_slots) enter(a, ++s);
            local = 0;
        }
    }

    __device__ Task task(const FfnArgs &a) const
    {
        const FfnPlan *plan = a.plan;
        const int tc = GU ? a.tc_gu : a.tc_dn;
        Task t;
        t.slot = slot;
        t.e = plan->expert[slot];
        t.sh = t.e < 0 ? 1 : 0;
        const int ch = local / nblk, blk = local - ch * nblk;
        t.j0 = ch * tc;
        t.nt = min(tc, plan->ntok[slot] - t.j0);
        t.rowbase = plan->rowbase[slot] + t.j0;
        t.r0 = blk * geo(a, t.sh).rb;
        t.tokbase = plan->tokbase[slot];
        return t;
    }
};

// lanes per row: a launch whose lanes own two or more chunks gives every row the whole warp
// (the host configures both matrices so), which makes the chunk offsets compile-time
template <int NC>
__device__ __forceinline__ int lpr_of(const Geo &g)
{
    return NC >= 2 ? 32 : g.lpr;
}

template <int NC, int TC, int RU, int N, bool GU, bool PROBE>
__device__ __forceinline__ void run_task(const FfnArgs &a, const Task &t, const Geo &g,
                                         const uint32_t (&act)[TC][NC][8], const int (&csum)[TC][NC],
                                         const float (&ascale)[TC])
{
    constexpr int NM = GU ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const int lpr = lpr_of<NC>(g), rpw = 32 / lpr;
    const int sub = lane / lpr, gl = lane - sub * lpr;
    const int nch = g.kdim / 32;
    const bool shared = t.sh != 0;
    const moe_expert_weights &W = shared ? a.shared : a.routed;
    const size_t erow = shared ? 0 : (size_t)t.e * g.nrows;
    const uint8_t *wm[2] = {GU ? W.w_gate : W.w_down, W.w_up};
    const float *smat[2] = {GU ? W.s_gate : W.s_down, W.s_up};

    // issue every load of the task first
    uint4 w[RU][NM][NC];
    float sc[RU][NM][NC];
#pragma unroll
    for (int u = 0; u < RU; ++u) {
        const int r = t.r0 + u * rpw + sub;
        const bool rv = r < g.nrows;
        const size_t row = erow + (size_t)(rv ? r : 0);
#pragma unroll
        for (int m = 0; m < NM; ++m) {
            const uint8_t *wrow = wm[m] + row * g.rowbytes + (size_t)gl * 16;
            const float *srow = smat[m] + row * g.G;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int ci = gl + c * lpr;
                if (rv && ci < nch) {
                    w[u][m][c] = ld_stream_v4(wrow + c * lpr * 16);
                    sc[u][m][c] = ld_stream_f32(srow + (ci >> 1));
                } else {
                    w[u][m][c] = make_uint4(0u, 0u, 0u, 0u);
                    sc[u][m][c] = 0.0f;
                }
            }
        }
    }

#pragma unroll
    for (int u = 0; u < RU; ++u) {
        const int r = t.r0 + u * rpw + sub;
        const bool rv = r < g.nrows;
        float acc[NM][N];
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int j = 0; j < N; ++j) acc[m][j] = 0.0f;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int ci = gl + c * lpr;
                const uint32_t wv[4] = {w[u][m][c].x, w[u][m][c].y, w[u][m][c].z, w[u][m][c].w};
                int a0[N], a1[N];   // two independent chains per token
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    a0[j] = -8 * csum[j][c];
                    a1[j] = 0;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t lo = wv[q] & 0x0F0F0F0Fu;
                    const uint32_t hi = (wv[q] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        int &x = q < 2 ? a0[j] : a1[j];
                        x = dp4a_us(lo, act[j][c][2 * q], x);
                        x = dp4a_us(hi, act[j][c][2 * q + 1], x);
                    }
                }
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const int ai = a0[j] + a1[j];
                    acc[m][j] = fmaf(sc[u][m][c], (float)ai, acc[m][j]);
                    if (PROBE) {
                        // exact per-64-group accumulators: the two chunks of a group sit in
                        // lanes gl and gl ^ 1 (lpr is even)
                        const int other = __shfl_xor_sync(0xffffffffu, ai, 1);
                        if (rv && ci < nch && !shared && j < t.nt && (ci & 1) == 0) {
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
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int j = 0; j < N; ++j)
                for (int off = lpr >> 1; off > 0; off >>= 1)
                    acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], off);
        if (gl == 0 && rv) {
#pragma unroll
            for (int j = 0; j < N; ++j) {
                if (j >= t.nt) continue;
                const size_t orow = (size_t)(t.rowbase + j);
                if (GU) {
                    const float gate = ascale[j] * acc[0][j];
                    const float up = ascale[j] * acc[NM - 1][j];
                    a.h[orow * a.hstride + r] = gate / (1.0f + expf(-gate)) * up;
                } else {
                    a.y[orow * a.H + r] = ascale[j] * acc[0][j];
                }
            }
        }
    }
}

template <int NC, int TC, int RU, bool GU, int MINB, bool PROBE>
__global__ void __launch_bounds__(kFfnThreads, MINB) ffn_kernel(const __grid_constant__ FfnArgs a)
{
    const int lane = threadIdx.x & 31;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
    const int total = GU ? a.plan->gu_tiles : a.plan->dn_tiles;
    const int t_begin = (int)(gw * total / nw), t_end = (int)((gw + 1) * total / nw);
    if (t_begin >= t_end) return;
    const QuantRows &src = GU ? a.xq : a.hq;

    Walker<GU> walk;
    walk.start(a, t_begin);

    uint32_t act[TC][NC][8];
    int csum[TC][NC];
    float ascale[TC];
    int cur_slot = -1, cur_j0 = -1;

    for (int task = t_begin; task < t_end; ++task) {
        if (task > t_begin) walk.next(a);
        const Task t = walk.task(a);
        const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];

        // activations of this lane's chunks for the task's tokens (kept across tasks)
        if (t.slot != cur_slot || t.j0 != cur_j0) {
            cur_slot = t.slot;
            cur_j0 = t.j0;
            const int lpr = lpr_of<NC>(g);
            const int gl = lane % lpr, nch = g.kdim / 32;
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
                    const int ci = gl + c * lpr;
                    if (j < t.nt && ci < nch) {
                        const uint4 *p = reinterpret_cast<const uint4 *>(
                            src.q + (size_t)row * src.q_ld + (size_t)ci * 32);
                        const uint4 v0 = p[0], v1 = p[1];
                        act[j][c][0] = v0.x; act[j][c][1] = v0.y; act[j][c][2] = v0.z; act[j][c][3] = v0.w;
                        act[j][c][4] = v1.x; act[j][c][5] = v1.y; act[j][c][6] = v1.z; act[j][c][7] = v1.w;
                        csum[j][c] = src.csum[(size_t)row * src.c_ld + ci];
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) act[j][c][q] = 0;
                        csum[j][c] = 0;
                    }
                }
            }
        }

        // the chunk's real token count picks the variant, so padding costs little
        if (t.nt == 1 || TC == 1)
            run_task<NC, TC, RU, 1, GU, PROBE>(a, t, g, act, csum, ascale);
        else if (t.nt == 2 || TC == 2)
            run_task<NC, TC, RU, (TC >= 2 ? 2 : 1), GU, PROBE>(a, t, g, act, csum, ascale);
        else
            run_task<NC, TC, RU, TC, GU, PROBE>(a, t, g, act, csum, ascale);
    }
}

typedef void (*FfnKernel)(const FfnArgs);

// Each (kind, chunks, tokens) combination is built three ways: with two CTAs (16 warps) per
// SM, with one CTA and twice the rows in flight, and as the probe-writing twin of the latter.
// The host takes the 16-warp build unless the compiler had to spill it to local memory.
struct Variant {
    FfnKernel k2;       // 16 warps per SM
    int ru2;
    FfnKernel k1;       // 8 warps per SM
    int ru1;
    FfnKernel kprobe;   // the 8-warp build that also writes the test probes
};

// Rows in flight per task: about 12 (two CTAs) or 24 (one CTA) 16-byte loads per lane, so
// that roughly 100 KB of weight loads are outstanding per SM (the streaming rate of a GB300
// saturates near 50 KB per SM, measured); fewer once a token chunk's activations take more
// than 64 registers.
constexpr int ru_for(int nc, int tc, int nm, int ctas)
{
    int ru = 12 * (3 - ctas) / (nm * nc);
    ru = ru < 1 ? 1 : (ru > 8 ? 8 : ru);
    if (nc * 8 * tc > 64 && ru > 1) ru = ru / 2;
    return ru;
}

template <bool GU, int NC, int TC>
Variant variant_tc()
{
    constexpr int NM = GU ? 2 : 1;
    constexpr int R2 = ru_for(NC, TC, NM, 2), R1 = ru_for(NC, TC, NM, 1);
    return {ffn_kernel<NC, TC, R2, GU, 2, false>, R2, ffn_kernel<NC, TC, R1, GU, 1, false>, R1,
            ffn_kernel<NC, TC, R1, GU, 1, true>};
}

// largest tokens-per-chunk whose activations fit the registers
constexpr int tc_max(int nc) { return nc <= 2 ? 8 : (nc <= 4 ? 4 : 2); }

template <bool GU, int NC>
Variant variant_nc(int tc)
{
    switch (tc) {
    case 1: return variant_tc<GU, NC, 1>();
    case 2: return variant_tc<GU, NC, 2>();
    case 4: if constexpr (NC <= 4) return variant_tc<GU, NC, 4>(); else break;
    case 8: if constexpr (NC <= 2) return variant_tc<GU, NC, 8>(); else break;
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
