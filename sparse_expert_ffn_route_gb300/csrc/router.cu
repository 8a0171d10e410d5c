// router.cu -- router of the MoE layer: logits, sigmoid scoring, noaux_tc selection bias,
// iterated-argmax top-k, adaptive top-p, norm_topk_prob, routed_scaling_factor
// ["MoE 路由与专家流式加载" §1.1, §1.2].
//
// Decode-sized batches (T <= kRouteClusterMaxT):
//   router_cluster_kernel  up to 8 tokens: one cluster of CS CTAs per 16 experts; CTA rank r
//                          holds the r-th slice of H, each warp two experts x all tokens, so
//                          a lane keeps its experts' router weights in registers and streams
//                          x from shared memory.
//   router_tokens_kernel   more tokens: one cluster per 8 experts, tokens on the lanes (below).
//                          Both sum the CS partial logits in rank order through distributed
//                          shared memory and quantise x to int8 (the layer's activation
//                          quantisation): cluster c takes tokens t = c (mod clusters), the
//                          ranks' partial |x| maxima meet the same way.
//   route_tail_kernel      (permute.cu) selection, batch-union and FFN plan: one CTA up to
//                          32 tokens; beyond, the selection over one CTA per 8 tokens and the
//                          rest in the last of them.
// Larger batches:
//   router_logits_kernel   fp32 x . W_router^T, tiled 128 tokens x 64 experts, split along
//                          H so that the grid covers the GPU; partial sums to [S][T][E].
//   router_select_kernel   one warp per token: sums the S partials in a fixed order, then
//                          selects (router_select.cuh).
#include <float.h>

#include <cooperative_groups.h>

#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"
#include "router_select.cuh"

namespace moe {

namespace {

constexpr int kBT = 128;  // tokens per tile
constexpr int kBE = 64;   // experts per tile
constexpr int kBK = 16;   // floats of H per stage
constexpr int kTargetCtas = 2 * 152;

// fp32 x . W_router^T on one 128-token x 64-expert tile over the H range of split s.  Each
// thread sums 8 x 4 outputs: tokens {4ty .. 4ty+3, 64+4ty .. 64+4ty+3} x experts 4tx ..
// 4tx+3, so a warp's shared-memory reads are 16-byte lanes at a 16-byte stride.  The next
// stage's x and W are loaded into registers while the current one is multiplied, then
// stored into the other shared-memory buffer.  Two CTAs fit an SM.
__global__ void __launch_bounds__(256, 2) router_logits_kernel(const float *__restrict__ x,
                                                               const float *__restrict__ wr, int T,
                                                               int H, int E, int S,
                                                               float *__restrict__ part)
{
    __shared__ __align__(16) float xs[2][kBK][kBT + 4];
    __shared__ __align__(16) float ws[2][kBK][kBE + 4];
    pdl_wait();
    pdl_launch_dependents();
    const int t0 = blockIdx.x * kBT, e0 = blockIdx.y * kBE, s = blockIdx.z;
    const int nch = H / kBK;
    const int c0 = (int)((long long)s * nch / S), c1 = (int)((long long)(s + 1) * nch / S);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    // stage loads: 128 rows x 16 floats of x (two float4 per thread), 64 rows of W (one)
    float4 xv[2], wv;
    auto load = [&](int c) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + 256 * i, r = idx >> 2, c4 = idx & 3;
            const int t = t0 + r;
            xv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T) xv[i] = *reinterpret_cast<const float4 *>(x + (size_t)t * H + c * kBK + c4 * 4);
        }
        const int r = tid >> 2, c4 = tid & 3, e = e0 + r;
        wv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < E) {
            const uint4 u = ld_stream_v4(wr + (size_t)e * H + c * kBK + c4 * 4);
            wv = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                             __uint_as_float(u.w));
        }
    };
    auto store = [&](int b) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + 256 * i, r = idx >> 2, c4 = idx & 3;
            xs[b][c4 * 4 + 0][r] = xv[i].x; xs[b][c4 * 4 + 1][r] = xv[i].y;
            xs[b][c4 * 4 + 2][r] = xv[i].z; xs[b][c4 * 4 + 3][r] = xv[i].w;
        }
        const int r = tid >> 2, c4 = tid & 3;
        ws[b][c4 * 4 + 0][r] = wv.x; ws[b][c4 * 4 + 1][r] = wv.y;
        ws[b][c4 * 4 + 2][r] = wv.z; ws[b][c4 * 4 + 3][r] = wv.w;
    };
    if (c0 < c1) {
        load(c0);
        store(0);
    }
    __syncthreads();
    for (int c = c0; c < c1; ++c) {
        const int b = (c - c0) & 1;
        if (c + 1 < c1) load(c + 1);
#pragma unroll
        for (int k = 0; k < kBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&xs[b][k][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&xs[b][k][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&ws[b][k][tx * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[4] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (c + 1 < c1) store(b ^ 1);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int t = t0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) part[((size_t)s * T + t) * E + e] = acc[i][j];
        }
    }
}

// A warp of router_cluster_kernel forms two experts' partial logits 16 tokens at a time: the
// 32 values of a pass are summed over the lanes by one reduce-scatter.  A cluster covers the
// 8 warps' 16 experts.
constexpr int kMaxExpertsPerCluster = 16;
constexpr int kRouteStageT = 32;   // tokens of x staged in shared memory at a time
// Batches above this take router_tokens_kernel (GLM decode router + route tail, µs per call
// on a GB300: T = 32 21.4 -> 18.8, T = 64 37.8 -> 33.5; at 8 or fewer tokens the per-expert
// form is as fast).
constexpr int kRouteTokensMinT = 8;

size_t router_stage_bytes(int H, int cs) { return sizeof(float) * kRouteStageT * (H / cs); }

// The end of both cluster routers, once s_part[t][j] holds this CTA's partial logits of the
// cluster's kEPC experts over its slice of H: the |x| maxima of the tokens this cluster
// quantises (t = c mod clusters), the logits of the tokens t = r (mod CS) summed over the
// ranks in rank order through distributed shared memory, then the int8 codes of x.  xs, when
// not null, holds this rank's slice of every token's x in shared memory ([T][L/4] float4s),
// which is then read instead of global memory.
template <int kEPC>
__device__ __forceinline__ void cluster_router_finish(cooperative_groups::cluster_group &cl,
                                                      const float *__restrict__ x, int T, int H,
                                                      int E, float *__restrict__ logits,
                                                      const QuantRows &xq, int quant,
                                                      float (*s_part)[kMaxExpertsPerCluster],
                                                      float *s_amax, float *s_red,
                                                      const float4 *xs)
{
    const int CS = (int)cl.num_blocks(), r = (int)cl.block_rank();
    const int c = blockIdx.x / CS, ncl = gridDim.x / CS;
    const int L = H / CS, k0 = r * L, nunit = L / 4;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    // |x| maximum of this slice for the tokens this cluster quantises
    if (quant) {
        for (int i = 0, t = c; t < T; ++i, t += ncl) {
            float m = 0.0f;
            for (int idx = tid; idx < nunit; idx += blockDim.x) {
                const float4 v = xs ? xs[(size_t)t * nunit + idx]
                                    : __ldg(reinterpret_cast<const float4 *>(x + (size_t)t * H + k0 + idx * 4));
                m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) s_red[wid] = m;
            __syncthreads();
            if (tid == 0) {
                float v = s_red[0];
                for (int q = 1; q < 8; ++q) v = fmaxf(v, s_red[q]);
                s_amax[i] = v;
            }
            __syncthreads();
        }
    }
    cl.sync();

    // logits of the tokens t = r (mod CS): the CS slices summed in rank order
    const int mine = r < T ? (T - r + CS - 1) / CS : 0;
    for (int pidx = tid; pidx < mine * kEPC; pidx += blockDim.x) {
        const int t = r + (pidx / kEPC) * CS, j = pidx % kEPC;
        const int e = c * kEPC + j;
        if (e >= E) continue;
        float sum = 0.0f;
        for (int q = 0; q < CS; ++q) sum += *cl.map_shared_rank(&s_part[t][j], q);
        logits[(size_t)t * E + e] = sum;
    }
    // int8 codes of this slice for the cluster's tokens (runs of 8 as [e0 e2 e4 e6|e1 e3 e5 e7],
    // code sums per 32-element chunk), the row scale from rank 0
    if (quant) {
        for (int i = 0, t = c; t < T; ++i, t += ncl) {
            float amax = 0.0f;
            for (int q = 0; q < CS; ++q) amax = fmaxf(amax, *cl.map_shared_rank(&s_amax[i], q));
            const float inv = quant_inv(amax);
            const int runs = L / 8;
            for (int base = 0; base < runs; base += blockDim.x) {
                const int run = base + tid;
                if (base + (tid & ~31) >= runs) break;   // whole warp past the end
                int sum = 0;
                if (run < runs) {
                    const float *v = x + (size_t)t * H + k0 + run * 8;
                    const float4 a = xs ? xs[(size_t)t * nunit + 2 * run] : __ldg(reinterpret_cast<const float4 *>(v));
                    const float4 b = xs ? xs[(size_t)t * nunit + 2 * run + 1]
                                        : __ldg(reinterpret_cast<const float4 *>(v + 4));
                    const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                    const uint2 pk = quant_pack8(xv, inv, sum);
                    *reinterpret_cast<uint2 *>(xq.q + (size_t)t * xq.q_ld + k0 + run * 8) = pk;
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if ((lane & 3) == 0 && run < runs) xq.csum[(size_t)t * xq.c_ld + (k0 + run * 8) / 32] = sum;
            }
            if (r == 0 && tid == 0) xq.scale[t] = quant_scale(amax);
        }
    }
    cl.sync();   // no CTA leaves while another still reads its shared memory
}

// Decode-sized batches of up to kRouteTokensMinT tokens: logits of 16 experts x all T tokens
// per cluster, x quantisation.  MAXU bounds the float4 units of the H slice that one lane
// holds per expert.
template <int MAXU>
__global__ void __launch_bounds__(256, 2) router_cluster_kernel(const float *__restrict__ x,
                                                                const float *__restrict__ wr,
                                                                int T, int H, int E,
                                                                float *__restrict__ logits,
                                                                QuantRows xq, int quant)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) char router_smem[];
    constexpr int XPW = 2, kEPC = 8 * XPW, kTP = 32 / XPW;
    __shared__ float s_part[kRouteClusterMaxT][kMaxExpertsPerCluster];
    __shared__ float s_amax[kRouteClusterMaxT];
    __shared__ float s_red[8];

    const int CS = (int)cl.num_blocks(), r = (int)cl.block_rank();
    const int c = blockIdx.x / CS;
    const int L = H / CS, k0 = r * L, nunit = L / 4;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int e0 = c * kEPC + XPW * wid;

    // The router weights are a layer parameter, not an output of earlier work on the stream:
    // they are loaded (without L1 allocation) before the dependency wait, so the loads
    // overlap the end of the kernel before this one.
    // Read once per call: evict-first in L2.
    const uint64_t pol = l2_policy_evict_first();
    float4 wv[XPW][MAXU];
#pragma unroll
    for (int j = 0; j < XPW; ++j) {
        const int e = e0 + j;
#pragma unroll
        for (int u = 0; u < MAXU; ++u) {
            const int idx = u * 32 + lane;
            wv[j][u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < E && idx < nunit) {
                const uint4 q = ld_stream_v4_hint(wr + (size_t)e * H + k0 + idx * 4, pol);
                wv[j][u] = make_float4(__uint_as_float(q.x), __uint_as_float(q.y),
                                       __uint_as_float(q.z), __uint_as_float(q.w));
            }
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    // x slices of kRouteStageT tokens at a time, staged in shared memory by cp.async; each
    // warp then forms its experts' partial logits for kTP tokens at once and sums the 32
    // values over its lanes with one reduce-scatter (lane l: expert l / kTP, token l % kTP)
    float4 *s_x = reinterpret_cast<float4 *>(router_smem);
    for (int t0 = 0; t0 < T; t0 += kRouteStageT) {
        const int nt = min(kRouteStageT, T - t0);
        for (int idx = tid; idx < nt * nunit; idx += blockDim.x) {
            const int tt = idx / nunit, u = idx - tt * nunit;
            cp_async16(s_x + idx, x + (size_t)(t0 + tt) * H + k0 + u * 4, true);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        for (int tg = 0; tg < nt; tg += kTP) {
            float acc[32];
#pragma unroll
            for (int o = 0; o < 32; ++o) acc[o] = 0.0f;
#pragma unroll
            for (int u = 0; u < MAXU; ++u) {
                const int idx = u * 32 + lane;
                if (idx < nunit) {
#pragma unroll
                    for (int tt = 0; tt < kTP; ++tt) {
                        if (tg + tt < nt) {
                            const float4 xv = s_x[(tg + tt) * nunit + idx];
#pragma unroll
                            for (int j = 0; j < XPW; ++j) {
                                float &a_ = acc[j * kTP + tt];
                                a_ = fmaf(xv.x, wv[j][u].x, a_);
                                a_ = fmaf(xv.y, wv[j][u].y, a_);
                                a_ = fmaf(xv.z, wv[j][u].z, a_);
                                a_ = fmaf(xv.w, wv[j][u].w, a_);
                            }
                        }
                    }
                }
            }
            ReduceScatter<32, 16>::run(acc, lane);
            const int tt = lane % kTP;
            if (tg + tt < nt) s_part[t0 + tg + tt][XPW * wid + lane / kTP] = acc[0];
        }
        __syncthreads();   // before the next slice of x overwrites s_x
    }
    // at most kRouteTokensMinT tokens, i.e. one stage: s_x still holds every token's slice
    cluster_router_finish<kEPC>(cl, x, T, H, E, logits, xq, quant, s_part, s_amax, s_red,
                                T <= kRouteStageT ? s_x : nullptr);
}


// Batches of more than kRouteTokensMinT tokens: the same clusters (CS ranks over H, 8 experts
// per cluster), with tokens on the lanes instead.  Warp w of rank r takes the w-th eighth of
// the rank's H slice for all 8 experts and 32 tokens at a time (lane = token): a lane reads its
// token's x from L2 once and the experts' router weights as shared-memory broadcasts, so no
// lane re-reads x from shared memory per expert (the per-expert form of router_cluster_kernel
// is bound by shared-memory bandwidth there).  A lane's sum runs over its eighth in k order;
// the eight warps' sums are added in warp order, the ranks' in rank order.
__global__ void __launch_bounds__(256, 2) router_tokens_kernel(const float *__restrict__ x,
                                                               const float *__restrict__ wr,
                                                               int T, int H, int E,
                                                               float *__restrict__ logits,
                                                               QuantRows xq, int quant)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    constexpr int kEPC = 8;
    extern __shared__ __align__(16) char router_smem[];
    __shared__ float s_part[kRouteClusterMaxT][kMaxExpertsPerCluster];
    __shared__ float s_tp[8][32][kEPC + 1];   // the warps' partial sums (padded rows)
    __shared__ float s_amax[kRouteClusterMaxT];
    __shared__ float s_red[8];

    const int CS = (int)cl.num_blocks(), r = (int)cl.block_rank();
    const int c = blockIdx.x / CS;
    const int L = H / CS, k0 = r * L;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int e0 = c * kEPC;
    const int nq = L / 32;           // float4 units of a warp's eighth of the slice
    const int kw = wid * (L / 8);    // its first element within the slice

    // the cluster's router weights for this slice, [expert][L] in shared memory; a layer
    // parameter, so copied (evict-first in L2: read once per call) before the dependency wait
    float4 *s_w = reinterpret_cast<float4 *>(router_smem);
    {
        const uint64_t pol = l2_policy_evict_first();
        const int units = L / 4;
        for (int idx = tid; idx < kEPC * units; idx += blockDim.x) {
            const int j = idx / units, u = idx - j * units;
            const int e = e0 + j;
            cp_async16_hint(s_w + idx, wr + (size_t)(e < E ? e : 0) * H + k0 + u * 4, e < E, pol);
        }
        cp_async_commit();
    }
    pdl_wait();
    pdl_launch_dependents();
    cp_async_wait<0>();
    __syncthreads();

    const float4 *sw = s_w + kw / 4;
    for (int t0 = 0; t0 < T; t0 += 32) {
        const int t = t0 + lane;
        const bool tv = t < T;
        const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)(tv ? t : 0) * H + k0 + kw);
        float acc[kEPC];
#pragma unroll
        for (int j = 0; j < kEPC; ++j) acc[j] = 0.0f;
        for (int q0 = 0; q0 < nq; q0 += 8) {
            float4 xv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                xv[i] = tv && q0 + i < nq ? __ldg(xr + q0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (q0 + i < nq) {
#pragma unroll
                    for (int j = 0; j < kEPC; ++j) {
                        const float4 w4 = sw[j * (L / 4) + q0 + i];
                        acc[j] = fmaf(xv[i].x, w4.x, acc[j]);
                        acc[j] = fmaf(xv[i].y, w4.y, acc[j]);
                        acc[j] = fmaf(xv[i].z, w4.z, acc[j]);
                        acc[j] = fmaf(xv[i].w, w4.w, acc[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kEPC; ++j) s_tp[wid][lane][j] = acc[j];
        __syncthreads();
        {
            // thread (token tok, expert j): the eight warps' sums in warp order
            const int tok = tid >> 3, j = tid & 7;
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) sum += s_tp[w][tok][j];
            if (t0 + tok < T) s_part[t0 + tok][j] = sum;
        }
        __syncthreads();   // before the next pass overwrites s_tp
    }
    cluster_router_finish<kEPC>(cl, x, T, H, E, logits, xq, quant, s_part, s_amax, s_red, nullptr);
}

__global__ void __launch_bounds__(256) router_select_kernel(const float *__restrict__ part, int S,
                                                            int T, SelectParams p,
                                                            int32_t *__restrict__ ids,
                                                            float *__restrict__ w,
                                                            int32_t *__restrict__ keff)
{
    pdl_wait();
    pdl_launch_dependents();
    const int wid = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + wid;
    if (t >= T) return;
    const int E = p.E;
    auto logit = [&](int e) {
        float l = 0.0f;
        for (int s = 0; s < S; ++s) l += part[((size_t)s * T + t) * E + e];
        return l;
    };
    select_token(p, logit, t, ids, w, keff);
}

}  // namespace

int router_splits(const moe_config &c, int T)
{
    const int nch = c.hidden / kBK;
    const long long base = (long long)((T + kBT - 1) / kBT) * ((c.n_experts + kBE - 1) / kBE);
    long long s = (kTargetCtas + base - 1) / (base > 0 ? base : 1);
    if (s > nch) s = nch;
    // partial logits within kRouteScratchFloats whenever one split fits
    const long long cap = (long long)kRouteScratchFloats / ((long long)(T > 0 ? T : 1) * c.n_experts);
    if (s > cap) s = cap;
    if (s < 1) s = 1;
    return (int)s;
}

int route_cluster_size(int H)
{
    for (int cs = 8; cs > 1; cs >>= 1)
        if ((H / cs) % 32 == 0) return cs;
    return 1;
}

cudaError_t launch_router_logits(const moe_config &c, const float *x, const float *wr, int T,
                                 float *scratch, const QuantRows *xq, int *splits, cudaStream_t st)
{
    *splits = 1;
    if (T <= 0) return cudaSuccess;
    const int H = c.hidden, E = c.n_experts;
    if (T <= kRouteClusterMaxT) {
        const int cs = route_cluster_size(H);
        const int units = (H / cs / 4 + 31) / 32;   // float4 units per lane and expert
        const QuantRows q = xq ? *xq : QuantRows{};
        const int quant = xq ? 1 : 0;
        // tokens on the lanes once a pass holds enough of them
        if (T > kRouteTokensMinT) {
            const dim3 grid(cs * ((E + 7) / 8));
            const size_t smem = sizeof(float) * 8 * (H / cs);
            return launch_kernel(router_tokens_kernel, grid, dim3(256), smem, st, cs, x, wr, T, H, E,
                                 scratch, q, quant);
        }
        const dim3 grid(cs * ((E + 15) / 16));
        const size_t smem = router_stage_bytes(H, cs);
        auto go = [&](auto kernel) {
            return launch_kernel(kernel, grid, dim3(256), smem, st, cs, x, wr, T, H, E, scratch,
                                 q, quant);
        };
        if (units <= 2) return go(router_cluster_kernel<2>);
        if (units <= 4) return go(router_cluster_kernel<4>);
        return go(router_cluster_kernel<8>);
    }
    const int S = router_splits(c, T);
    *splits = S;
    const dim3 grid((T + kBT - 1) / kBT, (E + kBE - 1) / kBE, S);
    return launch_kernel(router_logits_kernel, grid, dim3(256), 0, st, 1, x, wr, T, H, E, S,
                         scratch);
}

cudaError_t launch_router_select(const moe_config &c, const float *scratch, int splits,
                                 const float *bias, int T, int32_t *ids, float *w, int32_t *keff,
                                 cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    return launch_kernel(router_select_kernel, dim3((T + 7) / 8), dim3(256), 0, st, 1,
                         (const float *)scratch, splits, T, select_params(c, bias), ids, w, keff);
}

cudaError_t launch_router(const moe_config &c, const float *x, const float *wr, const float *bias,
                          int T, float *scratch, int32_t *ids, float *w, int32_t *keff,
                          cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    int S = 1;
    cudaError_t e = launch_router_logits(c, x, wr, T, scratch, nullptr, &S, st);
    if (e != cudaSuccess) return e;
    if (T <= kRouteClusterMaxT)
        return launch_route_tail(c, scratch, bias, T, ids, w, keff, nullptr, nullptr, st);
    return launch_router_select(c, scratch, S, bias, T, ids, w, keff, st);
}

}  // namespace moe
