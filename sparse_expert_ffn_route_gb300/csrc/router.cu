// router.cu -- router of the MoE layer: logits, sigmoid scoring, noaux_tc selection bias,
// iterated-argmax top-k, adaptive top-p, norm_topk_prob, routed_scaling_factor
// ["MoE 路由与专家流式加载" §1.1, §1.2].
//
// Two kernels:
//   router_logits_kernel  fp32 x . W_router^T, tiled 64 tokens x 64 experts, split along H
//                         so that even one token spreads the 4*E*H router bytes over the
//                         whole GPU; partial sums go to workspace [S][T][E].
//   router_select_kernel  one warp per token: sums the S partials in a fixed order, then
//                         sigmoid, + bias, K rounds of warp argmax, top-p, norm, scale.
#include <float.h>

#include "device_util.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kBT = 64;   // tokens per tile
constexpr int kBE = 64;   // experts per tile
constexpr int kBK = 32;   // floats of H per stage
constexpr int kTargetCtas = 2 * 152;

__global__ void __launch_bounds__(256) router_logits_kernel(const float *__restrict__ x,
                                                            const float *__restrict__ wr, int T,
                                                            int H, int E, int S,
                                                            float *__restrict__ part)
{
    __shared__ float xs[kBK][kBT + 4];
    __shared__ float ws[kBK][kBE + 4];
    const int t0 = blockIdx.x * kBT, e0 = blockIdx.y * kBE, s = blockIdx.z;
    const int nch = H / kBK;
    const int c0 = (int)((long long)s * nch / S), c1 = (int)((long long)(s + 1) * nch / S);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    for (int c = c0; c < c1; ++c) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int idx = tid + 256 * i, r = idx >> 3, c4 = idx & 7;
            const int t = t0 + r, e = e0 + r;
            float4 xv = make_float4(0.f, 0.f, 0.f, 0.f), wv = xv;
            if (t < T) xv = *reinterpret_cast<const float4 *>(x + (size_t)t * H + c * kBK + c4 * 4);
            if (e < E) {
                const uint4 u = ld_stream_v4(wr + (size_t)e * H + c * kBK + c4 * 4);
                wv = make_float4(__uint_as_float(u.x), __uint_as_float(u.y),
                                 __uint_as_float(u.z), __uint_as_float(u.w));
            }
            xs[c4 * 4 + 0][r] = xv.x; xs[c4 * 4 + 1][r] = xv.y;
            xs[c4 * 4 + 2][r] = xv.z; xs[c4 * 4 + 3][r] = xv.w;
            ws[c4 * 4 + 0][r] = wv.x; ws[c4 * 4 + 1][r] = wv.y;
            ws[c4 * 4 + 2][r] = wv.z; ws[c4 * 4 + 3][r] = wv.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kBK; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs[k][ty * 4]);
            const float4 b = *reinterpret_cast<const float4 *>(&ws[k][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + tx * 4 + j;
            if (e < E) part[((size_t)s * T + t) * E + e] = acc[i][j];
        }
    }
}

constexpr int kPerLane = kMaxExperts / 32;

struct Cand {
    float v;   // choice = sig + bias
    float g;   // sig (the applied gate)
    int e;     // expert id, INT_MAX = none
};

__device__ __forceinline__ bool better(const Cand &a, const Cand &b)
{
    // a beats b: any candidate beats none; larger choice wins; equal choice -> lower id
    if (b.e == 0x7fffffff) return a.e != 0x7fffffff;
    if (a.e == 0x7fffffff) return false;
    return a.v > b.v || (a.v == b.v && a.e < b.e);
}

__global__ void __launch_bounds__(256) router_select_kernel(
    const float *__restrict__ part, int S, int T, int E, int K, const float *__restrict__ bias,
    int norm, float scale, float top_p, int32_t *__restrict__ ids, float *__restrict__ w,
    int32_t *__restrict__ keff)
{
    __shared__ int s_sel[8][kMaxTopK];
    __shared__ float s_g[8][kMaxTopK];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + wid;
    if (t >= T) return;

    float sig[kPerLane], ch[kPerLane];
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
        const int e = lane + 32 * j;
        sig[j] = 0.0f;
        ch[j] = 0.0f;
        if (e < E) {
            float l = 0.0f;
            for (int s = 0; s < S; ++s) l += part[((size_t)s * T + t) * E + e];
            sig[j] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-l)));
            ch[j] = __fadd_rn(sig[j], bias[e]);
        }
    }

    unsigned taken = 0;
    for (int k = 0; k < K; ++k) {
        Cand best{0.0f, 0.0f, 0x7fffffff};
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !((taken >> j) & 1u)) {
                Cand c{ch[j], sig[j], e};
                if (better(c, best)) best = c;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            Cand o;
            o.v = __shfl_xor_sync(0xffffffffu, best.v, off);
            o.g = __shfl_xor_sync(0xffffffffu, best.g, off);
            o.e = __shfl_xor_sync(0xffffffffu, best.e, off);
            if (better(o, best)) best = o;
        }
        if ((best.e & 31) == lane) taken |= 1u << (best.e >> 5);
        if (lane == 0) {
            s_sel[wid][k] = best.e;
            s_g[wid][k] = best.g;
        }
    }
    __syncwarp();

    if (lane == 0) {
        int *sel = s_sel[wid];
        float *g = s_g[wid];
        int m = K;
        if (top_p > 0.0f && top_p < 1.0f) {
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
            const float thr = __fmul_rn(top_p, tot);
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
            if (i < m) {
                const float v = norm ? __fdiv_rn(g[i], ssum) : g[i];
                w[o] = __fmul_rn(v, scale);
                ids[o] = sel[i];
            } else {
                w[o] = 0.0f;
                ids[o] = -1;
            }
        }
        keff[t] = m;
    }
}

}  // namespace

int router_splits(const moe_config &c, int T)
{
    const int nch = c.hidden / kBK;
    const long long base = (long long)((T + kBT - 1) / kBT) * ((c.n_experts + kBE - 1) / kBE);
    long long s = (kTargetCtas + base - 1) / (base > 0 ? base : 1);
    if (s < 1) s = 1;
    if (s > nch) s = nch;
    return (int)s;
}

cudaError_t launch_router(const moe_config &c, const float *x, const float *wr, const float *bias,
                          int T, float *logits_part, int32_t *ids, float *w, int32_t *keff,
                          cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    const int S = router_splits(c, T);
    dim3 grid((T + kBT - 1) / kBT, (c.n_experts + kBE - 1) / kBE, S);
    router_logits_kernel<<<grid, 256, 0, st>>>(x, wr, T, c.hidden, c.n_experts, S, logits_part);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    router_select_kernel<<<(T + 7) / 8, 256, 0, st>>>(logits_part, S, T, c.n_experts, c.top_k,
                                                      bias, c.norm_topk_prob,
                                                      c.routed_scaling_factor, c.top_p, ids, w,
                                                      keff);
    return cudaGetLastError();
}

}  // namespace moe
