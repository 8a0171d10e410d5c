// lookahead.cu -- router look-ahead ["MoE 路由与专家流式加载" §5, la_predict]: a layer's
// top-K predicted from a residual state by the layer's own routing pipeline, RMSNorm with
// its norm weight and then its router (sigmoid, bias for the choice, top-K), plus the
// per-token hit count behind the pages' recall figure (the share of the true top-K that the
// prediction holds).
#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kNormThreads = 256;

// out[t][h] = x[t][h] / sqrt(mean_h x[t][h]^2 + eps) * g[h], one CTA per token, fp32; a row
// whose mean square plus eps is 0 normalises to zeros.  H is a multiple of 4.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float *__restrict__ x,
                                                               const float *__restrict__ g,
                                                               float eps, int H,
                                                               float *__restrict__ out)
{
    pdl_wait();
    pdl_launch_dependents();
    __shared__ float s_part[kNormThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)t * H);
    float ss = 0.0f;
    for (int i = tid; i < H / 4; i += kNormThreads) {
        const float4 v = xr[i];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) s_part[wid] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += s_part[w];
    const float ms = tot / (float)H + eps;
    const float inv = ms > 0.0f ? 1.0f / sqrtf(ms) : 0.0f;
    const float4 *gr = reinterpret_cast<const float4 *>(g);
    float4 *orow = reinterpret_cast<float4 *>(out + (size_t)t * H);
    for (int i = tid; i < H / 4; i += kNormThreads) {
        const float4 v = xr[i], w = gr[i];
        orow[i] = make_float4(v.x * inv * w.x, v.y * inv * w.y, v.z * inv * w.z, v.w * inv * w.w);
    }
}

// hits[t] = |{ids_pred[t][i], i < keff_pred[t]} ∩ {ids_true[t][j], j < keff_true[t]}|
__global__ void topk_hits_kernel(const int32_t *__restrict__ ids_pred,
                                 const int32_t *__restrict__ keff_pred,
                                 const int32_t *__restrict__ ids_true,
                                 const int32_t *__restrict__ keff_true, int T, int K,
                                 int32_t *__restrict__ hits)
{
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int kp = min(max(keff_pred[t], 0), K), kt = min(max(keff_true[t], 0), K);
    int n = 0;
    for (int i = 0; i < kp; ++i) {
        const int32_t e = ids_pred[(size_t)t * K + i];
        for (int j = 0; j < kt; ++j)
            if (ids_true[(size_t)t * K + j] == e) {
                ++n;
                break;
            }
    }
    hits[t] = n;
}

}  // namespace

cudaError_t launch_rmsnorm(const float *x, const float *g, float eps, int T, int H, float *out,
                           cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    return launch_kernel(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, st, 1, x, g, eps, H, out);
}

cudaError_t launch_topk_hits(const int32_t *ids_pred, const int32_t *keff_pred,
                             const int32_t *ids_true, const int32_t *keff_true, int T, int K,
                             int32_t *hits, cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    return launch_kernel(topk_hits_kernel, dim3((T + 255) / 256), dim3(256), 0, st, 1, ids_pred,
                         keff_pred, ids_true, keff_true, T, K, hits);
}

}  // namespace moe
