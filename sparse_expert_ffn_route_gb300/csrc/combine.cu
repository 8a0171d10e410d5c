// combine.cu -- gated sum of each token's kept experts plus the shared expert
// ["MoE 路由与专家流式加载" §1.3, §1.4]:
//     y[t] = sum_{i < keff[t]} w[t][i] * y_e(t, i) + y_shared[t]
// summed in slot order, then the shared term, one fp32 FMA chain per output element.  When
// the down rows were sliced, y_e and y_shared are first formed from their slice planes,
// added in slice order.
// The pair holding (t, i) is found by binary search in expert ids[t][i]'s token list,
// which the batch-union sorted by token.
#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kCThreads = 256;

// MAXK pairs and MAXP slice planes at most (the loads are held in registers, so the bounds
// set the register count: the launcher takes the smallest instantiation that covers the call)
template <int MAXK, int MAXP>
__global__ void __launch_bounds__(kCThreads) combine_kernel(
    const float *__restrict__ y_routed, int64_t rstride, const float *__restrict__ y_shared,
    const int32_t *__restrict__ ids, const int32_t *__restrict__ keff,
    const float *__restrict__ w, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ tok, const int32_t *__restrict__ pair_of, int K, int E, int H,
    int S_r, int S_s, int64_t plane, float *__restrict__ y)
{
    __shared__ int s_pair[kMaxTopK];
    __shared__ float s_w[kMaxTopK];
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.y;
    // the token's K entries are read alongside keff (not behind it): one round trip fewer
    // before the pairs' rows can be loaded
    const int kt = keff[t];
    if (threadIdx.x < K) {
        const int i = threadIdx.x;
        const int e = ids[(size_t)t * K + i];
        const float wi = w[(size_t)t * K + i];
        const int pk = pair_of ? pair_of[(size_t)t * K + i] : -1;
        int pair = -1;
        if (i >= max(0, min(K, kt))) {
            // not kept: no pair
        } else if (pair_of) {
            pair = pk;
        } else if (e >= 0 && e < E) {
            int lo = offsets[e], hi = offsets[e + 1];   // first entry >= t
            const int end = hi;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (tok[mid] < t) lo = mid + 1;
                else hi = mid;
            }
            if (lo < end && tok[lo] == t) pair = lo;
        }
        s_pair[i] = pair;   // -1: (t, i) has no pair (inconsistent routing); it adds nothing
        s_w[i] = wi;
    }
    const int k = max(0, min(K, kt));
    __syncthreads();
    const int c = (blockIdx.x * kCThreads + threadIdx.x) * 4;
    if (c >= H) return;
    // every pair's (and the shared expert's) planes are loaded before the ordered sums
    float4 v[MAXK][MAXP];
#pragma unroll
    for (int i = 0; i < MAXK; ++i) {
#pragma unroll
        for (int s = 0; s < MAXP; ++s) {
            v[i][s] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < k && s < S_r && s_pair[i] >= 0)
                v[i][s] = *reinterpret_cast<const float4 *>(y_routed + (size_t)s_pair[i] * rstride + c + s * plane);
        }
    }
    float4 sv[MAXP];
#pragma unroll
    for (int s = 0; s < MAXP; ++s) {
        sv[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (y_shared && s < S_s) sv[s] = *reinterpret_cast<const float4 *>(y_shared + (size_t)t * H + c + s * plane);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < MAXK; ++i) {
        if (i >= k || s_pair[i] < 0) continue;
        float4 e = v[i][0];
#pragma unroll
        for (int s = 1; s < MAXP; ++s) {
            if (s < S_r) {
                e.x += v[i][s].x; e.y += v[i][s].y; e.z += v[i][s].z; e.w += v[i][s].w;
            }
        }
        const float wi = s_w[i];
        acc.x = fmaf(wi, e.x, acc.x);
        acc.y = fmaf(wi, e.y, acc.y);
        acc.z = fmaf(wi, e.z, acc.z);
        acc.w = fmaf(wi, e.w, acc.w);
    }
    if (y_shared) {
        float4 e = sv[0];
#pragma unroll
        for (int s = 1; s < MAXP; ++s) {
            if (s < S_s) {
                e.x += sv[s].x; e.y += sv[s].y; e.z += sv[s].z; e.w += sv[s].w;
            }
        }
        acc.x += e.x; acc.y += e.y; acc.z += e.z; acc.w += e.w;
    }
    *reinterpret_cast<float4 *>(y + (size_t)t * H + c) = acc;
}

}  // namespace

cudaError_t launch_combine(const moe_config &c, const float *y_routed, int64_t routed_row_stride,
                           const float *y_shared, const int32_t *ids, const int32_t *keff,
                           const float *w, const int32_t *offsets, const int32_t *tok,
                           const int32_t *pair_of, int S_r, int S_s, int64_t plane, int T,
                           float *y, cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    dim3 grid((c.hidden / 4 + kCThreads - 1) / kCThreads, T);
    static_assert(kMaxCombinePlanes == 2 && kMaxTopK == 16, "combine instantiations");
    const bool k8 = c.top_k <= 8;
    const bool p1 = S_r <= 1 && (y_shared == nullptr || S_s <= 1);
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, grid, dim3(kCThreads), 0, st, 1, y_routed,
                             (int64_t)routed_row_stride, y_shared, ids, keff, w, offsets, tok,
                             pair_of, c.top_k, c.n_experts, c.hidden, S_r, S_s, plane, y);
    };
    if (k8) return p1 ? go(combine_kernel<8, 1>) : go(combine_kernel<8, 2>);
    return p1 ? go(combine_kernel<16, 1>) : go(combine_kernel<16, 2>);
}

}  // namespace moe
