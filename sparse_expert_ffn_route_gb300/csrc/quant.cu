// quant.cu -- per-row symmetric int8 quantisation of the layer input, done once per layer
// and shared by every expert that reads the token ["colibri 开发演进实录" §2.2: activation
// quantisation hoisted to the layer].  One CTA per row.
#include "device_util.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kQThreads = 256;

__global__ void __launch_bounds__(kQThreads) quant_rows_kernel(const float *__restrict__ src,
                                                               int n, int stride, QuantRows dst)
{
    __shared__ float s_max[kQThreads / 32];
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float *v = src + (size_t)row * stride;

    float amax = 0.0f;
    for (int i = tid * 4; i < n; i += kQThreads * 4) {
        const float4 x = *reinterpret_cast<const float4 *>(v + i);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) s_max[wid] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
    const float inv = quant_inv(amax);

    const int runs = n / 8, G = n / kGroup;
    for (int base = 0; base < runs; base += kQThreads) {
        const int run = base + tid;
        if (base + (tid & ~31) >= runs) break;   // whole warp past the end
        int sum = 0;
        if (run < runs) {
            const float4 a = *reinterpret_cast<const float4 *>(v + run * 8);
            const float4 b = *reinterpret_cast<const float4 *>(v + run * 8 + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            const uint2 pk = quant_pack8(x, inv, sum);
            *reinterpret_cast<uint2 *>(dst.q + (size_t)row * n + run * 8) = pk;
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if ((lane & 7) == 0 && run < runs) dst.gsum[(size_t)row * G + run / 8] = sum;
    }
    if (tid == 0) dst.scale[row] = quant_scale(amax);
}

}  // namespace

cudaError_t launch_quant_rows(const float *src, int rows, int n, int src_stride, QuantRows dst,
                              cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    quant_rows_kernel<<<rows, kQThreads, 0, st>>>(src, n, src_stride, dst);
    return cudaGetLastError();
}

}  // namespace moe
