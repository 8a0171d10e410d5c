// quant.cu -- per-row symmetric int8 quantisation: of the layer input x, done once per
// layer and shared by every expert that reads the token ["colibri 开发演进实录" §2.2:
// activation quantisation hoisted to the layer], and of h = SiLU(gate)*up before the down
// projection.  One CTA per row.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kQThreads = 256;

// the int8 codes of 8 consecutive values as bf16 (exact), 16 bytes in the tensor-core path's
// order e0 e4 e1 e5 e2 e6 e3 e7 (the order in which its weight nibbles unpack)
__device__ __forceinline__ void store_codes_bf16(__nv_bfloat16 *dst, const float v[8], float inv)
{
    __nv_bfloat162 p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = __floats2bfloat162_rn((float)quant_code(v[i], inv), (float)quant_code(v[i + 4], inv));
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(p);
}
constexpr int kMaxSlices = kMaxDim / (32 * kSliceChunks);   // slices of a row of kMaxDim inputs

// Quantises one row of n values (n a multiple of 32) with the whole block: codes in runs of
// 8 stored [e0 e2 e4 e6 | e1 e3 e5 e7], the code sum of every 32-element chunk, the scale.
// canon (nullable) receives the codes in element order.
__device__ void quant_row_block(const float *__restrict__ v, int n, int8_t *__restrict__ q,
                                int32_t *__restrict__ csum, float *__restrict__ scale,
                                int8_t *__restrict__ canon, float *__restrict__ canon_scale,
                                __nv_bfloat16 *__restrict__ qb)
{
    __shared__ float s_max[kQThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
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

    const int runs = n / 8;
    for (int base = 0; base < runs; base += kQThreads) {
        const int run = base + tid;
        if (base + (tid & ~31) >= runs) break;   // whole warp past the end
        int sum = 0;
        if (run < runs) {
            const float4 a = *reinterpret_cast<const float4 *>(v + run * 8);
            const float4 b = *reinterpret_cast<const float4 *>(v + run * 8 + 4);
            const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            const uint2 pk = quant_pack8(x, inv, sum);
            *reinterpret_cast<uint2 *>(q + run * 8) = pk;
            if (canon) {
#pragma unroll
                for (int i = 0; i < 8; ++i) canon[run * 8 + i] = (int8_t)quant_code(x[i], inv);
            }
            if (qb) store_codes_bf16(qb + run * 8, x, inv);
        }
        // the 4 runs of a 32-element chunk are 4 consecutive lanes
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((lane & 3) == 0 && run < runs) csum[run / 4] = sum;
    }
    if (tid == 0) {
        *scale = quant_scale(amax);
        if (canon_scale) *canon_scale = quant_scale(amax);
    }
}

__global__ void __launch_bounds__(kQThreads) quant_rows_kernel(const float *__restrict__ src,
                                                               int n, int stride, QuantRows dst)
{
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x;
    quant_row_block(src + (size_t)row * stride, n, dst.q + (size_t)row * dst.q_ld,
                    dst.csum + (size_t)row * dst.c_ld, dst.scale + row, nullptr, nullptr,
                    dst.bf16 ? dst.bf16 + (size_t)row * dst.q_ld : nullptr);
}

// Sliced gate/up rows: h = SiLU(gate) * up of the row, gate and up each the sum of the S
// slice planes in slice order, formed in registers -- run r (8 consecutive values) by thread
// r % 256 -- and quantised from there like quant_row_block does.
template <int MAXS>
__device__ void quant_h_planes_block(const float *__restrict__ gp, const float *__restrict__ up,
                                     int S, int64_t plane, int n, int8_t *__restrict__ q,
                                     int32_t *__restrict__ csum, float *__restrict__ scale,
                                     int8_t *__restrict__ canon, float *__restrict__ canon_scale,
                                     __nv_bfloat16 *__restrict__ qb)
{
    constexpr int kRuns = kMaxDim / 8 / kQThreads;   // runs per thread, at most
    __shared__ float s_max[kQThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int runs = n / 8;
    float h[kRuns][8];
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < kRuns; ++k) {
        const int run = tid + kQThreads * k;
#pragma unroll
        for (int i = 0; i < 8; ++i) h[k][i] = 0.0f;
        if (run >= runs) continue;
        float4 g[MAXS][2], u[MAXS][2];
#pragma unroll
        for (int s = 0; s < MAXS; ++s) {   // every plane's loads first
            if (s < S) {
                const float4 *gs = reinterpret_cast<const float4 *>(gp + s * plane + run * 8);
                const float4 *us = reinterpret_cast<const float4 *>(up + s * plane + run * 8);
                g[s][0] = gs[0]; g[s][1] = gs[1];
                u[s][0] = us[0]; u[s][1] = us[1];
            }
        }
        float gv[8] = {g[0][0].x, g[0][0].y, g[0][0].z, g[0][0].w, g[0][1].x, g[0][1].y, g[0][1].z, g[0][1].w};
        float uv[8] = {u[0][0].x, u[0][0].y, u[0][0].z, u[0][0].w, u[0][1].x, u[0][1].y, u[0][1].z, u[0][1].w};
#pragma unroll
        for (int s = 1; s < MAXS; ++s) {
            if (s < S) {
                const float ga[8] = {g[s][0].x, g[s][0].y, g[s][0].z, g[s][0].w, g[s][1].x, g[s][1].y, g[s][1].z, g[s][1].w};
                const float ua[8] = {u[s][0].x, u[s][0].y, u[s][0].z, u[s][0].w, u[s][1].x, u[s][1].y, u[s][1].z, u[s][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    gv[i] += ga[i];
                    uv[i] += ua[i];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            h[k][i] = gv[i] / (1.0f + expf(-gv[i])) * uv[i];
            amax = fmaxf(amax, fabsf(h[k][i]));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) s_max[wid] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, s_max[w]);
    const float inv = quant_inv(amax);
#pragma unroll
    for (int k = 0; k < kRuns; ++k) {
        const int run = tid + kQThreads * k;
        if (kQThreads * k >= runs) break;   // uniform: the whole block is past the end
        int sum = 0;
        if (run < runs) {
            const uint2 pk = quant_pack8(h[k], inv, sum);
            *reinterpret_cast<uint2 *>(q + run * 8) = pk;
            if (canon) {
#pragma unroll
                for (int i = 0; i < 8; ++i) canon[run * 8 + i] = (int8_t)quant_code(h[k][i], inv);
            }
            if (qb) store_codes_bf16(qb + run * 8, h[k], inv);
        }
        // the 4 runs of a 32-element chunk are 4 consecutive lanes
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((lane & 3) == 0 && run < runs) csum[run / 4] = sum;
    }
    if (tid == 0) {
        *scale = quant_scale(amax);
        if (canon_scale) *canon_scale = quant_scale(amax);
    }
}

// h rows: [0, first) of n_first values (the shared expert), then the routed pair rows,
// as many as *rest_count (device value; null = none), of n_rest values.  With `planes` the
// gate/up kernel left gate and up in planes (S per-slice planes of sliced rows, or one plane
// each from the tensor-core path) and h is formed from them (quant_h_planes_block).
// MAXS: slice planes at most (held in registers; 1 for the tensor path and unsliced rows)
template <int MAXS>
__global__ void __launch_bounds__(kQThreads) quant_h_kernel(const float *__restrict__ h, int ld,
                                                            int first, int n_first, int n_rest,
                                                            const int32_t *rest_count,
                                                            int routed_rowbase, QuantRows dst,
                                                            int8_t *probe_hq, float *probe_hs,
                                                            const float *__restrict__ gpart,
                                                            const float *__restrict__ upart,
                                                            int planes, int S, int64_t plane)
{
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x;
    const int rest = rest_count ? *rest_count : 0;
    if (row >= first + rest) return;
    const bool routed = row >= first;
    const int n = routed ? n_rest : n_first;
    const size_t pr = (size_t)(row - routed_rowbase);
    int8_t *canon = (routed && probe_hq) ? probe_hq + pr * n : nullptr;
    float *canon_scale = (routed && probe_hs) ? probe_hs + pr : nullptr;
    __nv_bfloat16 *qb = dst.bf16 ? dst.bf16 + (size_t)row * dst.q_ld : nullptr;
    if (planes)
        quant_h_planes_block<MAXS>(gpart + (size_t)row * ld, upart + (size_t)row * ld, S, plane, n,
                             dst.q + (size_t)row * dst.q_ld, dst.csum + (size_t)row * dst.c_ld,
                             dst.scale + row, canon, canon_scale, qb);
    else
        quant_row_block(h + (size_t)row * ld, n, dst.q + (size_t)row * dst.q_ld,
                        dst.csum + (size_t)row * dst.c_ld, dst.scale + row, canon, canon_scale, qb);
}

// The x codes of every output row of an FFN call as bf16, for the tensor-core path's B
// operand: rows [0, first) are the shared expert's (token = row), rows routed_rowbase + p
// the routed pairs (token = tok[p], p < *rest_count).  Codes come from the run layout
// [e0 e2 e4 e6 | e1 e3 e5 e7] and go out in the order e0 e4 e1 e5 e2 e6 e3 e7.
__global__ void __launch_bounds__(kQThreads) gather_x_bf16_kernel(QuantRows xq, int n, int first,
                                                                  int routed_rowbase,
                                                                  const int32_t *rest_count,
                                                                  const int32_t *tok,
                                                                  __nv_bfloat16 *dst)
{
    pdl_wait();
    pdl_launch_dependents();
    const int row = blockIdx.x;
    int token;
    if (row < first) {
        token = row;
    } else {
        const int p = row - routed_rowbase;
        const int rest = rest_count ? *rest_count : 0;
        if (p < 0 || p >= rest) return;
        token = tok[p];
    }
    const int8_t *src = xq.q + (size_t)token * xq.q_ld;
    __nv_bfloat16 *out = dst + (size_t)row * n;
    for (int run = threadIdx.x; run < n / 8; run += kQThreads) {
        const uint2 v = *reinterpret_cast<const uint2 *>(src + run * 8);
        // v.x bytes: e0 e2 e4 e6, v.y bytes: e1 e3 e5 e7
        auto code = [](uint32_t w, int b) { return (float)(int8_t)(w >> (8 * b)); };
        __nv_bfloat162 p[4];
        p[0] = __floats2bfloat162_rn(code(v.x, 0), code(v.x, 2));   // e0 e4
        p[1] = __floats2bfloat162_rn(code(v.y, 0), code(v.y, 2));   // e1 e5
        p[2] = __floats2bfloat162_rn(code(v.x, 1), code(v.x, 3));   // e2 e6
        p[3] = __floats2bfloat162_rn(code(v.y, 1), code(v.y, 3));   // e3 e7
        *reinterpret_cast<uint4 *>(out + run * 8) = *reinterpret_cast<const uint4 *>(p);
    }
}

}  // namespace

cudaError_t launch_gather_x_bf16(const FfnArgs &a, int first_rows, int max_rows, cudaStream_t st)
{
    if (max_rows <= 0) return cudaSuccess;
    const int32_t *rest = a.include_routed ? a.offsets + a.E : nullptr;
    return launch_kernel(gather_x_bf16_kernel, dim3(max_rows), dim3(kQThreads), 0, st, 1, a.xq, a.H,
                         first_rows, a.routed_rowbase, rest, a.tok, a.x_bf16);
}

cudaError_t launch_quant_rows(const float *src, int rows, int n, int src_stride, QuantRows dst,
                              cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    return launch_kernel(quant_rows_kernel, dim3(rows), dim3(kQThreads), 0, st, 1, src, n,
                         src_stride, dst);
}

cudaError_t launch_quant_h(const FfnArgs &a, int first_rows, int n_first, int n_rest,
                           int max_rows, cudaStream_t st)
{
    if (max_rows <= 0) return cudaSuccess;
    const int32_t *rest = a.include_routed ? a.offsets + a.E : nullptr;
    // gate/up left per-slice planes (sliced rows) or one plane per matrix (tensor path)
    const int S = a.tensor ? 1 : (a.slice_gu ? a.geo_gu[0].S : 1);
    const int planes = (a.tensor || S > 1) ? 1 : 0;
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, dim3(max_rows), dim3(kQThreads), 0, st, 1,
                             (const float *)a.h, a.hstride, first_rows, n_first, n_rest, rest,
                             a.routed_rowbase, a.hq, a.probe.hq, a.probe.h_scale,
                             (const float *)a.gpart, (const float *)a.upart, planes, S,
                             (int64_t)a.plane_rows * a.hstride);
    };
    return S <= 1 ? go(quant_h_kernel<1>) : go(quant_h_kernel<kMaxSlices>);
}

}  // namespace moe
