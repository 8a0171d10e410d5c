// quantize_weights.cu -- offline fp32 -> int4-gs64 weight quantiser, the container format the
// layer reads ["colibri 开发演进实录" §2.1 int4-gs64; the conversion tool, `coli convert`, §9],
// and its 3-bit variant int3-g64 (fmt=5, ibid. §8.3).
// Per 64-weight group: scale = amax / 7 and u = clamp(rint(w * (7 / amax)), -7, 7) + 8 in fp32
// (round half to even), so the group's largest magnitude lands on +-7; an all-zero group gets
// scale 0 and codes 8.  Byte j of a row holds element 2j in its low nibble, 2j+1 in its high.
#include "device_util.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kQwThreads = 256;   // 8 warps
constexpr int kQwPairs = 8;       // pairs of 64-weight groups per warp, all loads issued first

// A warp quantises 2*kQwPairs consecutive groups, a pair per step: half-warp h takes group
// 2p+h, its lane l (0..15) elements 4l..4l+3 (one float4) into bytes 2l and 2l+1.  Rows are
// contiguous and K is a multiple of 64, so group gi (row-major over all rows) starts at
// weight 64*gi, packed byte 32*gi and scale gi.
__global__ void __launch_bounds__(kQwThreads) quantize_int4_kernel(const float *__restrict__ w,
                                                                   long long groups,
                                                                   uint8_t *__restrict__ packed,
                                                                   float *__restrict__ scales)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, h = lane >> 4, l = lane & 15;
    const long long g0 = (((long long)blockIdx.x * kQwThreads + threadIdx.x) >> 5) * (2 * kQwPairs);
    if (g0 >= groups) return;
    float4 v[kQwPairs];
#pragma unroll
    for (int p = 0; p < kQwPairs; ++p) {
        const long long gi = g0 + 2 * p + h;
        v[p] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (gi < groups) v[p] = reinterpret_cast<const float4 *>(w + gi * 64)[l];
    }
#pragma unroll
    for (int p = 0; p < kQwPairs; ++p) {
        if (g0 + 2 * p >= groups) break;   // uniform across the warp
        const long long gi = g0 + 2 * p + h;
        float amax = fmaxf(fmaxf(fabsf(v[p].x), fabsf(v[p].y)), fmaxf(fabsf(v[p].z), fabsf(v[p].w)));
        // max over the half-warp (offsets below 16 stay inside it)
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float inv = amax > 0.0f ? 7.0f / amax : 0.0f;
        auto code = [inv](float x) {
            const float q = fminf(fmaxf(rintf(x * inv), -7.0f), 7.0f);
            return (uint32_t)((int)q + 8);
        };
        if (gi < groups) {
            const uint32_t b0 = code(v[p].x) | (code(v[p].y) << 4);
            const uint32_t b1 = code(v[p].z) | (code(v[p].w) << 4);
            reinterpret_cast<uint16_t *>(packed + gi * 32)[l] = (uint16_t)(b0 | (b1 << 8));
            if (l == 0) scales[gi] = amax / 7.0f;
        }
    }
}

// int3-g64 (fmt=5, "colibri 开发演进实录" §8.3): scale = amax / 3 and
// u = clamp(rint(w * (3 / amax)), -3, 3) + 4 per 64-weight group, the group packed into 24
// bytes with weight k in bits 3k .. 3k+2 of its little-endian bit string.  Same work split as
// the int4 kernel: half-warp h takes group 2p+h, lane l its elements 4l..4l+3 (12 bits, at
// bit 12l of the group); lane 2m joins its partner's 12 bits and stores bytes 3m .. 3m+2.
__global__ void __launch_bounds__(kQwThreads) quantize_int3_kernel(const float *__restrict__ w,
                                                                   long long groups,
                                                                   uint8_t *__restrict__ packed,
                                                                   float *__restrict__ scales)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, h = lane >> 4, l = lane & 15;
    const long long g0 = (((long long)blockIdx.x * kQwThreads + threadIdx.x) >> 5) * (2 * kQwPairs);
    if (g0 >= groups) return;
    float4 v[kQwPairs];
#pragma unroll
    for (int p = 0; p < kQwPairs; ++p) {
        const long long gi = g0 + 2 * p + h;
        v[p] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (gi < groups) v[p] = reinterpret_cast<const float4 *>(w + gi * 64)[l];
    }
#pragma unroll
    for (int p = 0; p < kQwPairs; ++p) {
        if (g0 + 2 * p >= groups) break;   // uniform across the warp
        const long long gi = g0 + 2 * p + h;
        float amax = fmaxf(fmaxf(fabsf(v[p].x), fabsf(v[p].y)), fmaxf(fabsf(v[p].z), fabsf(v[p].w)));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float inv = amax > 0.0f ? 3.0f / amax : 0.0f;
        auto code = [inv](float x) {
            const float q = fminf(fmaxf(rintf(x * inv), -3.0f), 3.0f);
            return (uint32_t)((int)q + 4);
        };
        const uint32_t c12 = code(v[p].x) | (code(v[p].y) << 3) | (code(v[p].z) << 6) | (code(v[p].w) << 9);
        const uint32_t hi = __shfl_down_sync(0xffffffffu, c12, 1);
        if (gi < groups) {
            if ((l & 1) == 0) {
                const uint32_t v24 = c12 | (hi << 12);
                uint8_t *dst = packed + gi * 24 + 3 * (l >> 1);
                dst[0] = (uint8_t)v24;
                dst[1] = (uint8_t)(v24 >> 8);
                dst[2] = (uint8_t)(v24 >> 16);
            }
            if (l == 0) scales[gi] = amax / 3.0f;
        }
    }
}

}  // namespace

cudaError_t launch_quantize_int3(const float *w, int rows, int K, uint8_t *packed, float *scales,
                                 cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    const int G = K / 64;
    const long long groups = (long long)rows * G;
    const long long warps = (groups + 2 * kQwPairs - 1) / (2 * kQwPairs);
    const long long blocks = (warps * 32 + kQwThreads - 1) / kQwThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_kernel(quantize_int3_kernel, dim3((unsigned)blocks), dim3(kQwThreads), 0, st, 1,
                         w, groups, packed, scales);
}

cudaError_t launch_quantize_int4(const float *w, int rows, int K, uint8_t *packed, float *scales,
                                 cudaStream_t st)
{
    if (rows <= 0) return cudaSuccess;
    const int G = K / 64;
    const long long groups = (long long)rows * G;
    const long long warps = (groups + 2 * kQwPairs - 1) / (2 * kQwPairs);
    const long long blocks = (warps * 32 + kQwThreads - 1) / kQwThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_kernel(quantize_int4_kernel, dim3((unsigned)blocks), dim3(kQwThreads), 0, st, 1,
                         w, groups, packed, scales);
}

}  // namespace moe
