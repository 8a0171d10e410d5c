// device_util.cuh -- small device helpers used by several kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    // read-only streaming load of 16 bytes that bypasses L1 allocation
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_stream_f32(const float *p)
{
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// 4-way byte dot product: unsigned bytes of a (nibbles, 0..15) times signed bytes of b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Lanes that cooperate on one matrix row whose reduction length has `g`
// 64-groups: the largest power of two <= min(g, 32).
__host__ __device__ __forceinline__ int lanes_per_row(int g)
{
    int l = 1;
    while (l * 2 <= g && l < 32) l *= 2;
    return l;
}

// Per-row symmetric int8 quantisation rule (decisions in fp32, IEEE ops):
// scale = amax / 127; code = clamp(round_half_even(v * (127 / amax)), -127, 127).
__device__ __forceinline__ float quant_inv(float amax)
{
    return amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
}

__device__ __forceinline__ float quant_scale(float amax)
{
    return amax > 0.0f ? __fdiv_rn(amax, 127.0f) : 0.0f;
}

__device__ __forceinline__ int quant_code(float v, float inv)
{
    int q = __float2int_rn(__fmul_rn(v, inv));
    return max(-127, min(127, q));
}

// Quantise 8 consecutive values and pack them as [e0 e2 e4 e6 | e1 e3 e5 e7].
__device__ __forceinline__ uint2 quant_pack8(const float v[8], float inv, int &sum)
{
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = quant_code(v[i], inv);
    sum = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    uint2 w;
    w.x = (uint32_t)(q[0] & 255) | ((uint32_t)(q[2] & 255) << 8) | ((uint32_t)(q[4] & 255) << 16) |
          ((uint32_t)(q[6] & 255) << 24);
    w.y = (uint32_t)(q[1] & 255) | ((uint32_t)(q[3] & 255) << 8) | ((uint32_t)(q[5] & 255) << 16) |
          ((uint32_t)(q[7] & 255) << 24);
    return w;
}

}  // namespace moe
