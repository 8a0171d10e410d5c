// device_util.cuh -- small device helpers used by several kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint4 ld_stream_v4_hint(const void *p, uint64_t pol)
{
    // ld_stream_v4 with an L2 eviction policy (createpolicy value)
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

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

// Sums each of n values (n a power of two, <= 32) over the 32 lanes: at offsets 16, 8, ...
// a lane keeps one half of its values, sends the other half to its partner and adds what
// it receives; once one value is left the remaining offsets add it up.  Lane l ends with the
// total of value l >> (5 - log2 n).
template <int n, int d>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int lane)
    {
        if constexpr (d > 0) {
            if constexpr (n > 1) {
                const bool up = (lane & d) != 0;
#pragma unroll
                for (int i = 0; i < n / 2; ++i) {
                    const float send = up ? v[i] : v[i + n / 2];
                    const float keep = up ? v[i + n / 2] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, d);
                }
                ReduceScatter<n / 2, d / 2>::run(v, lane);
            } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], d);
                ReduceScatter<1, d / 2>::run(v, lane);
            }
        }
    }
};

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

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

// ---------------------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA, 1-D) helpers.  Every wait is bounded: kWaitLimit polls of
// try_wait (each of which may suspend the thread for a short, hardware-defined time).
// ---------------------------------------------------------------------------------------
namespace moe {

constexpr int kWaitLimit = 1 << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// true once the phase with the given parity has completed; false after kWaitLimit polls
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (int n = 0; n < kWaitLimit; ++n)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) global -> shared,
// completing as transaction bytes on `bar`
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace moe

// ---------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with programmatic
// stream serialisation, so it may be scheduled while the kernel before it in the stream is
// still running.  Each kernel therefore calls pdl_wait() before its first access to global
// memory (the wait returns once the previous grid has completed and its writes are
// visible) and pdl_launch_dependents() to let the next kernel be scheduled early.
// ---------------------------------------------------------------------------------------
namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace moe

// ---------------------------------------------------------------------------------------
// cp.async (global -> shared, per thread, completion tracked per thread by commit groups).
// With `valid` false nothing is read and the destination is zero-filled; `src` must still
// be a mapped global address.
// ---------------------------------------------------------------------------------------
namespace moe {

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}

// The same copies with an L2 eviction policy (a createpolicy value, below).
__device__ __forceinline__ void cp_async16_hint(void *dst, const void *src, bool valid, uint64_t pol)
{
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(valid ? 16 : 0), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async4_hint(void *dst, const void *src, bool valid, uint64_t pol)
{
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2, %3;" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(valid ? 4 : 0), "l"(pol)
                 : "memory");
}

// L2 eviction policies.  The last read of a weight in a launch (an expert's matrices and
// scales by its last token chunk, the router's weights) is evict-first: the weight stream,
// larger than L2, then displaces itself rather than the layer's small reused state
// (activation codes, routing tables, partial sums, the kernels' code).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace moe
