// ffn_gemv.cu -- grouped int4 x int8 expert FFN for few tokens per expert (GEMV-shaped,
// HBM-bound): gate/up with SiLU(gate)*up fused, then the down projection with the per-row
// int8 quantisation of h done at the start of each down tile
// ["MoE 路由与专家流式加载" §1.3 (gate/up/SiLU/down on the integer-dot path);
//  "colibri 开发演进实录" §2.2 (K1: unsigned nibbles, dot(u-8, q) = dot(u, q) - 8*sum(q);
//  K1b: integer dot per 64-group, then the group scale)].
//
// Work decomposition: the planner numbers tiles (slot, row block, token chunk) over every
// slot (expert applied to its token list); a persistent grid strides over them.  In a tile,
// each warp owns consecutive rows; the lanes of a row each own whole 64-groups (lane gl owns
// groups gl, gl+L, gl+2L... with L lanes per row), so the int8 activations of a lane's groups
// stay in registers for every row of the tile while the packed nibbles stream from HBM with
// 16-byte read-only loads.  Per group and token:
//     A = sum over 32 bytes of dp4a(lo nibbles, even codes) + dp4a(hi nibbles, odd codes)
//         - 8 * sum(codes of the group)                          (exact int32)
//     acc += s_w[row][group] * A                                   (fp32)
// then the lane partials are summed across the row's lanes and scaled by the token's
// activation scale.
#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

__device__ __forceinline__ int find_slot(const int32_t *prefix, int nslots, int tile)
{
    int lo = 0, hi = nslots;   // prefix[lo] <= tile < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void load16(uint32_t (&dst)[16], const int8_t *src)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = p[i];
        dst[4 * i + 0] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ void load_w8(uint32_t (&dst)[8], const uint8_t *src)
{
    const uint4 a = ld_stream_v4(src), b = ld_stream_v4(src + 16);
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
    dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}

// int32 dots of one 64-group with TC tokens: w = 8 packed words (64 nibbles, u in 0..15),
// act[j] = 16 words of the token's codes in [e0 e2 e4 e6 | e1 e3 e5 e7] runs.  Returns
// sum u*q; the caller subtracts 8*sum(q).
template <int TC>
__device__ __forceinline__ void group_dot(const uint32_t (&w)[8], const uint32_t (&act)[TC][16],
                                          int (&acc)[TC])
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = w[i] & 0x0F0F0F0Fu;
        const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            acc[j] = dp4a_us(lo, act[j][2 * i], acc[j]);
            acc[j] = dp4a_us(hi, act[j][2 * i + 1], acc[j]);
        }
    }
}

struct TileInfo {
    int slot, e, ntok, rb, j0, nt, rowbase;
};

__device__ __forceinline__ TileInfo decode_tile(const FfnPlan *plan, const int32_t *prefix,
                                                int tile, int tc)
{
    TileInfo ti;
    ti.slot = find_slot(prefix, plan->n_slots, tile);
    ti.e = plan->expert[ti.slot];
    ti.ntok = plan->ntok[ti.slot];
    const int nch = (ti.ntok + tc - 1) / tc;
    const int local = tile - prefix[ti.slot];
    ti.rb = local / nch;
    const int ch = local - ti.rb * nch;
    ti.j0 = ch * tc;
    ti.nt = min(tc, ti.ntok - ti.j0);
    ti.rowbase = plan->rowbase[ti.slot] + ti.j0;
    return ti;
}

template <int TC>
__device__ __forceinline__ void row_reduce(float (&v)[TC], int lpr)
{
#pragma unroll
    for (int j = 0; j < TC; ++j)
        for (int off = lpr >> 1; off > 0; off >>= 1) v[j] += __shfl_xor_sync(0xffffffffu, v[j], off);
}

// ----------------------------------------------------------------------------------------
// gate/up + SiLU*up: h[row of (slot, token)][r] for r < F
// ----------------------------------------------------------------------------------------
template <int NG, int TC>
__global__ void __launch_bounds__(kFfnWarps * 32) ffn_gateup_kernel(const FfnArgs a)
{
    const FfnPlan *plan = a.plan;
    const int total = plan->gu_tiles;
    const int H = a.H, G = H / kGroup;
    const int lpr = lanes_per_row(G), rpw = 32 / lpr, ng = (G + lpr - 1) / lpr;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int sub = lane / lpr, gl = lane % lpr;
    const int rows_tile = kFfnWarps * rpw * kRitGu;
    const size_t rowbytes = (size_t)H / 2;
    const bool probe = a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr;

    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile(plan, plan->gu_prefix, tile, TC);
        const bool shared = ti.e < 0;
        const int Fu = shared ? a.Fs : a.F;
        const moe_expert_weights &W = shared ? a.shared : a.routed;
        const size_t erow = shared ? 0 : (size_t)ti.e * Fu;
        const uint8_t *wg = W.w_gate + erow * rowbytes;
        const uint8_t *wu = W.w_up + erow * rowbytes;
        const float *sg = W.s_gate + erow * G;
        const float *su = W.s_up + erow * G;

        // activations of this lane's groups for the tile's tokens
        uint32_t act[NG][TC][16];
        int gsum[NG][TC];
        float sx[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            sx[j] = 0.0f;
            int t = 0;
            if (j < ti.nt) {
                t = shared ? ti.j0 + j : a.tok[plan->tokbase[ti.slot] + ti.j0 + j];
                sx[j] = a.xq.scale[t];
            }
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const int g = gl + k * lpr;
                if (j < ti.nt && k < ng && g < G) {
                    load16(act[k][j], a.xq.q + (size_t)t * H + g * kGroup);
                    gsum[k][j] = a.xq.gsum[(size_t)t * G + g];
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) act[k][j][i] = 0;
                    gsum[k][j] = 0;
                }
            }
        }

        const int r0 = ti.rb * rows_tile + wid * rpw * kRitGu;
#pragma unroll 1
        for (int it = 0; it < kRitGu; ++it) {
            const int r = r0 + it * rpw + sub;
            const bool rv = r < Fu;
            uint32_t wgw[NG][8], wuw[NG][8];
            float sgv[NG], suv[NG];
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const int g = gl + k * lpr;
                if (rv && k < ng && g < G) {
                    load_w8(wgw[k], wg + (size_t)r * rowbytes + g * 32);
                    load_w8(wuw[k], wu + (size_t)r * rowbytes + g * 32);
                    sgv[k] = ld_stream_f32(sg + (size_t)r * G + g);
                    suv[k] = ld_stream_f32(su + (size_t)r * G + g);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) wgw[k][i] = wuw[k][i] = 0u;
                    sgv[k] = suv[k] = 0.0f;
                }
            }
            float accg[TC], accu[TC];
#pragma unroll
            for (int j = 0; j < TC; ++j) accg[j] = accu[j] = 0.0f;
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                int ig[TC], iu[TC];
#pragma unroll
                for (int j = 0; j < TC; ++j) ig[j] = iu[j] = 0;
                group_dot<TC>(wgw[k], act[k], ig);
                group_dot<TC>(wuw[k], act[k], iu);
                const int g = gl + k * lpr;
                const bool gv = rv && k < ng && g < G;
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    ig[j] -= 8 * gsum[k][j];
                    iu[j] -= 8 * gsum[k][j];
                    accg[j] = fmaf(sgv[k], (float)ig[j], accg[j]);
                    accu[j] = fmaf(suv[k], (float)iu[j], accu[j]);
                    if (probe && gv && !shared && j < ti.nt) {
                        const size_t pr = (size_t)(ti.rowbase + j - a.routed_rowbase);
                        const size_t o = (pr * Fu + r) * G + g;
                        if (a.probe.acc_gate) a.probe.acc_gate[o] = ig[j];
                        if (a.probe.acc_up) a.probe.acc_up[o] = iu[j];
                    }
                }
            }
            row_reduce<TC>(accg, lpr);
            row_reduce<TC>(accu, lpr);
            if (gl == 0 && rv) {
#pragma unroll
                for (int j = 0; j < TC; ++j) {
                    if (j < ti.nt) {
                        const float gate = sx[j] * accg[j];
                        const float up = sx[j] * accu[j];
                        const float hval = gate / (1.0f + expf(-gate)) * up;
                        a.h[(size_t)(ti.rowbase + j) * a.hstride + r] = hval;
                    }
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------------------
// down: y[row of (slot, token)][r] for r < H, from h quantised per row at the tile start
// ----------------------------------------------------------------------------------------
template <int NG, int TC>
__global__ void __launch_bounds__(kFfnWarps * 32) ffn_down_kernel(const FfnArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int Fmax = a.hstride;
    int8_t *hq_s = reinterpret_cast<int8_t *>(smem);                          // [TC][Fmax]
    int *hg_s = reinterpret_cast<int *>(smem + (size_t)TC * Fmax);            // [TC][Fmax/64]
    float *hs_s = reinterpret_cast<float *>(hg_s + (size_t)TC * (Fmax / kGroup));  // [TC]

    const FfnPlan *plan = a.plan;
    const int total = plan->dn_tiles;
    const int H = a.H;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const bool probe = a.probe.acc_down != nullptr;
    const bool probe_h = a.probe.hq != nullptr || a.probe.h_scale != nullptr;

    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile(plan, plan->dn_prefix, tile, TC);
        const bool shared = ti.e < 0;
        const int Fu = shared ? a.Fs : a.F;
        const int G = Fu / kGroup;
        const int lpr = lanes_per_row(G), rpw = 32 / lpr, ng = (G + lpr - 1) / lpr;
        const int sub = lane / lpr, gl = lane % lpr;
        const int rows_tile = kFfnWarps * rpw * kRitDn;
        const size_t rowbytes = (size_t)Fu / 2;
        const moe_expert_weights &W = shared ? a.shared : a.routed;
        const size_t erow = shared ? 0 : (size_t)ti.e * H;
        const uint8_t *wd = W.w_down + erow * rowbytes;
        const float *sd = W.s_down + erow * G;

        // 1. quantise the tile's h rows into shared memory: warp j takes token j
        if (wid < ti.nt) {
            const float *hrow = a.h + (size_t)(ti.rowbase + wid) * a.hstride;
            float amax = 0.0f;
            for (int i = lane * 4; i < Fu; i += 128) {
                const float4 v = *reinterpret_cast<const float4 *>(hrow + i);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float inv = quant_inv(amax);
            const int runs = Fu / 8;
            for (int base = 0; base < runs; base += 32) {
                const int run = base + lane;
                int sum = 0;
                if (run < runs) {
                    const float4 v0 = *reinterpret_cast<const float4 *>(hrow + run * 8);
                    const float4 v1 = *reinterpret_cast<const float4 *>(hrow + run * 8 + 4);
                    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                    const uint2 pk = quant_pack8(v, inv, sum);
                    *reinterpret_cast<uint2 *>(hq_s + (size_t)wid * Fmax + run * 8) = pk;
                    if (probe_h && !shared && ti.rb == 0 && a.probe.hq) {
                        const size_t pr = (size_t)(ti.rowbase + wid - a.routed_rowbase);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            a.probe.hq[pr * Fu + run * 8 + i] = (int8_t)quant_code(v[i], inv);
                    }
                }
                // runs of one 64-group are 8 consecutive lanes
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                if ((lane & 7) == 0 && run < runs) hg_s[wid * (Fmax / kGroup) + run / 8] = sum;
            }
            if (lane == 0) {
                hs_s[wid] = quant_scale(amax);
                if (probe_h && !shared && ti.rb == 0 && a.probe.h_scale)
                    a.probe.h_scale[ti.rowbase + wid - a.routed_rowbase] = quant_scale(amax);
            }
        }
        __syncthreads();

        // 2. this lane's groups of the tile's tokens into registers
        uint32_t act[NG][TC][16];
        int gsum[NG][TC];
        float hs[TC];
#pragma unroll
        for (int j = 0; j < TC; ++j) {
            hs[j] = j < ti.nt ? hs_s[j] : 0.0f;
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const int g = gl + k * lpr;
                if (j < ti.nt && k < ng && g < G) {
                    load16(act[k][j], hq_s + (size_t)j * Fmax + g * kGroup);
                    gsum[k][j] = hg_s[j * (Fmax / kGroup) + g];
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) act[k][j][i] = 0;
                    gsum[k][j] = 0;
                }
            }
        }
        __syncthreads();   // shared memory is rewritten by the next tile

        // 3. rows of the down projection
        const int r0 = ti.rb * rows_tile + wid * rpw * kRitDn;
#pragma unroll 1
        for (int it = 0; it < kRitDn; it += kDnUnroll) {
            uint32_t ww[kDnUnroll][NG][8];
            float sv[kDnUnroll][NG];
#pragma unroll
            for (int u = 0; u < kDnUnroll; ++u) {
                const int r = r0 + (it + u) * rpw + sub;
#pragma unroll
                for (int k = 0; k < NG; ++k) {
                    const int g = gl + k * lpr;
                    if (r < H && k < ng && g < G) {
                        load_w8(ww[u][k], wd + (size_t)r * rowbytes + g * 32);
                        sv[u][k] = ld_stream_f32(sd + (size_t)r * G + g);
                    } else {
#pragma unroll
                        for (int i = 0; i < 8; ++i) ww[u][k][i] = 0u;
                        sv[u][k] = 0.0f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kDnUnroll; ++u) {
                const int r = r0 + (it + u) * rpw + sub;
                float acc[TC];
#pragma unroll
                for (int j = 0; j < TC; ++j) acc[j] = 0.0f;
#pragma unroll
                for (int k = 0; k < NG; ++k) {
                    int id[TC];
#pragma unroll
                    for (int j = 0; j < TC; ++j) id[j] = 0;
                    group_dot<TC>(ww[u][k], act[k], id);
                    const int g = gl + k * lpr;
                    const bool gv = r < H && k < ng && g < G;
#pragma unroll
                    for (int j = 0; j < TC; ++j) {
                        id[j] -= 8 * gsum[k][j];
                        acc[j] = fmaf(sv[u][k], (float)id[j], acc[j]);
                        if (probe && gv && !shared && j < ti.nt) {
                            const size_t pr = (size_t)(ti.rowbase + j - a.routed_rowbase);
                            a.probe.acc_down[(pr * H + r) * G + g] = id[j];
                        }
                    }
                }
                row_reduce<TC>(acc, lpr);
                if (gl == 0 && r < H) {
#pragma unroll
                    for (int j = 0; j < TC; ++j)
                        if (j < ti.nt) a.y[(size_t)(ti.rowbase + j) * H + r] = hs[j] * acc[j];
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------------------
// dispatch
// ----------------------------------------------------------------------------------------
typedef void (*FfnKernel)(const FfnArgs);

template <int NG>
FfnKernel pick_gu(int tc)
{
    switch (tc) {
    case 1: return ffn_gateup_kernel<NG, 1>;
    case 2: return ffn_gateup_kernel<NG, 2>;
    case 4: return NG <= 2 ? ffn_gateup_kernel<NG, (NG <= 2 ? 4 : 1)> : nullptr;
    case 8: return NG == 1 ? ffn_gateup_kernel<NG, (NG == 1 ? 8 : 1)> : nullptr;
    }
    return nullptr;
}

template <int NG>
FfnKernel pick_dn(int tc)
{
    switch (tc) {
    case 1: return ffn_down_kernel<NG, 1>;
    case 2: return ffn_down_kernel<NG, 2>;
    case 4: return NG <= 2 ? ffn_down_kernel<NG, (NG <= 2 ? 4 : 1)> : nullptr;
    case 8: return NG == 1 ? ffn_down_kernel<NG, (NG == 1 ? 8 : 1)> : nullptr;
    }
    return nullptr;
}

FfnKernel gu_kernel(int ng, int tc)
{
    switch (ng) {
    case 1: return pick_gu<1>(tc);
    case 2: return pick_gu<2>(tc);
    case 3: return pick_gu<3>(tc);
    case 4: return pick_gu<4>(tc);
    }
    return nullptr;
}

FfnKernel dn_kernel(int ng, int tc)
{
    switch (ng) {
    case 1: return pick_dn<1>(tc);
    case 2: return pick_dn<2>(tc);
    case 3: return pick_dn<3>(tc);
    case 4: return pick_dn<4>(tc);
    }
    return nullptr;
}

int grid_for(FfnKernel k, size_t smem)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kFfnWarps * 32, smem) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    return per_sm * num_sms();
}

}  // namespace

int groups_per_lane(int n)
{
    const int g = n / kGroup;
    const int l = lanes_per_row(g);
    return (g + l - 1) / l;
}

int choose_tc(int ng, double tokens_per_expert)
{
    const int tcmax = ng == 1 ? 8 : (ng == 2 ? 4 : 2);
    int tc = 1;
    while (tc < tcmax && tc < tokens_per_expert) tc *= 2;
    return tc;
}

size_t down_smem_bytes(int tc, int fmax)
{
    return (size_t)tc * fmax + (size_t)tc * (fmax / kGroup) * 4 + (size_t)tc * 4;
}

namespace {

int down_ng(const FfnArgs &a)
{
    int ng = groups_per_lane(a.F);
    if (a.n_shared && groups_per_lane(a.Fs) > ng) ng = groups_per_lane(a.Fs);
    return ng;
}

}  // namespace

cudaError_t launch_ffn_gate_up(const FfnArgs &a, cudaStream_t st)
{
    FfnKernel gu = gu_kernel(groups_per_lane(a.H), a.tc_gu);
    if (!gu) return cudaErrorInvalidConfiguration;
    gu<<<grid_for(gu, 0), kFfnWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ffn_down(const FfnArgs &a, cudaStream_t st)
{
    FfnKernel dn = dn_kernel(down_ng(a), a.tc_dn);
    if (!dn) return cudaErrorInvalidConfiguration;
    const size_t smem = down_smem_bytes(a.tc_dn, a.hstride);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(dn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    dn<<<grid_for(dn, smem), kFfnWarps * 32, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
