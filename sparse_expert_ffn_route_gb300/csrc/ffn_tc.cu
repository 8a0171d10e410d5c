// ffn_tc.cu -- grouped expert FFN on the tcgen05 tensor cores, for experts that receive
// many tokens (prefill-sized batches) ["MoE 路由与专家流式加载" §1.3; "colibri 开发演进实录"
// §2.2 K1b: an integer dot per 64-group, then the group scale].
//
// The contraction is exact integer arithmetic carried in bf16: a weight code minus its
// zero point (u - 8, in [-8, 7]) and an activation code (in [-127, 127]) are both exact in
// bf16, their products are exact in fp32, and so is a 64-term group sum (|sum| <= 65024).
// Each group is one MMA chain of its own (4 x K16) into a TMEM accumulator, so the integer
// group sums A[row][token] come out exactly, and the epilogue applies the group scale:
// acc += s[row][g] * A.  The token's activation scale multiplies at the end.
//
// Tile: 128 weight rows (one matrix of one expert) x up to 128 tokens of the expert's list;
// one task per tile, all K groups.  Warp roles in a CTA of 9 warps:
//   warps 0-3  one weight row each per thread: load the row's nibbles of the next groups
//              from HBM (16-byte non-allocating loads, 8 groups ahead in registers),
//              convert them to bf16 (u - 8) and store them into the group's A buffer in
//              TMEM; copy the B tile (the tile's token rows of the bf16 activation codes,
//              128 bytes per row per group) into a 128-byte-swizzled shared-memory stage
//              with cp.async, kPre groups ahead.
//   warp 4     allocates TMEM; one thread issues the 4 MMAs of each group
//              (A from TMEM, B from shared memory) and commits them to mbarriers.
//   warps 5-8  the epilogue: per group, the accumulator (32 TMEM lanes = 32 rows each) is
//              loaded 32 columns at a time and added into registers with the group scale.
// A groups' stages rotate through kStages A buffers / B stages and 2 accumulators.  Every
// wait is bounded; a timeout sets the error word, and every role leaves its loops.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "ffn_tiles.cuh"
#include "launch.cuh"
#include "moe_internal.cuh"
#include "tcgen05.cuh"

namespace moe {

namespace {

constexpr int kM = 128;             // weight rows per tile (MMA M)
constexpr int kN = 128;             // tokens per tile, at most (MMA N)
constexpr int kGK = 64;             // inputs per group (one scale; 4 MMAs of K = 16)
constexpr int kStages = 6;          // A buffers (TMEM) and B stages (shared memory)
constexpr int kPre = kStages - 2;   // B copies run this many groups ahead
constexpr int kNibAhead = 8;        // groups of nibbles held in registers ahead of use
constexpr int kThreads = 9 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;                  // 2 accumulators of kN columns
constexpr uint32_t kColA = 2 * kN;             // kStages A buffers of 32 columns (64 bf16)
constexpr int kBStageBytes = kN * 128;         // 16 KB, 1024-byte aligned
constexpr int kSmemBytes = kStages * kBStageBytes + 128 * 16 * 4 /* epilogue scales */ +
                           1024 /* alignment */ + 256 /* barriers */;

static_assert(kColA + kStages * 32 <= kTmemCols, "TMEM budget");

struct TcTask {
    int slot, e, sh, m, r0, j0, nt, np, rowbase, tokbase, ngroups;
    const uint8_t *w;    // first nibble byte of row r0 of matrix m
    const float *s;      // first scale of row r0
    int rowbytes, G;
};

// task = (slot, token chunk of kN, matrix, block of 128 rows), numbered like the GEMV tasks
// (geo: rb = 128, S = matrices, tc = kN)
template <bool GU>
__device__ __forceinline__ TcTask tc_task(const FfnArgs &a, int task)
{
    const FfnPlan *plan = a.plan;
    const int32_t *prefix = GU ? plan->gu_prefix : plan->dn_prefix;
    int lo = 0, hi = plan->n_slots;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= task) lo = mid;
        else hi = mid;
    }
    TcTask t;
    t.slot = lo;
    t.e = plan->expert[lo];
    t.sh = t.e < 0 ? 1 : 0;
    const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
    const int nblk = g.nrows / kM;
    const int local = task - prefix[lo];
    const int cs = local / nblk, blk = local - cs * nblk;
    const int ch = cs / g.S;
    t.m = cs - ch * g.S;
    t.r0 = blk * kM;
    t.j0 = ch * kN;
    const int ntok = plan->ntok[lo];
    t.nt = min(kN, ntok - t.j0);
    t.np = (t.nt + 15) & ~15;
    t.rowbase = plan->rowbase[lo] + t.j0;
    t.tokbase = plan->tokbase[lo];
    t.ngroups = g.kdim / kGK;
    t.rowbytes = g.rowbytes;
    t.G = g.G;
    const moe_expert_weights &W = t.sh ? a.shared : a.routed;
    const size_t erow = t.sh ? 0 : (size_t)t.e * g.nrows;
    const uint8_t *wm = GU ? (t.m == 0 ? W.w_gate : W.w_up) : W.w_down;
    const float *sm = GU ? (t.m == 0 ? W.s_gate : W.s_up) : W.s_down;
    t.w = wm + (erow + t.r0) * g.rowbytes;
    t.s = sm + (erow + t.r0) * g.G;
    return t;
}

struct TcShared {
    uint64_t full[kStages];    // A stored + B landed (128 converter threads)
    uint64_t sfree[kStages];   // the group's MMAs are done with A buffer / B stage
    uint64_t dfull[2];         // accumulator ready (MMA commit)
    uint64_t dempty[2];        // accumulator read (128 epilogue threads)
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool aborted(const TcShared *sh) { return *(volatile const int *)&sh->abort != 0; }

// bounded wait; on timeout the block is told to stop and the error word is set
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, TcShared *sh, int32_t *err)
{
    if (mbar_wait(bar, parity)) return true;
    atomicOr(err, kErrTimeout);
    atomicExch(&sh->abort, 1);
    return false;
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t *>(&v); }

// 8 nibbles (elements 8c .. 8c+7: element 2b in the low nibble of byte b, 2b+1 in the high)
// -> 4 words of bf16 pairs holding u - 8, element order
__device__ __forceinline__ void nibbles_to_bf16(uint32_t w, uint32_t *out)
{
    const uint32_t L = w & 0x0F0F0F0Fu, Hh = (w >> 4) & 0x0F0F0F0Fu;
    const uint32_t p01 = __byte_perm(L, Hh, 0x5140);   // lo0 hi0 lo1 hi1
    const uint32_t p23 = __byte_perm(L, Hh, 0x7362);   // lo2 hi2 lo3 hi3
    constexpr uint32_t C = 0x43434343u;                // bf16 0x43XX = 128 + XX for XX < 128
    const uint32_t t[4] = {__byte_perm(p01, C, 0x4140), __byte_perm(p01, C, 0x4342),
                           __byte_perm(p23, C, 0x4140), __byte_perm(p23, C, 0x4342)};
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&t[i]);
        out[i] = bf16x2_bits(__hsub2(v, k136));   // (128 + u) - 136 = u - 8, exact
    }
}

template <bool GU, bool PROBE>
__global__ void __launch_bounds__(kThreads, 1) ffn_tc_kernel(const __grid_constant__ FfnArgs a)
{
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    pdl_wait();
    pdl_launch_dependents();
    // B stages on a 1024-byte boundary (128-byte swizzle atoms), then the control block
    uint8_t *bstage = reinterpret_cast<uint8_t *>(((uintptr_t)tc_smem_raw + 1023) & ~(uintptr_t)1023);
    float *escl = reinterpret_cast<float *>(bstage + kStages * kBStageBytes);   // [128][2][8]
    TcShared *sh = reinterpret_cast<TcShared *>(escl + 128 * 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = GU ? a.plan->gu_tiles : a.plan->dn_tiles;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh->full[i], 128);
            mbar_init(&sh->sfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sh->dfull[i], 1);
            mbar_init(&sh->dempty[i], 128);
        }
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == 4) {
        tc::tmem_alloc(&sh->tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh->tmem;

    if (warp < 4) {
        // ---------------- converters / loaders: thread i owns weight row r0 + i ----------
        const int i = tid;
        const __nv_bfloat16 *act = GU ? a.x_bf16 : a.h_bf16;
        const int act_ld = GU ? a.H : a.hstride;
        // B-copy cursor (kPre groups ahead of the conversion cursor)
        int ptask = blockIdx.x, pg = 0;
        TcTask pt;
        if (ptask < total) pt = tc_task<GU>(a, ptask);
        long long pit = 0;   // global group index of the B copy cursor
        auto issue_b = [&]() {
            // copy B of (ptask, pg) into stage pit % kStages
            if (ptask < total) {
                const int st = (int)(pit % kStages);
                if (pit >= kStages &&
                    !tc_wait(&sh->sfree[st], (uint32_t)((pit / kStages - 1) & 1), sh, a.err))
                    return;
                uint8_t *dst = bstage + st * kBStageBytes;
                const bool valid = i < pt.nt;
                int row = 0;
                if (valid) {
                    if (GU) row = pt.sh ? pt.j0 + i : a.tok[pt.tokbase + pt.j0 + i];
                    else row = pt.rowbase + i;
                }
                const __nv_bfloat16 *s = act + (size_t)row * act_ld + pg * kGK;
                if (i < pt.np) {
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        cp_async16(dst + (i >> 3) * 1024 + (i & 7) * 128 + ((c ^ (i & 7)) << 4),
                                   s + c * 8, valid);
                }
                if (++pg == pt.ngroups) {
                    pg = 0;
                    ptask += gridDim.x;
                    if (ptask < total) pt = tc_task<GU>(a, ptask);
                }
                ++pit;
            }
        };
        for (int k = 0; k < kPre; ++k) {
            issue_b();
            cp_async_commit();
        }
        long long it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, task);
            const uint8_t *wrow = t.w + (size_t)i * t.rowbytes;
            // nibbles of the next kNibAhead groups in registers (2 x 16 bytes per group)
            uint4 nib[kNibAhead][2];
#pragma unroll
            for (int q = 0; q < kNibAhead; ++q) {
                if (q < t.ngroups) {
                    nib[q][0] = ld_stream_v4(wrow + q * 32);
                    nib[q][1] = ld_stream_v4(wrow + q * 32 + 16);
                }
            }
            for (int g0 = 0; g0 < t.ngroups && !aborted(sh); g0 += kNibAhead) {
#pragma unroll
                for (int q = 0; q < kNibAhead; ++q) {
                    const int g = g0 + q;
                    if (g >= t.ngroups || aborted(sh)) break;
                    const int st = (int)(it % kStages);
                    // the B copy kPre groups ahead; its stage was freed by the MMA of an
                    // earlier group, which also freed this group's A buffer
                    issue_b();
                    cp_async_commit();
                    if (it >= kStages &&
                        !tc_wait(&sh->sfree[st], (uint32_t)((it / kStages - 1) & 1), sh, a.err))
                        break;
                    uint32_t av[32];
                    const uint32_t wv[8] = {nib[q][0].x, nib[q][0].y, nib[q][0].z, nib[q][0].w,
                                            nib[q][1].x, nib[q][1].y, nib[q][1].z, nib[q][1].w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) nibbles_to_bf16(wv[c], av + 4 * c);
                    // refill this register slot with the group kNibAhead further on
                    if (g + kNibAhead < t.ngroups) {
                        nib[q][0] = ld_stream_v4(wrow + (g + kNibAhead) * 32);
                        nib[q][1] = ld_stream_v4(wrow + (g + kNibAhead) * 32 + 16);
                    }
                    tc::st32(tmem + ((uint32_t)(warp * 32) << 16) + kColA + st * 32, av);
                    tc::wait_st();
                    cp_async_wait<kPre>();          // this group's B rows have landed
                    tc::fence_proxy_async_smem();   // ... and are visible to the MMA
                    tc::fence_before_sync();
                    mbar_arrive(&sh->full[st]);
                    ++it;
                }
            }
        }
        cp_async_wait<0>();
    } else if (warp == 4) {
        // ---------------- MMA issue ---------------------------------------------------
        long long it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, task);
            const uint32_t idesc = tc::idesc_bf16_f32(kM, t.np);
            for (int g = 0; g < t.ngroups && !aborted(sh); ++g, ++it) {
                const int st = (int)(it % kStages), buf = (int)(it & 1);
                bool ok = true;
                if (lane == 0) {
                    ok = tc_wait(&sh->full[st], (uint32_t)((it / kStages) & 1), sh, a.err);
                    if (ok && it >= 2) ok = tc_wait(&sh->dempty[buf], (uint32_t)((it / 2 - 1) & 1), sh, a.err);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint32_t bsaddr = smem_u32(bstage + st * kBStageBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_ts(tmem + kColD + buf * kN, tmem + kColA + st * 32 + kk * 8,
                                   tc::sdesc_kmajor_sw128(bsaddr + kk * 32), idesc, kk > 0);
                    tc::commit(&sh->sfree[st]);
                    tc::commit(&sh->dfull[buf]);
                }
                __syncwarp();
            }
        }
    } else {
        // ---------------- epilogue: warp q reads TMEM lanes 32q .. 32q+31 = rows ------
        const int q = warp & 3;
        const int i = q * 32 + lane;   // row within the tile
        const QuantRows &src = GU ? a.xq : a.hq;
        long long it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, task);
            cp_async_wait<0>();   // the last task's scale copies (none pending otherwise)
            float acc[kN];
#pragma unroll
            for (int j = 0; j < kN; ++j) acc[j] = 0.0f;
            // the row's group scales, copied 8 at a time into this thread's two shared slots,
            // one block of 8 ahead (G is a multiple of 8)
            const float *srow = t.s + (size_t)i * t.G;
            float *myscl = escl + (size_t)i * 16;
            cp_async16(myscl, srow, true);
            cp_async16(myscl + 4, srow + 4, true);
            cp_async_commit();
            for (int g = 0; g < t.ngroups; ++g, ++it) {
                const int gi = g & 7;
                if (gi == 0) {
                    const int nb = g + 8;
                    float *nxt = myscl + ((nb >> 3) & 1) * 8;
                    if (nb < t.ngroups) {
                        cp_async16(nxt, srow + nb, true);
                        cp_async16(nxt + 4, srow + nb + 4, true);
                    }
                    cp_async_commit();
                    cp_async_wait<1>();   // this block's 8 scales have landed
                }
                const float scl = myscl[((g >> 3) & 1) * 8 + gi];
                const int buf = (int)(it & 1);
                if (!tc_wait(&sh->dfull[buf], (uint32_t)((it / 2) & 1), sh, a.err)) break;
                tc::fence_after_sync();
#pragma unroll
                for (int c = 0; c < kN / 16; ++c) {
                    if (c * 16 < t.np) {
                        uint32_t r[16];
                        tc::ld16(tmem + ((uint32_t)(q * 32) << 16) + kColD + buf * kN + c * 16, r);
                        tc::wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float d = __uint_as_float(r[j]);
                            acc[c * 16 + j] = fmaf(scl, d, acc[c * 16 + j]);
                            if (PROBE) {
                                const int jj = c * 16 + j;
                                if (jj < t.nt && t.sh == 0) {
                                    const size_t pr = (size_t)(t.rowbase + jj - a.routed_rowbase);
                                    const size_t o = (pr * (size_t)(GU ? a.F : a.H) + t.r0 + i) * t.G + g;
                                    int32_t *dst = GU ? (t.m == 0 ? a.probe.acc_gate : a.probe.acc_up)
                                                      : a.probe.acc_down;
                                    if (dst) dst[o] = (int32_t)d;   // an exact integer
                                }
                            }
                        }
                    }
                }
                tc::fence_before_sync();
                mbar_arrive(&sh->dempty[buf]);
            }
            if (aborted(sh)) break;
            // outputs: token scale x accumulated row value
            float *dst;
            int ld;
            if (GU) {
                dst = t.m == 0 ? a.gpart : a.upart;
                ld = a.hstride;
            } else {
                dst = a.y;
                ld = a.H;
            }
#pragma unroll
            for (int j = 0; j < kN; ++j) {
                if (j < t.nt) {
                    const int arow = GU ? (t.sh ? t.j0 + j : a.tok[t.tokbase + t.j0 + j]) : t.rowbase + j;
                    dst[(size_t)(t.rowbase + j) * ld + t.r0 + i] = src.scale[arow] * acc[j];
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 4) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool ffn_tc_supported(const FfnArgs &a)
{
    // every matrix of the call: rows in whole 128-row tiles, and reductions in whole blocks
    // of 8 groups (the epilogue copies a row's scales 8 at a time, 32-byte aligned)
    const bool sh = a.n_shared != 0;
    if (a.F % 512 || a.H % 512) return false;
    if (sh && a.Fs % 512) return false;
    return true;
}

size_t ffn_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_ffn_tc(bool gu, const FfnArgs &a, cudaStream_t st)
{
    const bool probe = gu ? (a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr)
                          : a.probe.acc_down != nullptr;
    const dim3 grid(num_sms()), block(kThreads);
    if (gu)
        return probe ? launch_kernel(ffn_tc_kernel<true, true>, grid, block, kSmemBytes, st, 1, a)
                     : launch_kernel(ffn_tc_kernel<true, false>, grid, block, kSmemBytes, st, 1, a);
    return probe ? launch_kernel(ffn_tc_kernel<false, true>, grid, block, kSmemBytes, st, 1, a)
                 : launch_kernel(ffn_tc_kernel<false, false>, grid, block, kSmemBytes, st, 1, a);
}

}  // namespace moe
