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
// one task per tile, all K groups.  Warp roles in a CTA of 16 warps:
//   warps 0-3  one weight row each per thread: take the row's nibbles of a group from the
//              nibble stages in shared memory, convert them to bf16 (u - 8) and store them
//              into the group's A buffer in TMEM.
//   warp 4     allocates TMEM; one thread issues the 4 MMAs of each group (A from TMEM, B
//              from shared memory) and commits them to the rings' mbarriers.
//   warp 5     loads the B tiles: the tile's activation rows (bf16 codes, laid out in
//              output-row order, 128 bytes per row per group) by 2-D TMA with the 128-byte
//              swizzle, one box per power-of-two part of the tile's height (a TMA instruction
//              costs the issuing warp hundreds of cycles, so boxes are as large as the tile
//              allows), into a ring of kBStages shared-memory stages.
//   warps 6-13 the epilogue, two warps per 32 TMEM lanes (32 rows), 64 token columns each:
//              per group the accumulator is loaded 16 columns at a time (the next load in
//              flight) and added into registers with the group scale (packed fp32x2 FMAs).
//   warp 14    loads the weight nibbles by 2-D TMA, 4 groups of the tile's 128 rows per box
//              (16 KB, 128-byte swizzle), into a ring of kNStages stages, so the converters
//              never wait on a global load (held in registers, as an earlier version did,
//              a few groups ahead did not cover the memory latency under load).
//   warp 15    idle (the block stays whole warpgroups at 128 registers a thread).
// Groups rotate through kAStages A buffers, kBStages B stages and kDBuf accumulators, each
// ring with a full and an empty mbarrier; warps arrive once each.  Within every run of 8
// inputs the contraction runs in the order e0 e4 e1 e5 e2 e6 e3 e7 on both operands (the
// order in which nibbles unpack cheapest); a group sum does not depend on it.  Every wait is
// bounded; a timeout sets the error word, and every role leaves its loops.
#include <cuda.h>           // CUtensorMap and its enums (types only: the encoder is looked up)
#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

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
constexpr int kAStages = 4;         // A buffers in TMEM
constexpr int kBStages = 8;         // B stages in shared memory
constexpr int kDBuf = 3;            // accumulators in TMEM
constexpr int kNStages = 3;         // nibble stages in shared memory (TMA-fed)
constexpr int kNGroups = 4;         // groups per nibble stage: [128 rows][128 B], 16 KB
constexpr int kBoxMaps = 4;         // B tensor maps with boxes of 16, 32, 64 and 128 rows
constexpr int kWarpMma = 4, kWarpTma = 5, kWarpEpi0 = 6, kWarpNib = 14;
constexpr int kEpiWarps = 8;        // two per TMEM lane quarter, 64 token columns each
// warps 0-3 converters, 4 MMA, 5 B loads, 6-13 epilogue, 14 nibble loads, 15 idle (whole
// warpgroups keep the launch at 128 registers a thread)
constexpr int kThreads = 16 * 32;
static_assert(kWarpNib == kWarpEpi0 + kEpiWarps, "warp layout");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD = 0;                  // kDBuf accumulators of kN columns
constexpr uint32_t kColA = kDBuf * kN;         // kAStages A buffers of 32 columns (64 bf16)
constexpr int kBStageBytes = kN * 128;         // 16 KB, 1024-byte aligned
constexpr int kNStageBytes = kM * 128;         // 16 KB: 4 groups of 128 rows' nibbles
constexpr int kSclFloats = kEpiWarps * 32 * 16;   // the epilogue's scale slots

static_assert(kColA + kAStages * 32 <= kTmemCols, "TMEM budget");


struct TcTask {
    int slot, e, sh, m, r0, j0, nt, np, rowbase, tokbase, ngroups;
    const uint8_t *w;    // first nibble byte of row r0 of matrix m
    const float *s;      // first scale of row r0
    int rowbytes, G;
};

// the plan's per-slot arrays, copied into shared memory once per CTA
struct PlanSmem {
    int n_slots;
    int32_t prefix[kMaxSlots + 1], expert[kMaxSlots], ntok[kMaxSlots], tokbase[kMaxSlots],
        rowbase[kMaxSlots];
};

// task = (slot, token chunk of kN, matrix, block of 128 rows), numbered like the GEMV tasks
// (geo: rb = 128, S = matrices, tc = kN)
template <bool GU>
__device__ __forceinline__ TcTask tc_task(const FfnArgs &a, const PlanSmem &ps, int task)
{
    int lo = 0, hi = ps.n_slots;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ps.prefix[mid] <= task) lo = mid;
        else hi = mid;
    }
    TcTask t;
    t.slot = lo;
    t.e = ps.expert[lo];
    t.sh = t.e < 0 ? 1 : 0;
    const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
    const int nblk = g.nrows / kM;
    const int local = task - ps.prefix[lo];
    const int cs = local / nblk, blk = local - cs * nblk;
    const int ch = cs / g.S;
    t.m = cs - ch * g.S;
    t.r0 = blk * kM;
    t.j0 = ch * kN;
    const int ntok = ps.ntok[lo];
    t.nt = min(kN, ntok - t.j0);
    t.np = (t.nt + 15) & ~15;
    t.rowbase = ps.rowbase[lo] + t.j0;
    t.tokbase = ps.tokbase[lo];
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
    uint64_t afull[kAStages];    // A buffer stored (one arrival per converter warp)
    uint64_t aempty[kAStages];   // the MMAs that read the A buffer are done (commit)
    uint64_t bfull[kBStages];    // B stage landed (TMA transaction bytes)
    uint64_t bempty[kBStages];   // the MMAs that read the B stage are done (commit)
    uint64_t dfull[kDBuf];       // accumulator ready (commit)
    uint64_t dempty[kDBuf];      // accumulator read (one arrival per epilogue warp)
    uint64_t nfull[kNStages];    // nibble stage landed (TMA transaction bytes)
    uint64_t nempty[kNStages];   // nibble stage converted (one arrival per converter warp)
    uint64_t mfinal;             // every MMA of the CTA is done (commit before TMEM is freed)
    uint32_t tmem;
    int abort;
};

constexpr int kSmemBytes = 1024 /* alignment */ + kBStages * kBStageBytes + kNStages * kNStageBytes + kSclFloats * 4 +
                           (int)((sizeof(TcShared) + 15) / 16 * 16) + (int)sizeof(PlanSmem);

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

// 8 nibbles (elements 8c .. 8c+7 of a row; element n in bits 4n .. 4n+3) -> 4 words of
// bf16 pairs holding u - 8: word k = (element k, element k + 4), the low half first
__device__ __forceinline__ void nibbles_to_bf16(uint32_t w, uint32_t *out)
{
    const __nv_bfloat162 k136 = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        // bf16 0x43XX = 128 + XX for XX < 128: both nibbles become 128 + u
        const uint32_t t = ((w >> (4 * k)) & 0x000F000Fu) | 0x43004300u;
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&t);
        out[k] = bf16x2_bits(__hsub2(v, k136));   // (128 + u) - 136 = u - 8, exact
    }
}

// acc += (s, s) * (d0, d1) as one packed fp32x2 FMA (each lane rounded like fmaf)
__device__ __forceinline__ void ffma2(float2 &acc, float2 s2, uint32_t d0, uint32_t d1)
{
    acc = __ffma2_rn(s2, make_float2(__uint_as_float(d0), __uint_as_float(d1)), acc);
}

// 2-D tiled TMA load of one box into shared memory, completing as transaction bytes on bar;
// executed by a converged warp, issued by one elected lane
__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// mbarrier arrival with an expected transaction count, by one elected lane of a converged warp
__device__ __forceinline__ void arrive_expect_tx_elect(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
        : "memory");
}

// bounded wait by every lane of a converged warp; false (for all lanes) if any lane gave up
__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, uint32_t parity, TcShared *sh, int32_t *err)
{
    return __all_sync(0xffffffffu, tc_wait(bar, parity, sh, err));
}

// the B operand's tensor maps: map k has boxes of 64 columns x (16 << k) rows
struct BMaps {
    CUtensorMap m[kBoxMaps];
    // nibbles of [routed, shared][matrix] as [rows][row bytes] u8, boxes of 128 B x 128 rows
    // (128-byte swizzle); matrix 0 / 1 = gate / up for gate/up, 0 = down for down
    CUtensorMap nib[2][2];
};

template <bool GU, bool PROBE>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_tc_kernel(const __grid_constant__ FfnArgs a, const __grid_constant__ BMaps bmaps)
{
    extern __shared__ __align__(1024) uint8_t tc_smem_raw[];
    pdl_wait();
    pdl_launch_dependents();
    // B stages and nibble stages on 1024-byte boundaries (128-byte swizzle atoms), the
    // epilogue's scale slots, the control block, the plan
    uint8_t *bstage = reinterpret_cast<uint8_t *>(((uintptr_t)tc_smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *nstage = bstage + kBStages * kBStageBytes;
    float *escl = reinterpret_cast<float *>(nstage + kNStages * kNStageBytes);
    TcShared *sh = reinterpret_cast<TcShared *>(escl + kSclFloats);
    PlanSmem *ps = reinterpret_cast<PlanSmem *>(reinterpret_cast<uint8_t *>(sh) +
                                                (sizeof(TcShared) + 15) / 16 * 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = GU ? a.plan->gu_tiles : a.plan->dn_tiles;
    {
        const FfnPlan *plan = a.plan;
        const int ns = plan->n_slots;
        const int32_t *pre = GU ? plan->gu_prefix : plan->dn_prefix;
        if (tid == 0) ps->n_slots = ns;
        for (int k = tid; k <= ns; k += blockDim.x) {
            ps->prefix[k] = pre[k];
            if (k < ns) {
                ps->expert[k] = plan->expert[k];
                ps->ntok[k] = plan->ntok[k];
                ps->tokbase[k] = plan->tokbase[k];
                ps->rowbase[k] = plan->rowbase[k];
            }
        }
    }

    if (tid == 0) {
        for (int i = 0; i < kAStages; ++i) {
            mbar_init(&sh->afull[i], 4);
            mbar_init(&sh->aempty[i], 1);
        }
        for (int i = 0; i < kBStages; ++i) {
            mbar_init(&sh->bfull[i], 1);
            mbar_init(&sh->bempty[i], 1);
        }
        for (int i = 0; i < kDBuf; ++i) {
            mbar_init(&sh->dfull[i], 1);
            mbar_init(&sh->dempty[i], kEpiWarps);
        }
        for (int i = 0; i < kNStages; ++i) {
            mbar_init(&sh->nfull[i], 1);
            mbar_init(&sh->nempty[i], 4);
        }
        mbar_init(&sh->mfinal, 1);
        sh->abort = 0;
        fence_mbar_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(&sh->tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh->tmem;

    if (warp < 4) {
        // ---------------- converters: thread i owns weight row r0 + i; the nibbles come from
        // the nibble stages (4 groups each, 128-byte swizzle: 16-byte chunk c of row i sits at
        // chunk c ^ (i & 7) of its 128-byte line) ----------------------------------------------
        const int i = tid;
        const uint32_t arow = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t it = 0;   // groups of this CTA so far
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const int ng = tc_task<GU>(a, *ps, task).ngroups;
            bool ok = true;
            for (int g = 0; g < ng; ++g, ++it) {
                const uint32_t n = it / kNGroups, gi = it % kNGroups, ns = n % kNStages;
                if (gi == 0 && !(ok = tc_wait_warp(&sh->nfull[ns], (n / kNStages) & 1, sh, a.err))) break;
                const uint8_t *line = nstage + ns * kNStageBytes + i * 128;
                const uint4 w0 = *reinterpret_cast<const uint4 *>(line + (((2 * gi) ^ (i & 7)) << 4));
                const uint4 w1 = *reinterpret_cast<const uint4 *>(line + (((2 * gi + 1) ^ (i & 7)) << 4));
                if (gi == kNGroups - 1) {
                    // the stage is in registers: hand it back to the nibble loads (the reads
                    // are ordered before the next TMA write into it, another proxy)
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh->nempty[ns]);
                }
                const uint32_t st = it % kAStages;
                // this A buffer was last read by the MMAs of group it - kAStages
                if (it >= kAStages) {
                    if (!(ok = tc_wait_warp(&sh->aempty[st], ((it / kAStages) - 1) & 1, sh, a.err))) break;
                    tc::fence_after_sync();
                }
                uint32_t av[32];
                const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) nibbles_to_bf16(wv[c], av + 4 * c);
                tc::st32(arow + kColA + st * 32, av);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh->afull[st]);
            }
            if (!ok) break;
        }
    } else if (warp == kWarpNib) {
        // ---------------- nibble stages by TMA: 4 groups of the tile's 128 rows per box -----
        const uint32_t ns0 = smem_u32(nstage);
        uint32_t n = 0;   // stages of this CTA so far
        bool ok = true;
        for (int task = blockIdx.x; task < total && ok && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, *ps, task);
            const Geo &geo = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
            const int y = (t.sh ? 0 : t.e * geo.nrows) + t.r0;
            const CUtensorMap *map = &bmaps.nib[t.sh][GU ? t.m : 0];
            for (int j = 0; j < t.ngroups / kNGroups && !aborted(sh); ++j, ++n) {
                const uint32_t s = n % kNStages;
                if (n >= kNStages && !(ok = tc_wait_warp(&sh->nempty[s], ((n / kNStages) - 1) & 1, sh, a.err)))
                    break;
                const uint32_t full = smem_u32(&sh->nfull[s]);
                arrive_expect_tx_elect(full, kNStageBytes);
                tma_load_2d_elect(ns0 + s * kNStageBytes, map, j * kNGroups * 32, y, full);
            }
        }
        // copies still in flight (after a timeout elsewhere) land before the CTA exits
        for (uint32_t j = n > (uint32_t)kNStages ? n - kNStages : 0; j < n; ++j)
            mbar_wait(&sh->nfull[j % kNStages], (j / kNStages) & 1);
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ---------------- MMA issue: the whole warp runs the loop, one lane issues ----------
        const uint64_t bdesc0 = tc::sdesc_kmajor_sw128(smem_u32(bstage));
        uint32_t it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, *ps, task);
            const uint32_t idesc = tc::idesc_bf16_f32(kM, t.np);
            for (int g = 0; g < t.ngroups && !aborted(sh); ++g, ++it) {
                const uint32_t sa = it % kAStages, sb = it % kBStages, buf = it % kDBuf;
                if (!tc_wait_warp(&sh->afull[sa], (it / kAStages) & 1, sh, a.err) ||
                    !tc_wait_warp(&sh->bfull[sb], (it / kBStages) & 1, sh, a.err) ||
                    (it >= kDBuf && !tc_wait_warp(&sh->dempty[buf], ((it / kDBuf) - 1) & 1, sh, a.err)))
                    break;
                tc::fence_after_sync();
                // B descriptor: the stage's start address advanced 32 bytes per K step of 16
                const uint64_t bd = bdesc0 + (uint64_t)((sb * kBStageBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_ts_elect(tmem + kColD + buf * kN, tmem + kColA + sa * 32 + kk * 8,
                                     bd + (uint64_t)(kk * 2), idesc, kk > 0);
                tc::commit_elect(&sh->aempty[sa]);
                tc::commit_elect(&sh->bempty[sb]);
                tc::commit_elect(&sh->dfull[buf]);
            }
        }
        // every MMA issued here completes before TMEM is freed
        tc::commit_elect(&sh->mfinal);
        tc_wait_warp(&sh->mfinal, 0, sh, a.err);
    } else if (warp == kWarpTma) {
        // ---------------- B tiles by TMA: the whole warp runs the loop, one lane issues -----
        const uint32_t bs0 = smem_u32(bstage);
        uint32_t it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, *ps, task);
            const uint32_t bytes = (uint32_t)t.np * 128u;
            bool ok = true;
            for (int g = 0; g < t.ngroups && !aborted(sh); ++g, ++it) {
                const uint32_t sb = it % kBStages;
                if (it >= kBStages && !(ok = tc_wait_warp(&sh->bempty[sb], ((it / kBStages) - 1) & 1, sh, a.err)))
                    break;
                const uint32_t full = smem_u32(&sh->bfull[sb]);
                arrive_expect_tx_elect(full, bytes);
                // rows rowbase .. rowbase + np - 1 of the activation codes (rows past nt feed
                // only the padding columns of the accumulator): np (a multiple of 16, at most
                // 128) as a sum of boxes of 128, 64, 32 and 16 rows, largest first
                int r = 0;
#pragma unroll
                for (int k = kBoxMaps - 1; k >= 0; --k) {
                    if (t.np - r >= (16 << k)) {
                        tma_load_2d_elect(bs0 + sb * kBStageBytes + r * 128, &bmaps.m[k], g * kGK, t.rowbase + r, full);
                        r += 16 << k;
                    }
                }
            }
            if (!ok) break;
        }
        // copies still in flight (after a timeout elsewhere) land before the CTA exits
        for (uint32_t j = it > (uint32_t)kBStages ? it - kBStages : 0; j < it; ++j)
            mbar_wait(&sh->bfull[j % kBStages], (j / kBStages) & 1);
        __syncwarp();
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + kEpiWarps) {
        // ---------------- epilogue: warp reads TMEM lanes 32q .. 32q+31 (rows), token
        // columns 64h .. 64h+63 ----------------------------------------------------------
        const int q = warp & 3, half = (warp - kWarpEpi0) >> 2;
        const int i = q * 32 + lane;   // row within the tile
        const int c0 = half * 64;      // first token column
        const QuantRows &src = GU ? a.xq : a.hq;
        float *myscl = escl + (size_t)(tid - kWarpEpi0 * 32) * 16;
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        uint32_t it = 0;
        for (int task = blockIdx.x; task < total && !aborted(sh); task += gridDim.x) {
            const TcTask t = tc_task<GU>(a, *ps, task);
            cp_async_wait<0>();   // the last task's scale copies (none pending otherwise)
            float2 acc[32];   // columns 2j, 2j + 1
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = make_float2(0.0f, 0.0f);
            // the row's group scales, copied 8 at a time into this thread's two shared slots,
            // one block of 8 ahead (G is a multiple of 8)
            const float *srow = t.s + (size_t)i * t.G;
            cp_async16(myscl, srow, true);
            cp_async16(myscl + 4, srow + 4, true);
            cp_async_commit();
            const int ncols = t.np - c0;   // this warp's token columns in the tile (may be <= 0)
            // activation scales of this warp's 64 token columns: lane l holds columns l, 32 + l
            float tsc[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int jj = c0 + h2 * 32 + lane;
                tsc[h2] = 0.0f;
                if (jj < t.nt) {
                    const int arow = GU ? (t.sh ? t.j0 + jj : a.tok[t.tokbase + t.j0 + jj]) : t.rowbase + jj;
                    tsc[h2] = src.scale[arow];
                }
            }
            bool ok = true;
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
                const float2 s2 = make_float2(scl, scl);
                const uint32_t buf = it % kDBuf;
                if (!(ok = tc_wait_warp(&sh->dfull[buf], (it / kDBuf) & 1, sh, a.err))) break;
                tc::fence_after_sync();
                const uint32_t col = tl + kColD + buf * kN + c0;
                // the warp's 64 columns in two halves of two loads each (both in flight at
                // once); the accumulator is released once the second half has landed
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t ra[16], rb[16];
                    const int cb = hh * 32;
                    if (cb < ncols) tc::ld16(col + cb, ra);
                    if (cb + 16 < ncols) tc::ld16(col + cb + 16, rb);
                    tc::wait_ld();
                    if (hh == 1) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh->dempty[buf]);
                    }
                    if (cb < ncols) {
#pragma unroll
                        for (int j = 0; j < 16; j += 2) ffma2(acc[(cb + j) >> 1], s2, ra[j], ra[j + 1]);
                    }
                    if (cb + 16 < ncols) {
#pragma unroll
                        for (int j = 0; j < 16; j += 2) ffma2(acc[(cb + 16 + j) >> 1], s2, rb[j], rb[j + 1]);
                    }
                    if (PROBE) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int jj = c0 + cb + j;
                            if (jj < t.nt && t.sh == 0) {
                                const size_t pr = (size_t)(t.rowbase + jj - a.routed_rowbase);
                                const size_t o = (pr * (size_t)(GU ? a.F : a.H) + t.r0 + i) * t.G + g;
                                int32_t *dst = GU ? (t.m == 0 ? a.probe.acc_gate : a.probe.acc_up) : a.probe.acc_down;
                                const uint32_t d = j < 16 ? ra[j] : rb[j - 16];
                                if (dst) dst[o] = (int32_t)__uint_as_float(d);   // an exact integer
                            }
                        }
                    }
                }
            }
            if (!ok || aborted(sh)) break;
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
            for (int j = 0; j < 64; ++j) {
                const int jj = c0 + j;
                const float sx = __shfl_sync(0xffffffffu, tsc[j >> 5], j & 31);
                const float v = (j & 1) ? acc[j >> 1].y : acc[j >> 1].x;
                if (jj < t.nt) dst[(size_t)(t.rowbase + jj) * ld + t.r0 + i] = sx * v;
            }
        }
        cp_async_wait<0>();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
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

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map of a [rows][ld] bf16 matrix of which the first `cols` columns are read: boxes of
// 64 columns (128 bytes) x box_rows rows, 128-byte swizzle, rows past the end read as zero.
cudaError_t bf16_rows_map(CUtensorMap *m, const __nv_bfloat16 *base, int cols, int ld, int rows, int box_rows)
{
    const auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kGK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of packed nibble rows [rows][rowbytes] u8: boxes of 128 bytes (4 groups of 64
// inputs) x 128 rows, 128-byte swizzle.
cudaError_t nibble_rows_map(CUtensorMap *m, const uint8_t *base, int rowbytes, long long rows)
{
    const auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)rowbytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)rowbytes};
    const cuuint32_t box[2] = {128, (cuuint32_t)kM};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ffn_tc(bool gu, const FfnArgs &a, cudaStream_t st)
{
    const bool probe = gu ? (a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr)
                          : a.probe.acc_down != nullptr;
    // B operand rows = output rows of the call: the x codes laid out by launch_gather_x_bf16
    // (gate/up) or the h codes written by the h quantisation (down)
    BMaps bmaps;
    memset(&bmaps, 0, sizeof bmaps);
    const int rows = a.plane_rows > 0 ? a.plane_rows : 1;
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < kBoxMaps && e == cudaSuccess; ++k)
        e = gu ? bf16_rows_map(&bmaps.m[k], a.x_bf16, a.H, a.H, rows, 16 << k)
               : bf16_rows_map(&bmaps.m[k], a.h_bf16, a.hstride, a.hstride, rows, 16 << k);
    // nibble maps: routed weights [E * rows][kdim / 2], shared [rows][kdim / 2]
    for (int sh = 0; sh < 2 && e == cudaSuccess; ++sh) {
        if (sh == 0 && !a.include_routed) continue;
        if (sh == 1 && !a.n_shared) continue;
        const moe_expert_weights &W = sh ? a.shared : a.routed;
        const long long nexp = sh ? 1 : a.E;
        if (gu) {
            const int F = sh ? a.Fs : a.F;
            e = nibble_rows_map(&bmaps.nib[sh][0], W.w_gate, a.H / 2, nexp * F);
            if (e == cudaSuccess) e = nibble_rows_map(&bmaps.nib[sh][1], W.w_up, a.H / 2, nexp * F);
        } else {
            const int F = sh ? a.Fs : a.F;
            e = nibble_rows_map(&bmaps.nib[sh][0], W.w_down, F / 2, nexp * a.H);
        }
    }
    if (e != cudaSuccess) return e;
    if (gu) {
        const int first = a.n_shared ? a.T : 0;
        e = launch_gather_x_bf16(a, first, first + (a.include_routed ? a.T * a.K : 0), st);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(num_sms()), block(kThreads);
    if (gu)
        return probe ? launch_kernel(ffn_tc_kernel<true, true>, grid, block, kSmemBytes, st, 1, a, bmaps)
                     : launch_kernel(ffn_tc_kernel<true, false>, grid, block, kSmemBytes, st, 1, a, bmaps);
    return probe ? launch_kernel(ffn_tc_kernel<false, true>, grid, block, kSmemBytes, st, 1, a, bmaps)
                 : launch_kernel(ffn_tc_kernel<false, false>, grid, block, kSmemBytes, st, 1, a, bmaps);
}

}  // namespace moe
