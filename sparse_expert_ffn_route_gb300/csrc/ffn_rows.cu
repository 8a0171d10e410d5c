// ffn_rows.cu -- grouped int4 x int8 expert FFN for decode-sized batches: every weight block
// is streamed once per chunk of up to 8 tokens ["MoE 路由与专家流式加载" §1.3: gate/up/SiLU/down
// on the integer-dot path; "colibri 开发演进实录" §2.2 K1 / K1b: int4-gs64 weights against int8
// activations, an integer dot per 64-group, then the group scale].
//
// A CTA is kRwWarps compute warps and one copy warp, one CTA per SM.  A task is (slot, rows,
// chunk of at most kRwTok tokens) over the whole reduction (geometry make_rows_geo): one block
// of kRowBlock rows for gate/up, two for down.  The copy warp takes tasks
// one at a time from a counter in the plan, so a CTA that drew long tasks (the shared
// expert's 8-token chunks) takes fewer, and streams each through a ring of stages in shared
// memory with TMA, 1024 inputs per stage: per matrix a [64 rows][4 lines][128 B] box of
// nibbles (128-byte swizzle) and the [64][16] group scales, plus one [4][256 B] box of int8
// codes per token (the row picked by token id for gate/up, by output row for down).  One TMA
// instruction per stage issues all of them, a box per lane.
//
// Compute warp w owns rows 4w .. 4w+3 of the block; lane l takes row 4w + l/8 and chunk
// c = l % 8 (16 bytes, 32 weights) of every 128-byte line, so the eight lanes of a row split
// its reduction.  Shared-memory reads run at the minimum number of wavefronts: the swizzle
// spreads a warp's nibble chunks over all banks, the codes are broadcast to the rows' lanes,
// and lanes c >= 4 read the two halves of their 32 codes (and of their 32 weights) in the
// other order, so the eight chunks of a read fall on distinct banks.
//
// Per chunk of 32 weights and token (integer, exact): with
//     lo = ((w << 4) & 0xF0F0F0F0) ^ 0x80808080,   hi = (w & 0xF0F0F0F0) ^ 0x80808080
// every byte holds 16 (u - 8) as a signed byte (u ^ 8 is u - 8 in 4-bit two's complement,
// read from the high half of a byte it counts 16 times), so
//     A = sum over the 4 words of dp4a(lo, even codes) + dp4a(hi, odd codes) = 16 dot(u - 8, q)
// needs no zero-point correction.  acc += s_group * A in fp32; the 1/16 joins the activation
// scale in the epilogue.  Three shuffles add the eight lanes' partial sums; gate/up ends with
// h = SiLU(sx * gate) * (sx * up), down with y = sh * acc.
#include <cuda.h>           // CUtensorMap and its enums (types only: the encoder is looked up)
#include <cudaTypedefs.h>   // PFN_cuTensorMapEncodeTiled

#include <cstring>
#include <mutex>

#include "ffn_kernels.cuh"
#include "launch.cuh"

namespace moe {

namespace {

using ffn_impl::Task;

constexpr int kRwWarps = 16;                           // compute warps
constexpr int kRwRowsPerWarp = 4;
constexpr int kRwThreads = (kRwWarps + 1) * 32;        // + the copy warp
constexpr int kRwTok = kRowTok;                        // tokens per task at most
constexpr int kRwLines = 4;                            // 128-byte lines per row and stage
constexpr int kRwInputs = kRwLines * 256;              // inputs per stage
constexpr int kRwWBytes = kRowBlock * kRwLines * 128;  // nibbles of one matrix per stage
constexpr int kRwSBytes = kRowBlock * kRwLines * 4 * 4;   // its group scales
constexpr int kRwTokBytes = kRwLines * 256;            // codes of one token per stage
constexpr int kRwABytes = kRwTok * kRwTokBytes;

static_assert(kRowBlock == kRwWarps * kRwRowsPerWarp, "the compute warps cover the row block");
static_assert(kRwTok % 8 == 0 && kRwTok <= 16, "a lane stores tokens c, c+8, ...; lanes issue the code boxes");

// operand blocks per stage, each with its own nibble and scale boxes: gate and up of the same
// 64 rows, or the two 64-row blocks of a down task.  Both share every code read.
template <bool GU>
constexpr int rw_nm() { return 2; }
template <bool GU>
constexpr int rw_stage_bytes() { return rw_nm<GU>() * (kRwWBytes + kRwSBytes) + kRwABytes; }
// as many stages as fit the budget (beside the plan copy, within 227 KB)
constexpr int kRwRingBudget = 180 * 1024;
template <bool GU>
constexpr int rw_stages() { return kRwRingBudget / rw_stage_bytes<GU>(); }

static_assert(rw_stage_bytes<true>() % 1024 == 0 && rw_stage_bytes<false>() % 1024 == 0,
              "stages keep the 1024-byte alignment of the swizzled boxes");
static_assert(rw_stages<false>() >= rw_stages<true>(), "RwShared holds the deeper ring");

// Written by the copy warp into the slot of a task's first stage, before the stage's arrival:
// the task, decoded, and the code row of each of its tokens.  task -1: no more tasks.
struct RwHdr {
    int task, e, r0, j0, nt, rowbase, tokbase, pad;
    int arow[kRwTok];
};

// The activation scales of the call (x by token, or h by output row), copied into shared
// memory once per CTA when there are at most this many: a global load issued at a task's start
// would not return before its end while the ring keeps HBM saturated.
constexpr int kRwScaleTable = 4096;

struct RwShared {
    uint64_t full[rw_stages<false>()];    // stage landed (TMA transaction bytes)
    uint64_t empty[rw_stages<false>()];   // stage read (one arrival per compute warp)
    RwHdr hdr[rw_stages<false>()];
    int abort;
};

// the plan's per-slot arrays, copied into shared memory once per CTA
struct RwPlan {
    int n_slots;
    int32_t prefix[kMaxSlots + 1], expert[kMaxSlots], ntok[kMaxSlots], tokbase[kMaxSlots],
        rowbase[kMaxSlots];
};

template <bool GU>
constexpr size_t rw_smem_bytes()
{
    return 1024 /* alignment */ + (size_t)rw_stages<GU>() * rw_stage_bytes<GU>() + sizeof(RwShared) +
           sizeof(RwPlan) + kRwScaleTable * sizeof(float);
}

// Tensor maps (all 3-D, so that one instruction issues every box of a stage): nibbles and
// scales of [routed, shared][matrix], and the codes.
struct RowMaps {
    CUtensorMap w[2][2];
    CUtensorMap s[2][2];
    CUtensorMap act;
};

__device__ __forceinline__ bool rw_aborted(const RwShared *sh) { return *(volatile const int *)&sh->abort != 0; }

// bounded wait by every lane of a converged warp; false for all lanes once any lane gave up
// or the CTA was told to stop
__device__ __forceinline__ bool rw_wait_warp(uint64_t *bar, uint32_t parity, RwShared *sh, int32_t *err)
{
    bool ok = !rw_aborted(sh);
    if (ok && !mbar_wait(bar, parity)) {
        atomicOr(err, kErrTimeout);
        atomicExch(&sh->abort, 1);
        ok = false;
    }
    return __all_sync(0xffffffffu, ok);
}

// 3-D tiled TMA load with an L2 eviction policy (createpolicy value)
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                       uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// the 8 nibbles of word w as two words of signed bytes 16 (u - 8): even elements, odd elements
__device__ __forceinline__ void signed_nibbles(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    lo = ((w << 4) & 0xF0F0F0F0u) ^ 0x80808080u;
    hi = (w & 0xF0F0F0F0u) ^ 0x80808080u;
}

// row of the codes of token j of the task: x by token id (gate/up), h by output row (down)
template <bool GU>
__device__ __forceinline__ int act_row(const FfnArgs &a, const Task &t, int j)
{
    if (GU) return t.sh ? t.j0 + j : a.tok[t.tokbase + t.j0 + j];
    return t.rowbase + j;
}

// task -> (slot, rows, token chunk): tasks run (chunk, rows) within a slot, rows first
template <bool GU>
__device__ __forceinline__ Task rw_task(const FfnArgs &a, const RwPlan &ps, int task)
{
    int lo = 0, hi = ps.n_slots;   // the last slot whose first task is at or before `task`
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ps.prefix[mid] <= task) lo = mid;
        else hi = mid;
    }
    Task t;
    t.slot = lo;
    t.e = ps.expert[lo];
    t.sh = t.e < 0 ? 1 : 0;
    const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
    const int nblk = (g.nrows + g.rb - 1) / g.rb;
    const int local = task - ps.prefix[lo];
    const int ch = local / nblk, blk = local - ch * nblk;
    t.j0 = ch * kRwTok;
    t.nt = min(kRwTok, ps.ntok[lo] - t.j0);
    t.r0 = blk * g.rb;
    t.tokbase = ps.tokbase[lo];
    t.rowbase = ps.rowbase[lo] + t.j0;
    t.s = 0;
    return t;
}

// The compute warps' share of one task, computed for N tokens (N >= the task's token count):
// every stage of the reduction, then the epilogue.  Operand block m is gate (m = 0) and up
// (m = 1) of rows t.r0 .. t.r0+63 for gate/up, rows t.r0 + 64 m .. for down.  k counts the
// stages of the CTA.
template <bool GU, bool PROBE, int N>
__device__ __forceinline__ bool rows_task(const FfnArgs &a, const Task &t, const Geo &g, int nst,
                                          const uint8_t *ring, RwShared *sh, uint32_t &k, int rin,
                                          int c, int lane, const float (&sx)[kRwTok / 8])
{
    constexpr int NM = rw_nm<GU>();
    constexpr int D = rw_stages<GU>();
    constexpr int SB = rw_stage_bytes<GU>();
    float acc[NM][N];
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int j = 0; j < N; ++j) acc[m][j] = 0.0f;
    const int sw = c >> 2;   // lanes c >= 4 take the second half of their codes first

    for (int s = 0; s < nst; ++s, ++k) {
        const int slot = (int)(k % D);
        if (!rw_wait_warp(&sh->full[slot], (k / D) & 1, sh, a.err)) return false;
        const uint8_t *stg = ring + (size_t)slot * SB;
        const uint8_t *sbase = stg + NM * kRwWBytes;
        const uint8_t *abase = stg + NM * (kRwWBytes + kRwSBytes);
#pragma unroll
        for (int kb = 0; kb < kRwLines; ++kb) {
            const int line = rin * kRwLines + kb;
            const int woff = line * 128 + ((c ^ (line & 7)) << 4);
            const int gl = kb * 4 + (c >> 1);   // group within the stage
            uint32_t lo[NM][4], hi[NM][4];
            float sc[NM];
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                // the chunk as two 8-byte halves, in the order this lane reads its codes
                const uint2 *wp = reinterpret_cast<const uint2 *>(stg + m * kRwWBytes + woff);
                const uint2 w0 = wp[sw], w1 = wp[sw ^ 1];
                const uint4 wq = make_uint4(w0.x, w0.y, w1.x, w1.y);
                signed_nibbles(wq.x, lo[m][0], hi[m][0]);
                signed_nibbles(wq.y, lo[m][1], hi[m][1]);
                signed_nibbles(wq.z, lo[m][2], hi[m][2]);
                signed_nibbles(wq.w, lo[m][3], hi[m][3]);
                sc[m] = *reinterpret_cast<const float *>(sbase + m * kRwSBytes + (rin * kRwLines * 4 + gl) * 4);
            }
#pragma unroll
            for (int j = 0; j < N; ++j) {
                const uint4 *ap = reinterpret_cast<const uint4 *>(abase + j * kRwTokBytes + kb * 256 + c * 32);
                const uint4 a0 = ap[sw], a1 = ap[sw ^ 1];
#pragma unroll
                for (int m = 0; m < NM; ++m) {
                    int d0 = dp4a_ss(lo[m][0], a0.x, 0);
                    int d1 = dp4a_ss(lo[m][2], a1.x, 0);
                    d0 = dp4a_ss(hi[m][0], a0.y, d0);
                    d1 = dp4a_ss(hi[m][2], a1.y, d1);
                    d0 = dp4a_ss(lo[m][1], a0.z, d0);
                    d1 = dp4a_ss(lo[m][3], a1.z, d1);
                    d0 = dp4a_ss(hi[m][1], a0.w, d0);
                    d1 = dp4a_ss(hi[m][3], a1.w, d1);
                    const int d = d0 + d1;   // 16 x the chunk's dot(u - 8, q)
                    acc[m][j] = fmaf(sc[m], (float)d, acc[m][j]);
                    if (PROBE) {
                        // exact per-64-group accumulators: the group's other chunk sits in
                        // lane l ^ 1
                        const int other = __shfl_xor_sync(0xffffffffu, d, 1);
                        const int grp = s * (kRwInputs / 64) + gl;
                        const int prow = t.r0 + (GU ? 0 : m * kRowBlock) + rin;
                        if (t.sh == 0 && j < t.nt && (c & 1) == 0 && grp < g.G && prow < g.nrows) {
                            const size_t pr = (size_t)(t.rowbase + j - a.routed_rowbase);
                            const size_t o = (pr * g.nrows + prow) * g.G + grp;
                            int32_t *dst = GU ? (m == 0 ? a.probe.acc_gate : a.probe.acc_up)
                                              : a.probe.acc_down;
                            if (dst) dst[o] = (d + other) >> 4;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->empty[slot]);
    }

    // the row's total over its eight lanes, then lane c stores tokens c, c+8
#pragma unroll
    for (int m = 0; m < NM; ++m)
#pragma unroll
        for (int j = 0; j < N; ++j) {
            acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 1);
            acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 2);
            acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], 4);
        }
    const int row = t.r0 + rin;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if ((j & 7) != c || j >= t.nt) continue;
        const size_t orow = (size_t)(t.rowbase + j);
        const float s = sx[j >> 3] * 0.0625f;
        if (GU) {
            const float gate = s * acc[0][j], up = s * acc[1][j];
            a.h[orow * a.hstride + row] = gate / (1.0f + expf(-gate)) * up;
        } else {
#pragma unroll
            for (int m = 0; m < NM; ++m)
                if (row + m * kRowBlock < g.nrows) a.y[orow * a.H + row + m * kRowBlock] = s * acc[m][j];
        }
    }
    return true;
}

template <bool GU, bool PROBE>
__global__ void __launch_bounds__(kRwThreads, 1)
    ffn_rows_kernel(const __grid_constant__ FfnArgs a, const __grid_constant__ RowMaps maps)
{
    constexpr int NM = rw_nm<GU>();
    constexpr int D = rw_stages<GU>();
    constexpr int SB = rw_stage_bytes<GU>();
    extern __shared__ __align__(1024) uint8_t rw_smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(((uintptr_t)rw_smem_raw + 1023) & ~(uintptr_t)1023);
    RwShared *sh = reinterpret_cast<RwShared *>(ring + (size_t)D * SB);
    RwPlan *ps = reinterpret_cast<RwPlan *>(sh + 1);
    float *stab = reinterpret_cast<float *>(ps + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < D; ++i) {
            mbar_init(&sh->full[i], 1);
            mbar_init(&sh->empty[i], kRwWarps);
        }
        sh->abort = 0;
        fence_mbar_init();
    }
    // Early mode (gate/up with a shared expert whose x codes were written at least two
    // launches back): the shared expert's tasks need neither the routing nor the plan, so
    // the copy warp issues them before the dependency wait, while the route finishes; only
    // the copy warp waits before it reads the plan.
    const bool early = GU && a.shared_early && a.n_shared;
    // Down: the plan (written at least three launches back) and the weights are older than
    // the h codes, so the slot table is read, and the copy warp arms the first ring stages of
    // the CTA's first task and sends their weight and scale boxes, before the dependency
    // wait; the token boxes and the h scales follow it.
    const bool early_dn = !GU;
    if (!early && !early_dn) pdl_wait();
    pdl_launch_dependents();
    FfnPlan *plan = const_cast<FfnPlan *>(a.plan);
    // the plan's slot table (written by the planner, which runs before this kernel)
    auto copy_plan = [&](int i0, int stride) {
        const int32_t *pre = GU ? plan->gu_prefix : plan->dn_prefix;
        const int ns = plan->n_slots;
        for (int i = i0; i <= ns; i += stride) {
            ps->prefix[i] = pre[i];
            if (i < ns) {
                ps->expert[i] = plan->expert[i];
                ps->ntok[i] = plan->ntok[i];
                ps->tokbase[i] = plan->tokbase[i];
                ps->rowbase[i] = plan->rowbase[i];
            }
        }
        if (i0 == 0) ps->n_slots = ns;
    };
    if (!early) copy_plan(threadIdx.x, blockDim.x);
    const float *gscale = GU ? a.xq.scale : a.hq.scale;
    const int nscale = GU ? a.T : a.plane_rows;
    const bool table = nscale <= kRwScaleTable;
    int32_t *next = &plan->next[GU ? 0 : 1];
    uint32_t k = 0;      // stages of this CTA so far
    uint32_t kpre = 0;   // (down, copy warp) stages armed and sent weights before the wait
    const uint64_t pol_last = l2_policy_evict_first(), pol_again = l2_policy_evict_normal();
    // (copy warp) Issues every stage of task `task` (t; arow: this lane's token row).  `last`:
    // the task is its slot's last token chunk (the slot's chunks are taken in order), whose
    // weight and scale reads are the last in this launch, so evict-first.  `weights_only`:
    // arm the task's first (at most D) stages and send only their weight and scale boxes;
    // the stages below kpre were so armed, and get only their token boxes.  False on a
    // timeout.
    auto issue = [&](int task, const Task &t, int arow, bool last, bool weights_only) -> bool {
        const Geo &geo = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
        const int nst = (geo.kdim + kRwInputs - 1) / kRwInputs;
        const int wrow = (t.sh ? 0 : t.e * geo.nrows) + t.r0;
        const uint32_t bytes = NM * (kRwWBytes + kRwSBytes) + t.nt * kRwTokBytes;
        // this lane's box: map, shared-memory offset, coordinates (the line or group
        // coordinate advances with the stage)
        const CUtensorMap *map = &maps.act;
        // (gate/up: matrix m; down: the m-th 64-row block of the one matrix)
        // z: the row coordinate of the nibble boxes (weight lanes; independent of the token
        // rows, so those lanes' copies do not wait for the arow loads)
        int off = 0, x = 0, y = 0, z = 0, dx = 0, dy = 0;
        const bool active = lane < 2 * NM + t.nt;
        const uint64_t pol = lane < 2 * NM && last ? pol_last : pol_again;
        if (lane < NM) {
            map = &maps.w[t.sh][GU ? lane : 0];
            off = lane * kRwWBytes;
            z = wrow + (GU ? 0 : lane * kRowBlock);
            dy = kRwLines;
        } else if (lane < 2 * NM) {
            map = &maps.s[t.sh][GU ? lane - NM : 0];
            off = NM * kRwWBytes + (lane - NM) * kRwSBytes;
            y = wrow + (GU ? 0 : (lane - NM) * kRowBlock);
            dx = kRwLines * 4;
        } else {
            off = NM * (kRwWBytes + kRwSBytes) + (lane - 2 * NM) * kRwTokBytes;
            dy = kRwLines;
        }
        const int smax = weights_only ? min(nst, D) : nst;
        for (int s = 0; s < smax; ++s, ++k) {
            const bool armed = !weights_only && k < kpre;
            const int slot = (int)(k % D);
            if (k >= (uint32_t)D && !rw_wait_warp(&sh->empty[slot], ((k / D) - 1) & 1, sh, a.err))
                return false;
            const uint32_t fb = smem_u32(&sh->full[slot]);
            if (s == 0 && !armed) {
                RwHdr &h = sh->hdr[slot];
                if (lane == 0) {
                    h.task = task;
                    h.e = t.e;
                    h.r0 = t.r0;
                    h.j0 = t.j0;
                    h.nt = t.nt;
                    h.rowbase = t.rowbase;
                    h.tokbase = t.tokbase;
                }
                if (lane >= 2 * NM && lane < 2 * NM + kRwTok) h.arow[lane - 2 * NM] = arow;
                __syncwarp();
            }
            if (lane == 0 && !armed) mbar_arrive_expect_tx(&sh->full[slot], bytes);
            __syncwarp();
            // the weight and scale boxes first: they need no token row
            if (lane < 2 * NM && !armed)
                tma_3d(smem_u32(ring + (size_t)slot * SB + off), map, x + s * dx, y + s * dy, z, fb,
                       pol);
            else if (active && lane >= 2 * NM && !weights_only)
                tma_3d(smem_u32(ring + (size_t)slot * SB + off), map, x + s * dx, y + s * dy, arow,
                       fb, pol);
        }
        return true;
    };
    if (early_dn) {
        __syncthreads();   // the slot table and the barriers' initialisation
        if (warp == kRwWarps && (int)blockIdx.x < plan->dn_tiles) {
            const Task t = rw_task<GU>(a, *ps, (int)blockIdx.x);
            const int j = lane - 2 * NM;
            const int arow = j >= 0 && j < t.nt ? act_row<GU>(a, t, j) : 0;
            issue((int)blockIdx.x, t, arow, ps->ntok[t.slot] <= t.j0 + kRwTok, true);
            kpre = k;
            k = 0;   // the task is issued again from its first stage: token boxes only below kpre
        }
        pdl_wait();
    }
    if (table)
        for (int i = threadIdx.x; i < nscale; i += blockDim.x) stab[i] = gscale[i];
    __syncthreads();

    if (warp == kRwWarps) {
        // ------------------------------- copy warp ------------------------------------
        // Tasks are taken one at a time from the shared counter, two ahead: the counter's
        // answer (slow while HBM is saturated) has two tasks' time to arrive.  While task i is
        // issued, task i+1 is decoded and its code rows are loaded.
        // Lane L of the stage's one TMA instruction copies: L < NM nibbles of matrix L;
        // NM <= L < 2 NM scales of matrix L - NM; 2 NM <= L < 2 NM + nt the codes of token
        // L - 2 NM.
        const int grid = (int)gridDim.x;
        // early mode: CTA b issues the shared expert's tasks b, b + grid, ... (slot 0, decoded
        // without the plan: task = chunk * row blocks + block, as the plan numbers them)
        int base = 0;   // the first task taken after the wait
        bool failed = false;
        if (early) {
            const Geo &g = a.geo_gu[1];
            const int nblk = (g.nrows + g.rb - 1) / g.rb;
            base = nblk * ((a.T + kRwTok - 1) / kRwTok);
            for (int task = (int)blockIdx.x; task < base; task += grid) {
                Task ts{};
                const int ch = task / nblk, blk = task - ch * nblk;
                ts.slot = 0;
                ts.e = -1;
                ts.sh = 1;
                ts.j0 = ch * kRwTok;
                ts.nt = min(kRwTok, a.T - ts.j0);
                ts.r0 = blk * g.rb;
                ts.tokbase = 0;
                ts.rowbase = ts.j0;
                const int j = lane - 2 * NM;
                if (!issue(task, ts, j >= 0 && j < ts.nt ? ts.j0 + j : 0, a.T <= ts.j0 + kRwTok, false)) {
                    failed = true;
                    break;
                }
            }
            pdl_wait();
            copy_plan(lane, 32);
            __syncwarp();
        }
        // after a timeout no further task is taken (the stop stage below still goes out)
        const int total = failed ? 0 : (GU ? plan->gu_tiles : plan->dn_tiles);
        if (failed) base = 0;
        auto decode = [&](int task, Task &t, int &arow) {
            if (task < total) {
                t = rw_task<GU>(a, *ps, task);
                const int j = lane - 2 * NM;
                arow = j >= 0 && j < t.nt ? act_row<GU>(a, t, j) : 0;
            }
        };
        // CTA b's first task after the wait is task base + b; the counter hands out the rest
        // from base + gridDim.x on
        int task = base + (int)blockIdx.x;
        // counter requests in flight (lane 0): the answers for tasks i+1 and, with at least
        // four tasks per CTA, i+2 (with fewer, the CTAs that start first would take them all)
        const bool deep = total - base >= 4 * grid;
        int g1 = lane == 0 && task < total ? base + grid + atomicAdd(next, 1) : total;
        int g2 = lane == 0 && task < total && deep ? base + grid + atomicAdd(next, 1) : total;
        Task t{};
        int arow = 0;
        decode(task, t, arow);
        // Issues task `task`; g holds the answer of a request made one or two tasks ago and
        // gets a new request.  The deep loop alternates g1 and g2, so no register waits on a
        // request made in the same step.  False once the stop stage is issued or on a timeout.
        auto step = [&](int &g) -> bool {
            if (task >= total) {
                // no more tasks: a stage without copies tells the compute warps to stop
                const int slot = (int)(k % D);
                if (k >= (uint32_t)D && !rw_wait_warp(&sh->empty[slot], ((k / D) - 1) & 1, sh, a.err)) return false;
                if (lane == 0) {
                    sh->hdr[slot].task = -1;
                    mbar_arrive(&sh->full[slot]);
                }
                ++k;
                return false;
            }
            const int ntask = __shfl_sync(0xffffffffu, g, 0);
            if (lane == 0 && ntask < total) g = base + grid + atomicAdd(next, 1);
            Task tn{};
            int narow = 0;
            decode(ntask, tn, narow);
            if (!issue(task, t, arow, ps->ntok[t.slot] <= t.j0 + kRwTok, false)) return false;
            task = ntask;
            t = tn;
            arow = narow;
            return true;
        };
        if (deep) {
            while (step(g1) && step(g2)) {
            }
        } else {
            while (step(g1)) {
            }
        }
        // before the CTA exits, every copy it issued has landed (the compute warps have seen
        // all of them unless the CTA stopped early)
        for (uint32_t kk = k > (uint32_t)D ? k - D : 0; kk < k; ++kk)
            if (!mbar_wait(&sh->full[kk % D], (kk / D) & 1)) atomicOr(a.err, kErrTimeout);
    } else {
        // ------------------------------- compute warps --------------------------------
        const int rin = warp * kRwRowsPerWarp + (lane >> 3), c = lane & 7;
        for (;;) {
            const int slot = (int)(k % D);
            if (!rw_wait_warp(&sh->full[slot], (k / D) & 1, sh, a.err)) break;
            const RwHdr &h = sh->hdr[slot];
            if (h.task < 0) break;
            // the header into registers: the slot is refilled while the task is still running
            Task t;
            t.e = h.e;
            t.sh = t.e < 0 ? 1 : 0;
            t.r0 = h.r0;
            t.j0 = h.j0;
            t.nt = h.nt;
            t.rowbase = h.rowbase;
            t.tokbase = h.tokbase;
            // the activation scales of this lane's tokens (c, c+8, ...), for the epilogue
            float sx[kRwTok / 8];
#pragma unroll
            for (int i = 0; i < kRwTok / 8; ++i) {
                const int j = c + 8 * i;
                const int r = j < t.nt ? h.arow[j] : 0;
                sx[i] = j < t.nt ? (table ? stab[r] : gscale[r]) : 0.0f;
            }
            const Geo &g = GU ? a.geo_gu[t.sh] : a.geo_dn[t.sh];
            const int nst = (g.kdim + kRwInputs - 1) / kRwInputs;
            // code paths for 1-6 and 8 tokens: the dot-product work follows the chunk's
            // token count (7 rounds up to 8)
            bool ok;
            switch (t.nt) {
            case 1: ok = rows_task<GU, PROBE, 1>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            case 2: ok = rows_task<GU, PROBE, 2>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            case 3: ok = rows_task<GU, PROBE, 3>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            case 4: ok = rows_task<GU, PROBE, 4>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            case 5: ok = rows_task<GU, PROBE, 5>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            case 6: ok = rows_task<GU, PROBE, 6>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            default: ok = rows_task<GU, PROBE, kRwTok>(a, t, g, nst, ring, sh, k, rin, c, lane, sx); break;
            }
            if (!ok) break;
        }
    }
    // the last CTA to finish puts the counters back to zero for the next launch (after the
    // planner, which zeroes them too: in early mode only the copy warp has waited so far)
    if (early) pdl_wait();
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&plan->done[GU ? 0 : 1], 1) == (int)gridDim.x - 1) {
            *next = 0;
            plan->done[GU ? 0 : 1] = 0;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 rw_encoder()
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

cudaError_t encode_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, const cuuint64_t (&dims)[3],
                      const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3], CUtensorMapSwizzle sw,
                      CUtensorMapL2promotion l2)
{
    const auto enc = rw_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// nibbles of `rows` rows of kdim inputs: {128 B, kdim/256 lines, rows}, boxes {128, 4, 64},
// 128-byte swizzle, reads past the end filled with zeros
cudaError_t nibble_map(CUtensorMap *m, const uint8_t *base, int kdim, long long rows)
{
    return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base,
                     {128, (cuuint64_t)(kdim / 256), (cuuint64_t)rows}, {128, (cuuint64_t)(kdim / 2)},
                     {128, kRwLines, kRowBlock}, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

// group scales [rows][kdim/64] fp32: {groups, rows, 1}, boxes of 16 groups x 64 rows
cudaError_t scale_map(CUtensorMap *m, const float *base, int kdim, long long rows)
{
    const cuuint64_t ld = (cuuint64_t)(kdim / 64) * 4;
    return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, {(cuuint64_t)(kdim / 64), (cuuint64_t)rows, 1},
                     {ld, ld * (cuuint64_t)rows}, {kRwLines * 4, kRowBlock, 1}, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// int8 codes [rows][ld], `cols` of them read: {256, cols/256, rows}, boxes {256, 4, 1}
cudaError_t code_map(CUtensorMap *m, const int8_t *base, int cols, int ld, int rows)
{
    return encode_3d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base,
                     {256, (cuuint64_t)(cols / 256), (cuuint64_t)(rows > 0 ? rows : 1)}, {256, (cuuint64_t)ld},
                     {256, kRwLines, 1}, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

bool ffn_rows_supported(const FfnArgs &a)
{
    auto ok = [](int k) { return k > 0 && k % 256 == 0; };
    if (!ok(a.H) || !ok(a.F) || (a.n_shared && !ok(a.Fs)) || a.hstride % 256 != 0) return false;
    if (a.xq.q_ld % 256 != 0 || a.hq.q_ld != a.hstride) return false;
    const moe_expert_weights *ws[2] = {&a.routed, &a.shared};
    for (const moe_expert_weights *w : ws) {
        const void *p[6] = {w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down};
        for (const void *x : p)
            if (!aligned16(x)) return false;
    }
    return aligned16(a.xq.q) && aligned16(a.hq.q);
}

cudaError_t launch_ffn_rows(bool gu, const FfnArgs &a, cudaStream_t st)
{
    RowMaps maps;
    memset(&maps, 0, sizeof maps);
    cudaError_t e = cudaSuccess;
    const bool sh = a.n_shared != 0;
    if (gu) {
        if (a.include_routed) {
            const long long rows = (long long)a.E * a.F;
            e = nibble_map(&maps.w[0][0], a.routed.w_gate, a.H, rows);
            if (e == cudaSuccess) e = nibble_map(&maps.w[0][1], a.routed.w_up, a.H, rows);
            if (e == cudaSuccess) e = scale_map(&maps.s[0][0], a.routed.s_gate, a.H, rows);
            if (e == cudaSuccess) e = scale_map(&maps.s[0][1], a.routed.s_up, a.H, rows);
        }
        if (sh && e == cudaSuccess) {
            e = nibble_map(&maps.w[1][0], a.shared.w_gate, a.H, a.Fs);
            if (e == cudaSuccess) e = nibble_map(&maps.w[1][1], a.shared.w_up, a.H, a.Fs);
            if (e == cudaSuccess) e = scale_map(&maps.s[1][0], a.shared.s_gate, a.H, a.Fs);
            if (e == cudaSuccess) e = scale_map(&maps.s[1][1], a.shared.s_up, a.H, a.Fs);
        }
        if (e == cudaSuccess) e = code_map(&maps.act, a.xq.q, a.H, a.xq.q_ld, a.T);
    } else {
        if (a.include_routed) {
            const long long rows = (long long)a.E * a.H;
            e = nibble_map(&maps.w[0][0], a.routed.w_down, a.F, rows);
            if (e == cudaSuccess) e = scale_map(&maps.s[0][0], a.routed.s_down, a.F, rows);
        }
        if (sh && e == cudaSuccess) {
            e = nibble_map(&maps.w[1][0], a.shared.w_down, a.Fs, a.H);
            if (e == cudaSuccess) e = scale_map(&maps.s[1][0], a.shared.s_down, a.Fs, a.H);
        }
        if (e == cudaSuccess) e = code_map(&maps.act, a.hq.q, a.hstride, a.hstride, a.plane_rows);
    }
    if (e != cudaSuccess) return e;
    const bool probe = gu ? (a.probe.acc_gate != nullptr || a.probe.acc_up != nullptr)
                          : a.probe.acc_down != nullptr;
    const dim3 grid(num_sms()), block(kRwThreads);
    if (gu)
        return probe ? launch_kernel(ffn_rows_kernel<true, true>, grid, block, rw_smem_bytes<true>(), st, 1, a, maps)
                     : launch_kernel(ffn_rows_kernel<true, false>, grid, block, rw_smem_bytes<true>(), st, 1, a, maps);
    return probe ? launch_kernel(ffn_rows_kernel<false, true>, grid, block, rw_smem_bytes<false>(), st, 1, a, maps)
                 : launch_kernel(ffn_rows_kernel<false, false>, grid, block, rw_smem_bytes<false>(), st, 1, a, maps);
}

}  // namespace moe
