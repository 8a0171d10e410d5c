// ffn_tiles.cuh -- work geometry of the grouped expert-FFN kernels, shared by the host-side
// configuration, the planner and the kernels so that all three cut a slot's work alike.
//
// A matrix row reducing over `kdim` inputs is kdim/2 bytes of packed nibbles, i.e. kdim/32
// 16-byte chunks of 32 codes.  The row may be cut into S slices of sch chunks (the last one
// ragged); each slice is reduced on its own and the S partial sums are added later in slice
// order.  `lpr` lanes of a warp share a row of a slice: the whole warp when the slice has
// more than 32 chunks or when the launch's other matrix does ("full"), else the smallest
// power of two covering the slice's chunks.  A warp covers rpw = 32/lpr rows at once and a
// lane owns nc chunks of the slice (gl, gl+lpr, ...), so nc > 1 only ever goes with
// lpr = 32.  A task is one block of ru*rpw consecutive rows of one expert, one slice, one
// chunk of at most tc tokens; a warp loads the ru row groups of a task together, so ru*nc
// 16-byte loads per matrix are in flight per lane.
#pragma once

#include "device_util.cuh"

namespace moe {

constexpr int kFfnWarpsPerCta = 12;
constexpr int kFfnThreads = kFfnWarpsPerCta * 32;
constexpr int kSliceChunks = 32;   // chunks per slice when rows are sliced (1024 inputs)

struct Geo {
    int kdim, nrows;      // reduction length and rows of the matrix (per expert)
    int S, sch;           // slices per row, chunks per slice
    int lpr, rpw, nc;     // lanes per row, rows per warp at once, chunks per lane
    int ru, rb;           // row groups per task, rows per task (ru * rpw)
    int rowbytes, G;      // bytes per row, 64-groups per row
};

__host__ __device__ __forceinline__ int pow2_ceil_ge(int v, int cap)
{
    int l = 1;
    while (l < v && l < cap) l *= 2;
    return l;
}

__host__ __device__ inline Geo make_geo(int kdim, int nrows, int ru, bool full, bool sliced)
{
    Geo g;
    g.kdim = kdim;
    g.nrows = nrows;
    const int nch = kdim / 32;
    g.sch = sliced && nch > kSliceChunks ? kSliceChunks : nch;
    g.S = (nch + g.sch - 1) / g.sch;
    g.lpr = full ? 32 : pow2_ceil_ge(g.sch, 32);
    g.rpw = 32 / g.lpr;
    g.nc = (g.sch + g.lpr - 1) / g.lpr;
    g.ru = ru;
    g.rb = ru * g.rpw;
    g.rowbytes = kdim / 2;
    g.G = kdim / 64;
    return g;
}

// Geometry of the tensor-core path: 128-row tiles of `matrices` matrices (gate and up, or
// down) over the whole reduction; the matrix index takes the place of the slice.
__host__ __device__ inline Geo make_tc_geo(int kdim, int nrows, int matrices)
{
    Geo g;
    g.kdim = kdim;
    g.nrows = nrows;
    g.S = matrices;
    g.sch = kdim / 32;
    g.lpr = 32;
    g.rpw = 1;
    g.nc = 1;
    g.ru = 128;
    g.rb = 128;
    g.rowbytes = kdim / 2;
    g.G = kdim / 64;
    return g;
}

// Geometry of the row-per-lane-group GEMV (ffn_rows.cu): tasks of `rows` rows (blocks of
// kRowBlock, done one after the other) over the whole reduction, every token of a chunk
// against one pass over the weights.  Down tasks take two blocks: their rows are a third as
// long as gate/up rows, and a task has costs of its own.
constexpr int kRowBlock = 64;
constexpr int kRowTok = 8;    // tokens per task at most
constexpr int kRowTaskGateUp = kRowBlock, kRowTaskDown = 2 * kRowBlock;
// Batches below this many tokens keep the warp GEMV.  Measured on the GLM decode layer
// (tokens/s, warp vs row GEMV): T = 1 14.4k vs 13.8k, T = 2 20.2k vs 20.2k, T = 3 24.1k vs
// 25.6k; with one token a 64-row task over the whole reduction is too coarse (about two per
// CTA), from three on the row GEMV's shared activation rows pay.
constexpr int kRowGemvMinT = 3;
// Warp-GEMV rows are cut into kSliceChunks-chunk slices only in batches of at least this
// many tokens.  With one or two tokens whole rows are faster (tokens/s, sliced vs whole:
// GLM decode T = 1 14.5k vs 15.9k, T = 2 20.2k vs 22.7k; wide layer T = 1 12.3k vs 13.6k;
// A3B-style T = 1 28.8k vs 30.5k): no partial-sum planes for the h quantisation and the
// combine to add up.  With more tokens (where the warp GEMV only runs for reductions the row
// GEMV does not take) a slice keeps each lane at one chunk, so the activations of 4 tokens
// fit the registers and an expert's weights are streamed once per 4 tokens, not per token.
constexpr int kSliceMinT = 3;

__host__ __device__ inline Geo make_rows_geo(int kdim, int nrows, int rows)
{
    Geo g;
    g.kdim = kdim;
    g.nrows = nrows;
    g.S = 1;
    g.sch = kdim / 32;
    g.lpr = 4;
    g.rpw = 8;
    g.nc = 1;
    g.ru = rows;
    g.rb = rows;
    g.rowbytes = kdim / 2;
    g.G = kdim / 64;
    return g;
}

// Tasks of a slot: (token chunk of at most tc tokens, slice, row block), in that order of
// significance.
__host__ __device__ __forceinline__ int tasks_of(const Geo &g, int ntok, int tc)
{
    if (ntok <= 0) return 0;
    return ((g.nrows + g.rb - 1) / g.rb) * g.S * ((ntok + tc - 1) / tc);
}

// Tokens a kernel built for chunks of tc computes for a chunk of nt (its code path: the
// smallest power of two that holds nt, at most tc) ...
__host__ __device__ __forceinline__ int chunk_width(int nt, int tc)
{
    int w = 1;
    while (w < nt && w < tc) w *= 2;
    return w;
}

// ... and the relative cost of one of its tasks: the per-token work plus about three
// tokens' worth of per-task work (copies, unpacking, reduction, stores).  Warps of the warp
// GEMV take equal shares of the summed cost, not of the task count.
__host__ __device__ __forceinline__ int task_weight(int nt, int tc) { return chunk_width(nt, tc) + 3; }

__host__ __device__ __forceinline__ long long slot_cost(const Geo &g, int ntok, int tc)
{
    if (ntok <= 0) return 0;
    const long long per_chunk = (long long)((g.nrows + g.rb - 1) / g.rb) * g.S;
    const int nch = (ntok + tc - 1) / tc, nlast = ntok - (nch - 1) * tc;
    return per_chunk * ((long long)(nch - 1) * task_weight(tc, tc) + task_weight(nlast, tc));
}

// the slot's task whose cost interval holds x (0 <= x < slot_cost)
__host__ __device__ __forceinline__ int task_at_cost(const Geo &g, int ntok, int tc, long long x)
{
    const long long per_chunk = (long long)((g.nrows + g.rb - 1) / g.rb) * g.S;
    const int nch = (ntok + tc - 1) / tc, nlast = ntok - (nch - 1) * tc;
    const long long wf = task_weight(tc, tc);
    const long long full = (long long)(nch - 1) * per_chunk * wf;
    if (x < full) return (int)(x / wf);
    return (int)((nch - 1) * per_chunk + (x - full) / task_weight(nlast, tc));
}

}  // namespace moe
