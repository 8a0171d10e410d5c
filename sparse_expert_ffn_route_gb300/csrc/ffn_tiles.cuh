// ffn_tiles.cuh -- work geometry of the grouped expert-FFN kernels, shared by the host-side
// configuration, the planner and the kernels so that all three cut a slot's work alike.
//
// A matrix row reducing over `kdim` inputs is kdim/2 bytes of packed nibbles, i.e. kdim/32
// 16-byte chunks of 32 codes.  `lpr` lanes of a warp share a row: the whole warp when the row
// has more than 32 chunks or when the launch's other matrix does ("full"), else the smallest
// power of two covering the chunks.  A warp covers rpw = 32/lpr rows at once and a lane owns
// nc chunks of the row (gl, gl+lpr, ...), so nc > 1 only ever goes with lpr = 32.  A task is one block of ru*rpw consecutive rows of
// one expert for one chunk of at most tc tokens; a warp loads the ru row groups of a task
// together, so ru*nc 16-byte loads per matrix are in flight per lane.
#pragma once

#include "device_util.cuh"

namespace moe {

constexpr int kFfnWarpsPerCta = 8;
constexpr int kFfnThreads = kFfnWarpsPerCta * 32;

struct Geo {
    int kdim, nrows;      // reduction length and rows of the matrix (per expert)
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

__host__ __device__ inline Geo make_geo(int kdim, int nrows, int ru, bool full)
{
    Geo g;
    g.kdim = kdim;
    g.nrows = nrows;
    const int nch = kdim / 32;
    g.lpr = full ? 32 : pow2_ceil_ge(nch, 32);
    g.rpw = 32 / g.lpr;
    g.nc = (nch + g.lpr - 1) / g.lpr;
    g.ru = ru;
    g.rb = ru * g.rpw;
    g.rowbytes = kdim / 2;
    g.G = kdim / 64;
    return g;
}

// Tasks of a slot: (token chunk of at most tc tokens, row block), chunk-major.
__host__ __device__ __forceinline__ int tasks_of(const Geo &g, int ntok, int tc)
{
    if (ntok <= 0) return 0;
    return ((g.nrows + g.rb - 1) / g.rb) * ((ntok + tc - 1) / tc);
}

}  // namespace moe
