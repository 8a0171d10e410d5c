// ffn_tiles.cuh -- tile geometry of the grouped expert-FFN kernels, shared by the planner
// and the kernels so both cut a slot's work the same way.
#pragma once

#include "device_util.cuh"

namespace moe {

constexpr int kFfnWarps = 8;   // warps per CTA of the FFN kernels
constexpr int kRitGu = 2;      // row iterations per warp in a gate/up tile
constexpr int kRitDn = 8;      // row iterations per warp in a down tile
constexpr int kDnUnroll = 4;   // down rows loaded together per warp

// Rows of a tile of a matrix whose rows reduce over `kdim` (= 64 * groups).
__host__ __device__ __forceinline__ int tile_rows(int kdim, int rit)
{
    return kFfnWarps * (32 / lanes_per_row(kdim / 64)) * rit;
}

__host__ __device__ __forceinline__ int gu_tiles_of(int F, int H, int ntok, int tc)
{
    if (ntok <= 0) return 0;
    const int rows = tile_rows(H, kRitGu);
    return ((F + rows - 1) / rows) * ((ntok + tc - 1) / tc);
}

__host__ __device__ __forceinline__ int dn_tiles_of(int F, int H, int ntok, int tc)
{
    if (ntok <= 0) return 0;
    const int rows = tile_rows(F, kRitDn);
    return ((H + rows - 1) / rows) * ((ntok + tc - 1) / tc);
}

}  // namespace moe
