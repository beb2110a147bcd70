// tdp_geom.h -- tile geometry of one TDP problem, as the plan stores it and
// as every kernel receives it (by value, as a __grid_constant__ parameter:
// ~2.4 KB, well inside the kernel-parameter limit, so no device allocation
// and no shared __constant__ bank that concurrent plans could race on).
//
// Along a dimension of extent L with n tiles and overlap o ("Tiled Data
// Parallelism (TDP)", "API / Tiling config": counts, not sizes), tile i spans
// [lo[i], hi[i]) = [c_i - floor(o/2), c_{i+1} + o - floor(o/2)) clipped at the
// outer edges, c_i = floor(i*L/n).  pre[i] is the sum of the sizes of tiles
// 0..i-1 and sum the sum of all sizes, so that the token offset of tile
// (iF, iH, iW) in the tile-major buffers is
//   off = pre_F[iF]*sum_H*sum_W + S_F[iF]*(pre_H[iH]*sum_W + S_H[iH]*pre_W[iW]).
#pragma once

#include <stdint.h>

#include "tdp.h"

struct tdp_dim_geom {
    int32_t L;                              // extent along this dimension
    int32_t n;                              // tiles
    int32_t o;                              // overlap (0 when n == 1)
    int32_t sum;                            // sum of tile sizes
    int32_t lo[TDP_MAX_TILES_PER_DIM];
    int32_t hi[TDP_MAX_TILES_PER_DIM];
    int32_t pre[TDP_MAX_TILES_PER_DIM];
};

struct tdp_geom {
    int32_t B, F, H, W, C;
    int32_t dtype;                          // tdp_dtype
    int32_t esize;                          // bytes per latent element
    int32_t nt;                             // n_F * n_H * n_W
    int64_t total;                          // sum_t T_t (tokens per batch item)
    tdp_dim_geom d[3];                      // F, H, W
};

struct tdp_plan_s {
    tdp_geom g;
};
