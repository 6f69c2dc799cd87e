// Tile-space arithmetic shared by the kernels (device) and the host API.
//
// The output C (M x N) is cut into a grid of bm x bn tiles, the partition
// view of the CUDA Programming Guide 13.4.2 (unofficial Chinese translation),
// section 2.4.6.1 "Tile-space load and store", Figure 19: tile (i, j) covers
// rows [i*bm, i*bm + bm) and columns [j*bn, j*bn + bn), clipped to the array;
// the grid is ceil(M/bm) x ceil(N/bn).
//
// A persistent CTA walks tile numbers bid = blockIdx.x, blockIdx.x + gridDim.x,
// ... and maps each to a tile with the grouped ("swizzled") order of "Writing
// high-performance matrix multiplication with NVIDIA CUDA Tile", section
// "Performance optimisation: Swizzle": tile numbers are dealt out in bands of
// group_m tile rows; within a band consecutive numbers go down the band's rows
// first and then move one tile column to the right, so CTAs running at the
// same time share A row-blocks and B column-blocks in L2.  The row inside the
// band is taken from the tile number itself (not from its offset inside the
// band), as that tutorial does; in the last, shorter band this rotates the
// rows but keeps the mapping one-to-one.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define TGEMM_HD __host__ __device__ __forceinline__
#else
#define TGEMM_HD inline
#endif

namespace tgemm {

TGEMM_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct TileGrid {
    int64_t tiles_m, tiles_n;

    TGEMM_HD TileGrid(int64_t M, int64_t N, int bm, int bn)
        : tiles_m(ceil_div(M, bm)), tiles_n(ceil_div(N, bn)) {}

    TGEMM_HD int64_t count() const { return tiles_m * tiles_n; }
};

// Tile number -> (tile row, tile column) in grouped order.
TGEMM_HD void grouped_tile(int64_t tiles_m, int64_t tiles_n, int group_m, int64_t bid,
                           int64_t &tile_row, int64_t &tile_col)
{
    const int64_t band_tiles = (int64_t)group_m * tiles_n;     // tiles in one full band
    const int64_t band = bid / band_tiles;
    const int64_t row0 = band * group_m;                         // first tile row of the band
    int64_t rows = tiles_m - row0;                               // the last band may be shorter
    if (rows > group_m) rows = group_m;
    tile_row = row0 + bid % rows;
    tile_col = (bid - band * band_tiles) / rows;
}

// The same mapping in 32-bit arithmetic, for the kernels (tile counts are
// kept below 2^31 by the host; 64-bit division is a long instruction
// sequence on the GPU, run at every tile start by the producer and epilogue).
TGEMM_HD void grouped_tile32(int32_t tiles_m, int32_t tiles_n, int32_t group_m, int32_t bid, int32_t &tile_row,
                             int32_t &tile_col)
{
    const int32_t band_tiles = group_m * tiles_n;
    const int32_t band = bid / band_tiles;
    const int32_t row0 = band * group_m;
    int32_t rows = tiles_m - row0;
    if (rows > group_m) rows = group_m;
    tile_row = row0 + bid % rows;
    tile_col = (bid - band * band_tiles) / rows;
}

// Stream-K split of the last tiles ("Stream-K" work decomposition: equal
// shares of multiply-accumulate iterations instead of whole tiles).  The
// sk_tiles tail tiles hold sk_tiles * kb k-block iterations, numbered tile by
// tile; unit u (a persistent CTA pair) takes iterations [bound(u),
// bound(u+1)).  A unit's share is cut at tile boundaries into segments; a
// tile covered by several units is summed from their partial results.  Every
// unit's share touches at most kMaxSegments tiles (the host keeps the share
// under two tiles' worth).
constexpr int kMaxSegments = 3;

struct StreamK {
    int64_t sk_tiles, sk_units, kb;

    TGEMM_HD int64_t total() const { return sk_tiles * kb; }
    TGEMM_HD int64_t bound(int64_t u) const { return u * total() / sk_units; }
    // The unit whose share contains iteration x (every share is non-empty).
    TGEMM_HD int64_t unit_of(int64_t x) const
    {
        int64_t u = x * sk_units / total();
        while (u + 1 < sk_units && bound(u + 1) <= x) ++u;
        while (u > 0 && bound(u) > x) --u;
        return u;
    }
    // Workspace slot of unit u's segment of tail tile t (unit-major, one slot
    // per segment in the order the unit meets its tiles).
    TGEMM_HD int64_t slot(int64_t u, int64_t t) const { return u * kMaxSegments + (t - bound(u) / kb); }
};

}  // namespace tgemm
