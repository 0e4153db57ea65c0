// Tile walk shared by the LSU transpose kernels: a linear tile index (one per
// block, grid-stride beyond the grid limit) split into plane, tile row and tile
// column, tile column fastest.
#pragma once

#include <cstdint>

#include "tr_internal.h"

namespace tr {

struct Geometry {
    int64_t batch, rows, cols, ld_in, ld_out, stride_in, stride_out;
    int64_t tiles_r, tiles_c;  // tiles along input rows / input columns
    int64_t total;             // batch * tiles_r * tiles_c
};

inline Geometry make_geometry(const Problem &p, int64_t tile_r, int64_t tile_c) {
    Geometry g{p.batch, p.rows, p.cols, p.ld_in, p.ld_out, p.stride_in, p.stride_out, 0, 0, 0};
    g.tiles_r = (p.rows + tile_r - 1) / tile_r;
    g.tiles_c = (p.cols + tile_c - 1) / tile_c;
    g.total = g.batch * g.tiles_r * g.tiles_c;
    return g;
}

inline unsigned grid_blocks(int64_t total) {
    const int64_t cap = int64_t(1) << 30;
    return unsigned(total < cap ? total : cap);
}

// Splits a linear tile index into plane / tile row / tile column.  With
// `diagonal`, the tile column is rotated by the tile row, so blocks that run
// at the same time spread their output rows over more of the address space.
__device__ __forceinline__ void split_tile(const Geometry &g, int64_t t, bool diagonal,
                                           int64_t &b, int64_t &tr, int64_t &tc) {
    const int64_t per_plane = g.tiles_r * g.tiles_c;
    b = t / per_plane;
    const int64_t r = t - b * per_plane;
    tr = r / g.tiles_c;
    tc = r - tr * g.tiles_c;
    if (diagonal) {
        tc += tr;
        if (tc >= g.tiles_c) tc -= g.tiles_c * (tc / g.tiles_c);
    }
}

}  // namespace tr
