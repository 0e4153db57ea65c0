// Transpose kernels that move data with ordinary loads and stores (the LSU
// path): the naive one-element-per-thread forms, the 32x32 tile with a padded
// shared row pitch, and the vectorised XOR-swizzled tile.
//
// Element words are moved as raw bits: uint32_t for fp32, uint16_t for bf16.
// All index arithmetic is 64-bit; tiles are walked through a 1-D grid whose
// block index is split into (plane, tile row, tile column), tile column
// fastest, with a grid-stride loop for problems beyond the grid limit.
#include "tr_internal.h"

namespace tr {
namespace {

struct Geometry {
    int64_t batch, rows, cols, ld_in, ld_out, stride_in, stride_out;
    int64_t tiles_r, tiles_c;  // tiles along input rows / input columns
    int64_t total;             // batch * tiles_r * tiles_c
};

Geometry make_geometry(const Problem &p, int64_t tile_r, int64_t tile_c) {
    Geometry g{p.batch, p.rows, p.cols, p.ld_in, p.ld_out, p.stride_in, p.stride_out, 0, 0, 0};
    g.tiles_r = (p.rows + tile_r - 1) / tile_r;
    g.tiles_c = (p.cols + tile_c - 1) / tile_c;
    g.total = g.batch * g.tiles_r * g.tiles_c;
    return g;
}

unsigned grid_blocks(int64_t total) {
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

// ---------------------------------------------------------------------------
// Naive forms: one element per thread, no shared memory.  A 32x8 block covers
// a 32x32 patch, 4 elements per thread.  With READ_ROWS the warp's 32 lanes
// walk along an input row (coalesced reads, each write lands in a different
// output row); otherwise they walk along an output row (coalesced writes,
// strided reads).  These are the "single-index" transposes the tiled kernel
// improves on ("Shared memory and the bank conflict", opening paragraph).
template <typename T, bool READ_ROWS>
__global__ void __launch_bounds__(256) k_naive(const T *__restrict__ in, T *__restrict__ out,
                                               Geometry g) {
    for (int64_t t = blockIdx.x; t < g.total; t += gridDim.x) {
        int64_t b, tr, tc;
        split_tile(g, t, false, b, tr, tc);
        const T *src = in + b * g.stride_in;
        T *dst = out + b * g.stride_out;
        if (READ_ROWS) {
            const int64_t j = tc * 32 + threadIdx.x;          // input column
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
                const int64_t i = tr * 32 + threadIdx.y + k;  // input row
                if (i < g.rows && j < g.cols) dst[j * g.ld_out + i] = src[i * g.ld_in + j];
            }
        } else {
            const int64_t i = tr * 32 + threadIdx.x;          // output column
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
                const int64_t j = tc * 32 + threadIdx.y + k;  // output row
                if (i < g.rows && j < g.cols) dst[j * g.ld_out + i] = src[i * g.ld_in + j];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Padded tile: a 32x8 block stages a 32x32 tile in shared memory with a row
// pitch of 32 + PAD elements ("Shared memory and the bank conflict", sections
// "Turn the tile around on chip" and "Banks"; the width-33 fp32 tile is PAD = 1,
// the width-32 tile PAD = 0).  Phase 1 reads input rows (lane = column) into
// tile rows; after the barrier, phase 2 reads tile columns (lane = tile row)
// and writes output rows, so both global accesses are coalesced.
//
// Bank of the phase-2 read, lane t, tile column c, 4-byte elements:
// (t*(32+PAD) + c) mod 32 = (t*PAD + c) mod 32: PAD = 0 puts all 32 lanes on
// one bank (32-way), PAD = 1 gives 32 distinct banks.  For 2-byte elements two
// lanes share a word: PAD = 2 (one word) is the conflict-free pitch.
template <typename T, int PAD>
__global__ void __launch_bounds__(256) k_tile_pad(const T *__restrict__ in, T *__restrict__ out,
                                                  Geometry g) {
    __shared__ T tile[32][32 + PAD];
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int64_t t = blockIdx.x; t < g.total; t += gridDim.x) {
        int64_t b, tr, tc;
        split_tile(g, t, false, b, tr, tc);
        const T *src = in + b * g.stride_in;
        T *dst = out + b * g.stride_out;
        const int64_t r0 = tr * 32, c0 = tc * 32;
        if (t != blockIdx.x) __syncthreads();  // previous tile fully read
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
            const int64_t i = r0 + ty + k, j = c0 + tx;
            if (i < g.rows && j < g.cols) tile[ty + k][tx] = src[i * g.ld_in + j];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
            const int64_t j = c0 + ty + k, i = r0 + tx;   // output row j, column i
            if (i < g.rows && j < g.cols) dst[j * g.ld_out + i] = tile[tx][ty + k];
        }
    }
}

// ---------------------------------------------------------------------------
// Vectorised swizzled tile.
//
// A 16-byte chunk holds V = 16 / sizeof(T) elements (4 fp32 or 8 bf16).  The
// block stages a 16V x 16V tile (64x64 fp32 = 16 KiB, 128x128 bf16 = 32 KiB):
// 16V rows of 16 chunks.  256 threads.
//
// Phase 1 (load): thread t takes chunk cc = t % 16 of rows t/16 + 16k,
//   k < V, with 16-byte global loads (a warp reads two 256-byte row segments),
//   all V loads in flight before the first shared store.
// Shared layout: chunk cc of tile row r is stored at chunk position
//   cc ^ ((r / V) % 8) of that row.  A shared 16-byte access is served in
//   quarter-warp phases of 8 lanes; it is conflict-free when the 8 lanes hit
//   8 distinct chunk positions modulo 8 (a 256-byte row covers 8 banks-worth of
//   chunks twice).  Phase-1 stores: 8 lanes = 8 consecutive chunks of one row,
//   XOR with one key -> distinct.
// Phase 2 (transpose): thread t owns the V x V micro-block of tile rows
//   V*A .. V*A+V-1 (A = t % 16) and chunk C = t / 16.  It reads V chunks
//   (rows V*A+m, chunk C) -> positions C ^ (A % 8): the 8 lanes of a phase
//   have A = 0..7 (or 8..15) and one C, so distinct.  A register transpose
//   turns the V input rows into V output rows (pure renaming for fp32; 32
//   byte permutes for bf16), and each output row V*C+m' gets one 16-byte store
//   at output columns V*A..: 16 lanes write 256 contiguous bytes of one row.
//
// VEC_IN / VEC_OUT: 16-byte global access on that side (needs 16-byte aligned
// base and pitches); otherwise that side moves single elements, which keeps
// every access in bounds and aligned for any pitch.
template <typename T>
struct VecTraits;
template <>
struct VecTraits<uint32_t> {
    static constexpr int V = 4;
};
template <>
struct VecTraits<uint16_t> {
    static constexpr int V = 8;
};

union Chunk {
    uint4 v;
    uint32_t w[4];
    uint16_t h[8];
};

// Register transpose of a V x V micro-block held as V chunks (rows) into V
// chunks (columns): out[m'] element e = in[e] element m'.
__device__ __forceinline__ void micro_transpose(const Chunk (&x)[4], Chunk (&y)[4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) y[m].w[k] = x[k].w[m];
}
__device__ __forceinline__ void micro_transpose(const Chunk (&x)[8], Chunk (&y)[8]) {
    // Output row m' takes half (m' & 1) of word (m' >> 1) from every input row;
    // output word w' pairs input rows 2w' (low half) and 2w'+1 (high half).
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int w = 0; w < 4; ++w)
            y[m].w[w] = __byte_perm(x[2 * w].w[m >> 1], x[2 * w + 1].w[m >> 1],
                                    (m & 1) ? 0x7632 : 0x5410);
}

template <typename T, bool VEC_IN, bool VEC_OUT>
__global__ void __launch_bounds__(256) k_tile_vec(const T *__restrict__ in, T *__restrict__ out,
                                                  Geometry g, bool diagonal) {
    constexpr int V = VecTraits<T>::V;
    constexpr int TILE = 16 * V;       // tile is TILE x TILE elements
    __shared__ uint4 smem[TILE * 16];  // TILE rows of 16 chunks

    const int t = threadIdx.x;
    const int lcc = t & 15, lr = t >> 4;  // phase 1: chunk, first row
    const int A = t & 15, C = t >> 4;     // phase 2: micro-block coordinates

    for (int64_t tile = blockIdx.x; tile < g.total; tile += gridDim.x) {
        int64_t b, tr, tc;
        split_tile(g, tile, diagonal, b, tr, tc);
        const T *src = in + b * g.stride_in;
        T *dst = out + b * g.stride_out;
        const int64_t r0 = tr * TILE, c0 = tc * TILE;
        const bool full = (r0 + TILE <= g.rows) && (c0 + TILE <= g.cols);

        // ---- phase 1: global -> registers -> swizzled shared tile
        Chunk ld[V];
        const int64_t gc = c0 + lcc * V;  // first input column of this chunk
        if (full && VEC_IN) {
#pragma unroll
            for (int k = 0; k < V; ++k)
                ld[k].v = __ldcs(reinterpret_cast<const uint4 *>(src + (r0 + lr + 16 * k) * g.ld_in + gc));
        } else {
#pragma unroll
            for (int k = 0; k < V; ++k) {
                const int64_t gr = r0 + lr + 16 * k;
                if (VEC_IN && gr < g.rows && gc + V <= g.cols) {
                    ld[k].v = __ldcs(reinterpret_cast<const uint4 *>(src + gr * g.ld_in + gc));
                } else {
                    T e[V];
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        e[q] = (gr < g.rows && gc + q < g.cols) ? src[gr * g.ld_in + gc + q] : T(0);
                    if (sizeof(T) == 4) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) ld[k].w[q] = uint32_t(e[q]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ld[k].w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                    }
                }
            }
        }
        if (tile != blockIdx.x) __syncthreads();  // previous tile fully read
#pragma unroll
        for (int k = 0; k < V; ++k) {
            const int r = lr + 16 * k;
            smem[r * 16 + (lcc ^ ((r / V) & 7))] = ld[k].v;
        }
        __syncthreads();

        // ---- phase 2: micro-block -> registers -> transpose -> global
        Chunk x[V], y[V];
#pragma unroll
        for (int m = 0; m < V; ++m) {
            const int r = V * A + m;
            x[m].v = smem[r * 16 + (C ^ (A & 7))];
        }
        micro_transpose(x, y);
        const int64_t oc = r0 + V * A;  // first output column of this chunk
        if (full && VEC_OUT) {
#pragma unroll
            for (int m = 0; m < V; ++m)
                __stcs(reinterpret_cast<uint4 *>(dst + (c0 + V * C + m) * g.ld_out + oc), y[m].v);
        } else {
#pragma unroll
            for (int m = 0; m < V; ++m) {
                const int64_t orow = c0 + V * C + m;
                if (orow >= g.cols) break;
                T *row = dst + orow * g.ld_out;
                if (VEC_OUT && oc + V <= g.rows) {
                    __stcs(reinterpret_cast<uint4 *>(row + oc), y[m].v);
                } else {
#pragma unroll
                    for (int q = 0; q < V; ++q) {
                        if (oc + q < g.rows) {
                            if (sizeof(T) == 4) row[oc + q] = T(y[m].w[q]);
                            else row[oc + q] = T(y[m].w[q >> 1] >> ((q & 1) * 16));
                        }
                    }
                }
            }
        }
    }
}

template <typename T>
cudaError_t launch_vec_typed(const Problem &p, bool vec_in, bool vec_out, bool diagonal) {
    constexpr int TILE = 16 * VecTraits<T>::V;
    const Geometry g = make_geometry(p, TILE, TILE);
    const unsigned grid = grid_blocks(g.total);
    const T *in = static_cast<const T *>(p.in);
    T *out = static_cast<T *>(p.out);
    if (vec_in && vec_out)
        k_tile_vec<T, true, true><<<grid, 256, 0, p.stream>>>(in, out, g, diagonal);
    else if (vec_in)
        k_tile_vec<T, true, false><<<grid, 256, 0, p.stream>>>(in, out, g, diagonal);
    else if (vec_out)
        k_tile_vec<T, false, true><<<grid, 256, 0, p.stream>>>(in, out, g, diagonal);
    else
        k_tile_vec<T, false, false><<<grid, 256, 0, p.stream>>>(in, out, g, diagonal);
    return cudaGetLastError();
}

template <typename T, int PAD>
void launch_pad_one(const Problem &p, const Geometry &g) {
    k_tile_pad<T, PAD><<<grid_blocks(g.total), dim3(32, 8), 0, p.stream>>>(
        static_cast<const T *>(p.in), static_cast<T *>(p.out), g);
}

template <typename T>
cudaError_t launch_pad_typed(const Problem &p, int pad) {
    const Geometry g = make_geometry(p, 32, 32);
    switch (pad) {
        case 0: launch_pad_one<T, 0>(p, g); break;
        case 1: launch_pad_one<T, 1>(p, g); break;
        case 2: launch_pad_one<T, 2>(p, g); break;
        case 3: launch_pad_one<T, 3>(p, g); break;
        case 4: launch_pad_one<T, 4>(p, g); break;
        case 8: launch_pad_one<T, 8>(p, g); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_naive_typed(const Problem &p, bool read_rows) {
    const Geometry g = make_geometry(p, 32, 32);
    const T *in = static_cast<const T *>(p.in);
    T *out = static_cast<T *>(p.out);
    if (read_rows)
        k_naive<T, true><<<grid_blocks(g.total), dim3(32, 8), 0, p.stream>>>(in, out, g);
    else
        k_naive<T, false><<<grid_blocks(g.total), dim3(32, 8), 0, p.stream>>>(in, out, g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_naive(const Problem &p, bool read_coalesced) {
    return p.esize == 4 ? launch_naive_typed<uint32_t>(p, read_coalesced)
                        : launch_naive_typed<uint16_t>(p, read_coalesced);
}

cudaError_t launch_tile_pad(const Problem &p, int pad) {
    return p.esize == 4 ? launch_pad_typed<uint32_t>(p, pad) : launch_pad_typed<uint16_t>(p, pad);
}

cudaError_t launch_tile_vec(const Problem &p, bool vec_in, bool vec_out, int tile_order) {
    const bool diag = tile_order == 1;
    return p.esize == 4 ? launch_vec_typed<uint32_t>(p, vec_in, vec_out, diag)
                        : launch_vec_typed<uint16_t>(p, vec_in, vec_out, diag);
}

}  // namespace tr
