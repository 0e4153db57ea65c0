// Transpose kernels that move one element per access with ordinary loads and
// stores: the naive one-element-per-thread forms and the 32x32 tile with a
// padded shared row pitch (the vectorised swizzled tile is in tile_vec_kernel.cuh).
//
// Element words are moved as raw bits: uint32_t for fp32, uint16_t for bf16.
// All index arithmetic is 64-bit; tiles are walked through a 1-D grid whose
// block index is split into (plane, tile row, tile column), tile column
// fastest, with a grid-stride loop for problems beyond the grid limit.
#include "bounds.cuh"
#include "launch.cuh"
#include "tile_geom.cuh"
#include "tr_internal.h"

namespace tr {
namespace {

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
    pdl_prologue();
    TR_SIDE(in_side, in, g.batch, g.rows, g.cols, g.ld_in, g.stride_in, int(sizeof(T)));
    TR_SIDE(out_side, out, g.batch, g.cols, g.rows, g.ld_out, g.stride_out, int(sizeof(T)));
    auto move = [&](T *d, const T *s) {
        if (TR_LOAD_OK(in_side, s, int(sizeof(T))) && TR_STORE_OK(out_side, d, int(sizeof(T)))) *d = *s;
    };
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
                if (i < g.rows && j < g.cols) move(dst + j * g.ld_out + i, src + i * g.ld_in + j);
            }
        } else {
            const int64_t i = tr * 32 + threadIdx.x;          // output column
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
                const int64_t j = tc * 32 + threadIdx.y + k;  // output row
                if (i < g.rows && j < g.cols) move(dst + j * g.ld_out + i, src + i * g.ld_in + j);
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
    pdl_prologue();
    const int tx = threadIdx.x, ty = threadIdx.y;
    TR_SIDE(in_side, in, g.batch, g.rows, g.cols, g.ld_in, g.stride_in, int(sizeof(T)));
    TR_SIDE(out_side, out, g.batch, g.cols, g.rows, g.ld_out, g.stride_out, int(sizeof(T)));
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
            if (i < g.rows && j < g.cols && TR_LOAD_OK(in_side, src + i * g.ld_in + j, int(sizeof(T))))
                tile[ty + k][tx] = src[i * g.ld_in + j];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
            const int64_t j = c0 + ty + k, i = r0 + tx;   // output row j, column i
            if (i < g.rows && j < g.cols && TR_STORE_OK(out_side, dst + j * g.ld_out + i, int(sizeof(T))))
                dst[j * g.ld_out + i] = tile[tx][ty + k];
        }
    }
}

template <typename T, int PAD>
cudaError_t launch_pad_one(const Problem &p, const Geometry &g) {
    return launch_pdl(k_tile_pad<T, PAD>, dim3(grid_blocks(g.total)), dim3(32, 8), 0, p.stream,
                      static_cast<const T *>(p.in), static_cast<T *>(p.out), g);
}

template <typename T>
cudaError_t launch_pad_typed(const Problem &p, int pad) {
    const Geometry g = make_geometry(p, 32, 32);
    switch (pad) {
        case 0: return launch_pad_one<T, 0>(p, g);
        case 1: return launch_pad_one<T, 1>(p, g);
        case 2: return launch_pad_one<T, 2>(p, g);
        case 3: return launch_pad_one<T, 3>(p, g);
        case 4: return launch_pad_one<T, 4>(p, g);
        case 8: return launch_pad_one<T, 8>(p, g);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_naive_typed(const Problem &p, bool read_rows) {
    const Geometry g = make_geometry(p, 32, 32);
    const T *in = static_cast<const T *>(p.in);
    T *out = static_cast<T *>(p.out);
    if (read_rows)
        return launch_pdl(k_naive<T, true>, dim3(grid_blocks(g.total)), dim3(32, 8), 0, p.stream,
                          in, out, g);
    return launch_pdl(k_naive<T, false>, dim3(grid_blocks(g.total)), dim3(32, 8), 0, p.stream, in,
                      out, g);
}

}  // namespace

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_lsu)

cudaError_t launch_naive(const Problem &p, bool read_coalesced) {
    return p.esize == 4 ? launch_naive_typed<uint32_t>(p, read_coalesced)
                        : launch_naive_typed<uint16_t>(p, read_coalesced);
}

cudaError_t launch_tile_pad(const Problem &p, int pad) {
    return p.esize == 4 ? launch_pad_typed<uint32_t>(p, pad) : launch_pad_typed<uint16_t>(p, pad);
}

}  // namespace tr
