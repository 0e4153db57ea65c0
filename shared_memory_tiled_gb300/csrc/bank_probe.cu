// Column-read microbenchmark of a 32 x 32 shared tile of 4-byte words: the
// experiment "Shared-memory tiling and bank conflicts" asks for ("Expose a
// shared-memory bank conflict": a column-read microbenchmark with an
// unpadded square tile and with one extra column) and the cheatsheet's
// "the classic case" (tile[32][32] vs tile[32][33]), plus an XOR-swizzled
// tile and a row read as the conflict-free reference.
//
// Each warp moves no global data in its loop: lane l reads logical element
// (l, c) of the tile for c = (r + warp) mod 32, r < reps, and folds the values
// (rotate left by one, then XOR) so the reads cannot be dropped.  Layouts (word
// index of logical element (row, col)):
//   0  row pitch 32:        row*32 + col          (column read: 32-way)
//   1  row pitch 33:        row*33 + col          (column read: conflict-free)
//   2  XOR swizzle:         row*32 + (col ^ row)  (column read: conflict-free)
//   3  row pitch 32, but each lane reads along a row: element (c, l) (reference)
// The tile holds value row*32 + col at every logical position, so the folded
// result of each thread is known in closed form.
#include "bounds.cuh"
#include "tr_internal.h"

namespace tr {
namespace {

template <int LAYOUT>
__device__ __forceinline__ int probe_word(int row, int col) {
    if (LAYOUT == 1) return row * 33 + col;
    if (LAYOUT == 2) return row * 32 + (col ^ row);
    return row * 32 + col;
}

template <int LAYOUT>
__global__ void __launch_bounds__(256) k_bank_probe(int reps, uint32_t *result) {
    __shared__ uint32_t tile[32 * 33];
    for (int i = threadIdx.x; i < 32 * 32; i += blockDim.x) {
        const int row = i >> 5, col = i & 31;
        tile[probe_word<LAYOUT>(row, col)] = uint32_t(row * 32 + col);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t acc = 0;
    for (int r = 0; r < reps; ++r) {
        const int c = (r + warp) & 31;
        const uint32_t v = LAYOUT == 3 ? tile[c * 32 + lane] : tile[probe_word<LAYOUT>(lane, c)];
        acc = ((acc << 1) | (acc >> 31)) ^ v;  // rotate-and-fold: no two reads cancel
    }
    uint32_t *slot = result + size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    TR_SIDE(out_side, result, 1, 1, int64_t(gridDim.x) * blockDim.x, int64_t(gridDim.x) * blockDim.x, 0, 4);
    if (TR_STORE_OK(out_side, slot, 4)) *slot = acc;
}

}  // namespace

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_bank_probe)

cudaError_t launch_bank_probe(int layout, int reps, int blocks, uint32_t *result,
                              cudaStream_t stream) {
    switch (layout) {
        case 0: k_bank_probe<0><<<blocks, 256, 0, stream>>>(reps, result); break;
        case 1: k_bank_probe<1><<<blocks, 256, 0, stream>>>(reps, result); break;
        case 2: k_bank_probe<2><<<blocks, 256, 0, stream>>>(reps, result); break;
        case 3: k_bank_probe<3><<<blocks, 256, 0, stream>>>(reps, result); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace tr
