// Vectorised swizzled tile transpose (kernel template and per-shape launch;
// the instantiations are spread over tile_vec_*.cu to compile in parallel):
// 16-byte global loads and stores, a
// shared tile read and written with 16-byte accesses in an XOR-swizzled layout,
// and a register micro-transpose.
//
// A 16-byte chunk holds V = 16 / sizeof(T) elements (4 fp32 or 8 bf16).  The
// block (NT = 128 or 256 threads) stages a TR x TC tile, TR = V*MR rows and TC = V*MC
// columns: MR x MC micro-blocks of V x V elements, e.g. 64x64 fp32 (16 KiB) or
// 128x128 bf16 (32 KiB) for MR = MC = 16.
//
// Phase 1 (load): thread t takes chunk cc = t % MC of tile rows t / MC + k*NT/MC,
//   with 16-byte global loads (a warp reads whole MC*16-byte row segments), all
//   of them in flight before the first shared store.
// Shared layout: chunk cc of tile row r is stored at chunk position
//   cc ^ ((r / V) % 8) of that row.  A 16-byte shared access is served in
//   phases of 8 lanes; it is conflict-free when the 8 lanes hit 8 distinct
//   positions modulo 8 (each 128 bytes of a row spans all 32 banks once).
//   Phase-1 stores: 8 lanes = 8 consecutive chunks of one row -> distinct.
// Phase 2 (transpose): micro-block u = t + NT*j has A = u % MR, C = u / MR and
//   covers tile rows V*A..V*A+V-1 of chunk C.  Its V shared reads (rows V*A+m,
//   chunk C) land at positions C ^ (A % 8); the 8 lanes of a phase have 8
//   consecutive A and one C -> distinct.  The register transpose (renaming
//   for fp32, 32 byte permutes for bf16) gives V output rows V*C+m', each with
//   one chunk at output columns V*A..: consecutive lanes write consecutive
//   chunks, MR*16 contiguous bytes of an output row.
//
// This is the padded tile of "Shared memory and the bank conflict" (sections
// "Turn the tile around on chip" and "Banks") moved to 16-byte accesses: the
// +1 padding that spreads a 4-byte column walk over the banks cannot keep
// 16-byte rows aligned, so the spreading is done by the XOR swizzle instead
// ("Shared-memory tiling and bank conflicts": pad or swizzle tiles when column
// access creates bank conflicts).
//
// Misaligned sides.  With VEC_IN = false (input rows need not start on
// 16-byte boundaries) bf16 tiles that lie wholly inside the matrix read every
// row segment as the aligned 16-byte chunks covering it and cut each thread's
// chunk out of its own and the next (the next lane's, by a warp shuffle); all
// other chunks whose elements are in range (fp32, edge tiles) are loaded with
// the widest accesses their own address allows -- one 16-byte, two 8-byte or
// four 4-byte loads, single elements for bf16 rows 2 bytes past a word.  With
// SHIFT_OUT the output rows need not start on 16-byte boundaries (e.g. a row
// pitch of 12289 fp32).  For each output row, d is the number of elements
// between the tile's first column r0 and the row's next 16-byte boundary
// (32-byte for bf16 tiles of 128 rows or more; the same for every tile of the
// row), and the tile owns the output columns [r0 + d, r0 + TR + d) -- plus
// [0, d) in the first tile row -- so every store inside the matrix is a whole
// aligned chunk, which draws on V (2V) extra input rows staged below the tile
// (the halo).  fp32: lane A stores its own last V-d elements followed by the first
// d of micro-block A+1, fetched from lane A+1 with a warp shuffle or, for the
// last micro-block row, from the halo.  bf16: each lane gathers its aligned
// chunk from the shared tile, one element per input row, the shift being an
// offset in shared addresses.  Single elements remain only at the matrix edges
// (the first d columns, the columns past the last input row).
// Tiles at the matrix edge use bounds-checked element accesses except where a
// whole chunk is in range on an aligned side, or (shifted stores) where the
// tile's output row segments are complete and only its last output rows are
// missing.
#pragma once

#include "bounds.cuh"
#include "launch.cuh"
#include "tile_geom.cuh"
#include "tr_internal.h"
#include "vec_common.cuh"

#include <atomic>
#include <mutex>

namespace tr {
namespace vec {

// Elements d .. d+V-1 of the 2V-element sequence (own, next), 0 <= d < V.
template <typename T>
__device__ __forceinline__ uint4 window(const Chunk &own, const Chunk &next, int d) {
    uint32_t e[8] = {own.w[0], own.w[1], own.w[2], own.w[3],
                     next.w[0], next.w[1], next.w[2], next.w[3]};
    const int words = sizeof(T) == 4 ? d : d >> 1;  // whole-word part of the shift
    if (words & 2) {
#pragma unroll
        for (int k = 0; k < 6; ++k) e[k] = e[k + 2];
    }
    if (words & 1) {
#pragma unroll
        for (int k = 0; k < 5; ++k) e[k] = e[k + 1];
    }
    if (sizeof(T) == 2 && (d & 1)) {
        // odd 16-bit shift: high half of word k, low half of word k+1
#pragma unroll
        for (int k = 0; k < 4; ++k) e[k] = __byte_perm(e[k], e[k + 1], 0x5432);
    }
    return make_uint4(e[0], e[1], e[2], e[3]);
}

// Whether misaligned input rows of 16-bit elements are read as aligned chunks
// and realigned on chip (see the kernel).  4-byte elements keep the per-chunk
// loads: four 4-byte loads per chunk already run near the copy's rate there.
template <typename T, bool VEC_IN>
constexpr bool kRealignInput = !VEC_IN && sizeof(T) == 2;

// Shifted stores: the granule (elements) whose boundaries a tile's owned output
// columns start on, and the input rows staged below the tile (the halo) to
// fill them.  bf16 tiles of 128 rows or more own 32-byte runs, so that a
// warp's store runs cover whole 32-byte sectors (a store run that splits
// sectors costs about 4% of the rate; see phase 2); their 2V halo rows
// add 12.5% to the rows a tile reads.  Shorter bf16 tiles and fp32 tiles own
// 16-byte runs (a 16-row halo on a 64-row tile costs more than it saves:
// 16384x16384 bf16 with both pitches 16385 on 64x128 tiles, 5039 GB/s with
// 16-byte runs against 4668 with 32-byte runs).
template <typename T, int MR>
constexpr int kShiftGranule = (sizeof(T) == 2 && MR >= 16 ? 2 : 1) * VecTraits<T>::V;
template <typename T, int MR, bool SHIFT_OUT>
constexpr int kHalo = SHIFT_OUT ? kShiftGranule<T, MR> : 0;

// Resident blocks per SM that the bf16 shifted-store shapes AUTO takes (128x128 on 256
// threads, 64x128 on 128 threads) are compiled for: 64 registers, 4 and 8 blocks.  Left
// free, the compiler keeps the gathered loads of several chunks in flight with up to 126
// registers.  Measured on 16384x16384 bf16 (GB/s), output pitch 16385 / both pitches
// 16385: 5916 / 4943 at 64 registers, 5560 / 4543 at 80 (3 and 6 blocks); at 48 the loads
// spill 100-228 bytes per thread.  0 leaves every other instantiation to the compiler.
template <typename T, int MR, int MC, int NT, bool SHIFT_OUT, bool PREFETCH>
constexpr int kMinBlocks =
    SHIFT_OUT && !PREFETCH && sizeof(T) == 2 && MC == 16 && ((NT == 256 && MR == 16) || (NT == 128 && MR == 8))
        ? 65536 / (NT * 64)
        : 0;

template <typename T, int MR, int MC, int NT, bool VEC_IN, bool SHIFT_OUT, bool PREFETCH>
__global__ void __launch_bounds__(NT, (kMinBlocks<T, MR, MC, NT, SHIFT_OUT, PREFETCH>)) k_tile_vec(const T *__restrict__ in, T *__restrict__ out,
                                                 Geometry g, bool diagonal) {
    constexpr int V = VecTraits<T>::V;
    constexpr int TR = V * MR, TC = V * MC;  // tile rows / columns in elements
    constexpr int MB = MR * MC / NT;         // micro-blocks per thread
    constexpr int RPP = NT / MC;             // tile rows per load pass
    constexpr int LOADS = TR / RPP;          // chunks each thread loads
    static_assert(MR >= 8 && MR <= 32 && MC >= 8 && NT % MC == 0 && (MR * MC) % NT == 0,
                  "unsupported tile shape");
    // With shifted stores the tile also stages the input rows below it (the
    // halo): the output chunks past its last micro-block row draw on them
    // (phase 2).
    constexpr int SG = kShiftGranule<T, MR>;      // shift granule, elements
    constexpr int HALO = kHalo<T, MR, SHIFT_OUT>; // extra tile rows
    constexpr int HCH = HALO * MC;                // halo chunks
    constexpr int HL = SHIFT_OUT ? (HCH + NT - 1) / NT : 1;  // halo chunks per thread
    // Misaligned input rows of 16-bit elements in a tile that lies wholly
    // inside the matrix, halo rows included: each row segment is read as the
    // aligned 16-byte chunks that cover it -- MC by the row's own threads, one
    // more past its end by a helper thread, staged in shared memory past the
    // tile -- and every thread then cuts its chunk's elements out of its own
    // aligned chunk and the next one.  The extra bytes those
    // chunks hold belong to the input's own extent (neighbouring columns,
    // pitch padding, the row before or after) except in two tiles, which take
    // the per-chunk path: the first tile of the first plane, whose first chunk
    // may start before the input, and in the last plane a tile reading the
    // last input row whose row segments end fewer than V elements before that
    // row's end, whose last aligned chunk may reach past the input.
    constexpr bool RAW = kRealignInput<T, VEC_IN>;
    constexpr int XL = RAW ? (TR + HALO + NT - 1) / NT : 1;  // extra chunks per thread
    static_assert(!RAW || (32 % MC == 0 || MC % 32 == 0), "a row's lanes share a warp");
    static_assert(!RAW || ((HALO * MC) % NT == 0 || (HALO * MC) % 32 == 0), "halo lanes fill whole warps");
    extern __shared__ uint4 smem[];  // TR + HALO rows of MC chunks (+ one chunk per row when RAW)

    pdl_prologue();
    const int t = threadIdx.x;
    const int lcc = t % MC, lr = t / MC;
    // Debug builds: the two sides every global access is checked against.
    TR_SIDE(in_side, in, g.batch, g.rows, g.cols, g.ld_in, g.stride_in, int(sizeof(T)));
    TR_SIDE(out_side, out, g.batch, g.cols, g.rows, g.ld_out, g.stride_out, int(sizeof(T)));
    // 16-byte global accesses (streaming loads and stores).
    auto ld16 = [&](const void *p) {
        return TR_LOAD_OK(in_side, p, 16) ? __ldcs(reinterpret_cast<const uint4 *>(p))
                                          : make_uint4(0u, 0u, 0u, 0u);
    };
    auto st16 = [&](T *p, uint4 v) {
        if (TR_STORE_OK(out_side, p, 16)) __stcs(reinterpret_cast<uint4 *>(p), v);
    };

    // Whether tile (b, tr, tc) takes the aligned-chunk path.
    auto raw_tile = [&](bool full, int64_t b, int64_t tr, int64_t tc) {
        const int64_t end = (tr + 1) * TR + HALO;  // one past the last row read
        const bool first = b == 0 && tr == 0 && tc == 0;
        const bool last = b == g.batch - 1 && end >= g.rows && (tc + 1) * TC + V > g.cols;
        return RAW && full && end <= g.rows && !first && !last;
    };
    auto aligned_chunk = [&](const T *p) {
        const uint4 *q = reinterpret_cast<const uint4 *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(15));
        return TR_LOAD_IN_EXTENT(in_side, q, 16) ? __ldcs(q) : make_uint4(0u, 0u, 0u, 0u);
    };

    // Phase 1a: this thread's chunks of tile `tile`, global -> registers, all
    // loads issued before any is used.
    Chunk ld[LOADS];
    Chunk hl[HL];
    Chunk xl[XL];
    auto load_tile = [&](int64_t tile) {
        int64_t b, tr, tc;
        split_tile(g, tile, diagonal, b, tr, tc);
        const T *src = in + b * g.stride_in;
        const int64_t r0 = tr * TR, c0 = tc * TC;
        const bool full = (r0 + TR <= g.rows) && (c0 + TC <= g.cols);
        const int64_t gc = c0 + lcc * V;
        bool raw = false;
        if constexpr (RAW) {
            raw = raw_tile(full, b, tr, tc);
            if (raw) {
                // The aligned chunk holding this thread's first element, and
                // for helper rows (tile and halo rows) the aligned chunk past
                // the segment (not needed when the segment ends on a 16-byte
                // boundary, i.e. when the row is aligned).
#pragma unroll
                for (int k = 0; k < LOADS; ++k)
                    ld[k].v = aligned_chunk(src + (r0 + lr + RPP * k) * g.ld_in + gc);
#pragma unroll
                for (int k = 0; k < XL; ++k) {
                    const int rr = t + NT * k;
                    if ((TR + HALO) % NT != 0 && rr >= TR + HALO) continue;
                    const T *p = src + (r0 + rr) * g.ld_in + c0 + TC;
                    if (reinterpret_cast<uintptr_t>(p) & 15u) xl[k].v = aligned_chunk(p);
                }
            }
        }
        if (full && VEC_IN) {
#pragma unroll
            for (int k = 0; k < LOADS; ++k)
                ld[k].v = ld16(src + (r0 + lr + RPP * k) * g.ld_in + gc);
        } else if (!raw) {
#pragma unroll
            for (int k = 0; k < LOADS; ++k) {
                const int64_t gr = r0 + lr + RPP * k;
                if (VEC_IN && gr < g.rows && gc + V <= g.cols) {
                    ld[k].v = ld16(src + gr * g.ld_in + gc);
                } else if (!VEC_IN && gr < g.rows && gc + V <= g.cols) {
                    // A whole chunk in range on a misaligned side (row starts
                    // differ from row to row): the widest loads this chunk's
                    // own address allows, touching only its own elements.
                    const T *p = src + gr * g.ld_in + gc;
                    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
                    if (!TR_LOAD_OK(in_side, p, 16)) {
                        ld[k].v = make_uint4(0u, 0u, 0u, 0u);
                    } else if ((a & 15u) == 0) {
                        ld[k].v = __ldcs(reinterpret_cast<const uint4 *>(p));
                    } else if ((a & 7u) == 0) {
                        const uint2 lo = __ldcs(reinterpret_cast<const uint2 *>(p));
                        const uint2 hi = __ldcs(reinterpret_cast<const uint2 *>(p) + 1);
                        ld[k].v = make_uint4(lo.x, lo.y, hi.x, hi.y);
                    } else if (sizeof(T) == 4 || (a & 3u) == 0) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ld[k].w[q] = __ldcs(reinterpret_cast<const unsigned int *>(p) + q);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ld[k].w[q] = uint32_t(p[2 * q]) | (uint32_t(p[2 * q + 1]) << 16);
                    }
                } else {
                    T e[V];
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        e[q] = (gr < g.rows && gc + q < g.cols &&
                                TR_LOAD_OK(in_side, src + gr * g.ld_in + gc + q, int(sizeof(T))))
                                   ? src[gr * g.ld_in + gc + q]
                                   : T(0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if constexpr (sizeof(T) == 4)
                            ld[k].w[q] = uint32_t(e[q]);
                        else
                            ld[k].w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                    }
                }
            }
        }
        if constexpr (SHIFT_OUT) {
            // Halo: input rows r0+TR .. r0+TR+V-1, bounds-checked (they lie
            // past the matrix at its last tile rows; zeros are never stored).
#pragma unroll
            for (int k = 0; k < HL; ++k) {
                const int h = t + NT * k;
                if (HCH % NT != 0 && h >= HCH) continue;
                const int64_t gr = r0 + TR + h / MC;
                const int64_t hc = c0 + (h % MC) * V;
                if (raw) {
                    hl[k].v = aligned_chunk(src + gr * g.ld_in + hc);
                } else if (VEC_IN && gr < g.rows && hc + V <= g.cols) {
                    hl[k].v = ld16(src + gr * g.ld_in + hc);
                } else {
                    T e[V];
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        e[q] = (gr < g.rows && hc + q < g.cols &&
                                TR_LOAD_OK(in_side, src + gr * g.ld_in + hc + q, int(sizeof(T))))
                                   ? src[gr * g.ld_in + hc + q]
                                   : T(0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if constexpr (sizeof(T) == 4)
                            hl[k].w[q] = uint32_t(e[q]);
                        else
                            hl[k].w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                    }
                }
            }
        }
    };

    // With PREFETCH the grid is persistent and the loads of a block's next
    // tile are issued as soon as the current tile sits in shared memory, so
    // they are in flight while the current tile is transposed and stored
    // ("Shared-memory tiling and bank conflicts", "Protect tile phases": one
    // stage loads future data while another is consumed).  The registers are
    // the second buffer; the shared tile is reused once every thread passed
    // the barrier that ends the previous tile's reads.
    if (PREFETCH && blockIdx.x < g.total) load_tile(blockIdx.x);

    for (int64_t tile = blockIdx.x; tile < g.total; tile += gridDim.x) {
        int64_t b, tr, tc;
        split_tile(g, tile, diagonal, b, tr, tc);
        T *dst = out + b * g.stride_out;
        const int64_t r0 = tr * TR, c0 = tc * TC;
        const bool full = (r0 + TR <= g.rows) && (c0 + TC <= g.cols);

        if (!PREFETCH) load_tile(tile);
        if (tile != blockIdx.x) __syncthreads();  // previous tile fully read
        if (RAW && raw_tile(full, b, tr, tc)) {
            // Realign: each thread takes elements s .. s+V-1 of (own chunk,
            // next chunk), s being the row's offset from its 16-byte boundary.
            // The next chunk is the next lane's own (a warp shuffle), except
            // for a row's last lane, which takes the chunk past the segment
            // that the helper thread of that row staged in shared memory past
            // the tile (consecutive lanes, consecutive 16-byte slots: no
            // conflicts).  The tile's own chunks never go through shared
            // memory unshifted.
            uint4 *ext = smem + (TR + HALO) * MC;  // one chunk per tile (and halo) row
#pragma unroll
            for (int k = 0; k < XL; ++k) {
                const int rr = t + NT * k;
                if ((TR + HALO) % NT != 0 && rr >= TR + HALO) continue;
                ext[rr] = xl[k].v;
            }
            __syncthreads();
            // Byte offsets from 16-byte boundaries: row lr's, and the step to
            // the thread's next row (low bits of the addresses suffice).
            const uint32_t a0 = uint32_t(reinterpret_cast<uintptr_t>(
                in + b * g.stride_in + (r0 + lr) * g.ld_in + c0));
            const uint32_t step = uint32_t(g.ld_in) * uint32_t(RPP * sizeof(T));
#pragma unroll
            for (int k = 0; k < LOADS; ++k) {
                const int sh = int(((a0 + uint32_t(k) * step) & 15u) / sizeof(T));
                Chunk nb;
#pragma unroll
                for (int q = 0; q < 4; ++q) nb.w[q] = __shfl_down_sync(0xffffffffu, ld[k].w[q], 1);
                if (lcc == MC - 1) nb.v = ext[lr + RPP * k];
                ld[k].v = window<T>(ld[k], nb, sh);
            }
            if constexpr (SHIFT_OUT) {
#pragma unroll
                for (int k = 0; k < HL; ++k) {
                    const int h = t + NT * k;  // whole warps run past HCH (it is a multiple of 32)
                    if (HCH % NT != 0 && h >= HCH) continue;
                    const int r = TR + h / MC;
                    const int sh = int((reinterpret_cast<uintptr_t>(
                                            in + b * g.stride_in + (r0 + r) * g.ld_in + c0) &
                                        15u) /
                                       sizeof(T));
                    Chunk nb;
#pragma unroll
                    for (int q = 0; q < 4; ++q) nb.w[q] = __shfl_down_sync(0xffffffffu, hl[k].w[q], 1);
                    if (h % MC == MC - 1) nb.v = ext[r];
                    hl[k].v = window<T>(hl[k], nb, sh);
                }
            }
        }
        // Phase 1b: registers -> swizzled shared tile.
#pragma unroll
        for (int k = 0; k < LOADS; ++k) {
            const int r = lr + RPP * k;
            smem[r * MC + (lcc ^ ((r / V) & 7))] = ld[k].v;
        }
        if constexpr (SHIFT_OUT) {
#pragma unroll
            for (int k = 0; k < HL; ++k) {
                const int h = t + NT * k;
                if (HCH % NT != 0 && h >= HCH) continue;
                const int r = TR + h / MC;
                smem[r * MC + ((h % MC) ^ ((r / V) & 7))] = hl[k].v;
            }
        }
        __syncthreads();
        if (PREFETCH && tile + gridDim.x < g.total) load_tile(tile + gridDim.x);

        // ---- phase 2, shifted output rows of 16-bit elements, when every
        // output row segment of the tile is complete (the tile may still stop
        // short of the last output rows).  Let d be the number of elements from
        // an output row's column r0 to its next boundary of SG elements (32
        // bytes for tiles of 128 rows or more, else 16; d < SG): the tile owns
        // the output columns [r0 + d, r0 + TR + d) of the row (and [0, d) in the
        // first tile row), i.e. whole aligned chunks (whose store runs start on
        // 32-byte sector boundaries when SG = 2V), and the chunk at r0 + d + V*A
        // holds input rows r0 + d + V*A .. + V-1 of the row's input column.
        // (With 16-byte boundaries instead, every 128-byte store run splits two
        // sectors: 16384x16384 bf16 transposed with the aligned path into an
        // output pitch of 16392 runs at 6573 GB/s, at 16400 at 6878.)  Each lane
        // gathers its chunk straight from the shared tile, one element per
        // input row (the SG halo rows below the tile supply the last d), so the
        // shift is only an offset in shared addresses.  Lane map per warp
        // instruction: RUN consecutive chunks A of KL = 32 / RUN output rows,
        // the rows' elements in distinct words of the chunk; RUN = 16 where the
        // tile has 16 chunks per output row segment, so that a warp stores
        // 256-byte runs, else 8.  Each element read hits bank 4 * (chunk
        // position) + (its word in the chunk), and 8 lanes of one output row
        // see 8 distinct chunk positions (rows V*A.. are V apart and the
        // swizzle XORs row / V): with RUN = 8 the 32 reads fall on 32 distinct
        // banks, with RUN = 16 two lanes share each bank (2 wavefronts per
        // read).  The longer store runs win: 16384x16384 bf16 with output pitch
        // 16385 runs at 6330 GB/s with RUN = 16 against 6195 with RUN = 8
        // (conflict-free).  d depends only on the plane and on the output
        // row's place in its group of SG (the tile's corner moves a row start
        // by multiples of SG elements).  4-byte elements keep the register
        // window of the micro-block phase below: with whole words to move it
        // costs less than four gathered loads per chunk (fp32 12289x7919,
        // output pitch 12289: 6778 GB/s against 6540 gathered), while for bf16
        // the window's byte permutes and the halo lane's element reads cost
        // more (16384x16384, output pitch 16385: 5921 gathered against 5567).
        if constexpr (SHIFT_OUT && sizeof(T) == 2) {
            if (r0 + TR <= g.rows) {
                const T *sm = reinterpret_cast<const T *>(smem);
                const int s0 = int((reinterpret_cast<uintptr_t>(dst) / sizeof(T)) % SG);
                const int L = int(g.ld_out % SG);
                constexpr int RUN = MR >= 16 ? 16 : 8;        // consecutive chunks of a row per instruction
                constexpr int KL = 32 / RUN;                  // output rows per instruction
                constexpr int PAR = V / KL;                   // output rows of a group a lane takes
                const int k = t % KL, a = (t / KL) % RUN, w = t >> 5;
                constexpr int ABLK = MR / RUN;                // runs per output row segment
                constexpr int STEPS = MC * PAR * ABLK;        // warp steps per tile
#pragma unroll
                for (int j = 0; j < STEPS / (NT / 32); ++j) {
                    const int step = w + (NT / 32) * j;
                    const int C = step / (PAR * ABLK);
                    const int par = (step / ABLK) % PAR;
                    const int A = (step % ABLK) * RUN + a;
                    const int cl = PAR * k + par;         // output row within the group of V
                    const int64_t orow = c0 + V * C + cl;
                    if (!full && orow >= g.cols) continue;
                    // row start offset within its granule (c0 is a multiple of SG)
                    const int s = (s0 + (V * C + cl) * L) % SG, d = (SG - s) % SG;
                    T e[V];
#pragma unroll
                    for (int q = 0; q < V; ++q) {
                        const int r = V * A + d + q;  // tile row (the halo from TR on)
                        e[q] = sm[(r * MC + (C ^ ((r / V) & 7))) * V + cl];
                    }
                    Chunk v;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if constexpr (sizeof(T) == 4)
                            v.w[q] = uint32_t(e[q]);
                        else
                            v.w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                    }
                    T *row = dst + orow * g.ld_out;
                    const int64_t wc = r0 + V * A + d;  // first column of the aligned chunk
                    if (wc + V <= g.rows) {
                        st16(row + wc, v.v);
                    } else {
                        // the halo ran past the last input row
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            if (wc + q < g.rows && TR_STORE_OK(out_side, row + wc + q, int(sizeof(T))))
                                row[wc + q] = e[q];
                    }
                    if (tr == 0 && A == 0) {
                        // columns [0, d): input rows 0 .. d-1
#pragma unroll
                        for (int q = 0; q < SG; ++q)
                            if (q < d && TR_STORE_OK(out_side, row + q, int(sizeof(T))))
                                row[q] = sm[(q * MC + (C ^ ((q / V) & 7))) * V + cl];
                    }
                }
                continue;
            }
        }

        // ---- phase 2: micro-blocks -> registers -> transpose -> global
#pragma unroll
        for (int j = 0; j < MB; ++j) {
            const int u = t + NT * j;
            const int A = u % MR, C = u / MR;
            Chunk x[V], y[V];
#pragma unroll
            for (int m = 0; m < V; ++m) x[m].v = smem[(V * A + m) * MC + (C ^ (A & 7))];
            micro_transpose(x, y);
            const int64_t oc = r0 + V * A;  // first output column of this lane's chunk
            if (full && !SHIFT_OUT) {
#pragma unroll
                for (int m = 0; m < V; ++m) st16(dst + (c0 + V * C + m) * g.ld_out + oc, y[m].v);
            } else if (SHIFT_OUT && sizeof(T) == 4 && r0 + TR <= g.rows) {
                // Every output row segment of the tile is complete (the tile may
                // still stop short of the last output rows).  For an output row
                // whose first 16-byte boundary lies d elements past column r0,
                // the tile owns columns [r0 + d, r0 + TR + d) (and [0, d) in
                // the first tile row): lane A stores the aligned chunk made of
                // its own last V-d elements and the first d of micro-block A+1,
                // taken from lane A+1 by a warp shuffle or, for A = MR-1, from
                // the halo micro-block below the tile.  The shuffles run on
                // every lane.
#pragma unroll
                for (int m = 0; m < V; ++m) {
                    const int64_t orow = c0 + V * C + m;
                    T *row = dst + orow * g.ld_out;
                    Chunk nb;
#pragma unroll
                    for (int k = 0; k < 4; ++k) nb.w[k] = __shfl_down_sync(0xffffffffu, y[m].w[k], 1);
                    if (A == MR - 1) {
                        // Column V*C+m of the halo rows TR .. TR+V-1, read as
                        // single elements (one lane per micro-block row).
                        const T *sm = reinterpret_cast<const T *>(smem);
                        T e[V];
#pragma unroll
                        for (int q = 0; q < V; ++q) e[q] = sm[((TR + q) * MC + (C ^ (MR & 7))) * V + m];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if constexpr (sizeof(T) == 4)
                                nb.w[q] = uint32_t(e[q]);
                            else
                                nb.w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                        }
                    }
                    if (!full && orow >= g.cols) continue;
                    const int s = int((reinterpret_cast<uintptr_t>(row + r0) / sizeof(T)) % V);
                    const int d = (V - s) % V;  // elements before the first 16-byte boundary
                    if (d == 0) {
                        st16(row + oc, y[m].v);
                        continue;
                    }
                    const int64_t wc = oc + d;  // first column of the aligned chunk
                    Chunk wv;
                    wv.v = window<T>(y[m], nb, d);
                    if (wc + V <= g.rows) {
                        st16(row + wc, wv.v);
                    } else {
                        // the halo ran past the last input row
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            if (wc + q < g.rows && TR_STORE_OK(out_side, row + wc + q, int(sizeof(T))))
                                row[wc + q] = elem<T>(wv, q);
                    }
                    if (tr == 0 && A == 0) {
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            if (q < d && TR_STORE_OK(out_side, row + q, int(sizeof(T))))
                                row[q] = elem<T>(y[m], q);
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < V; ++m) {
                    const int64_t orow = c0 + V * C + m;
                    if (orow >= g.cols) break;
                    T *row = dst + orow * g.ld_out;
                    if (!SHIFT_OUT && oc + V <= g.rows) {
                        st16(row + oc, y[m].v);
                    } else {
                        // With shifted stores the first d columns of the segment
                        // belong to the tile above (it wrote them from its halo).
                        int64_t lo = 0;
                        if constexpr (SHIFT_OUT) {
                            if (tr > 0) {
                                const int s = int((reinterpret_cast<uintptr_t>(row + r0) / sizeof(T)) % SG);
                                lo = r0 + (SG - s) % SG;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            if (oc + q < g.rows && oc + q >= lo &&
                                TR_STORE_OK(out_side, row + oc + q, int(sizeof(T))))
                                row[oc + q] = elem<T>(y[m], q);
                    }
                }
            }
        }
    }
}

// Shared memory of one instantiation; above 48 KiB it needs an opt-in, done
// once per device.
// One instantiation's launch.  Above 48 KiB of shared memory the kernel needs
// an opt-in, and a persistent grid needs the number of resident blocks per
// SM: both are found once per device and cached.
template <typename T, int MR, int MC, int NT, bool VI, bool SO, bool PF>
cudaError_t launch_one(const Problem &p, bool diagonal) {
    constexpr int V = VecTraits<T>::V;
    // The tile (+ halo rows), or when misaligned input rows are realigned on
    // chip the tile plus one staged chunk per row.
    constexpr size_t tile_chunks = size_t(V * MR + kHalo<T, MR, SO>) * MC;
    constexpr size_t raw_chunks = kRealignInput<T, VI> ? size_t(V * MR + kHalo<T, MR, SO>) * (MC + 1) : 0;
    constexpr size_t smem = (tile_chunks > raw_chunks ? tile_chunks : raw_chunks) * 16;
    auto kern = k_tile_vec<T, MR, MC, NT, VI, SO, PF>;
    // Resident blocks per SM on each device; 0 = not set up on that device yet.
    static std::atomic<int> resident[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int fit = resident[dev].load(std::memory_order_acquire);
    if (!fit) {
        std::lock_guard<std::mutex> lock(mu);
        fit = resident[dev].load(std::memory_order_relaxed);
        if (!fit) {
            if (smem > 48 * 1024) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
                if (e != cudaSuccess) return e;
            }
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, smem);
            if (e != cudaSuccess) return e;
            fit = n > 0 ? n : 1;
            resident[dev].store(fit, std::memory_order_release);
        }
    }
    const Geometry g = make_geometry(p, V * MR, V * MC);
    int64_t grid = g.total;
    if (PF) {
        const int64_t cap = int64_t(sm_count()) * fit;
        if (grid > cap) grid = cap;
    }
    return launch_pdl(kern, dim3(grid_blocks(grid)), dim3(NT), smem, p.stream,
                      static_cast<const T *>(p.in), static_cast<T *>(p.out), g, diagonal);
}

template <typename T, int MR, int MC, int NT, bool PF>
cudaError_t launch_align(const Problem &p, bool vec_in, bool vec_out, bool diagonal) {
    if (vec_in && vec_out) return launch_one<T, MR, MC, NT, true, false, PF>(p, diagonal);
    if (vec_in) return launch_one<T, MR, MC, NT, true, true, PF>(p, diagonal);
    if (vec_out) return launch_one<T, MR, MC, NT, false, false, PF>(p, diagonal);
    return launch_one<T, MR, MC, NT, false, true, PF>(p, diagonal);
}

// Supported shapes (micro-blocks MR x MC, threads NT).  256 threads for every
// shape; 128 threads for the smaller tiles, which doubles the loads each
// thread keeps in flight and lets more blocks share an SM.
template <typename T, bool PF>
cudaError_t launch_typed(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                         const char **why) {
    constexpr int V = VecTraits<T>::V;
    const bool diag = cfg.tile_order == 1;
    const int nt = cfg.threads ? cfg.threads : 256;
    int mr = cfg.tile_rows ? cfg.tile_rows / V : 16;
    int mc = cfg.tile_cols ? cfg.tile_cols / V : 16;
    if ((cfg.tile_rows % V) || (cfg.tile_cols % V)) mr = mc = 0;
    if (nt == 256) {
        if (mr == 16 && mc == 16) return launch_align<T, 16, 16, 256, PF>(p, vec_in, vec_out, diag);
        if (mr == 32 && mc == 8) return launch_align<T, 32, 8, 256, PF>(p, vec_in, vec_out, diag);
        if (mr == 32 && mc == 16) return launch_align<T, 32, 16, 256, PF>(p, vec_in, vec_out, diag);
        if (mr == 16 && mc == 32) return launch_align<T, 16, 32, 256, PF>(p, vec_in, vec_out, diag);
        if constexpr (sizeof(T) == 4) {
            if (mr == 32 && mc == 32) return launch_align<T, 32, 32, 256, PF>(p, vec_in, vec_out, diag);
        }
    } else if (nt == 128) {
        if (mr == 16 && mc == 16) return launch_align<T, 16, 16, 128, PF>(p, vec_in, vec_out, diag);
        if (mr == 8 && mc == 16) return launch_align<T, 8, 16, 128, PF>(p, vec_in, vec_out, diag);
        if constexpr (sizeof(T) == 4) {
            if (mr == 32 && mc == 16) return launch_align<T, 32, 16, 128, PF>(p, vec_in, vec_out, diag);
        }
    } else if (nt == 64) {
        if (mr == 8 && mc == 16) return launch_align<T, 8, 16, 64, PF>(p, vec_in, vec_out, diag);
        if (mr == 16 && mc == 8) return launch_align<T, 16, 8, 64, PF>(p, vec_in, vec_out, diag);
    } else if (nt == 32) {
        if (mr == 8 && mc == 8) return launch_align<T, 8, 8, 32, PF>(p, vec_in, vec_out, diag);
    }
    *why = sizeof(T) == 4
               ? "vector tile: 256 threads take 64x64, 128x32, 128x64, 64x128 or 128x128 fp32 tiles; "
                 "128 threads 64x64, 32x64 or 128x64; 64 threads 32x64 or 64x32; 32 threads 32x32"
               : "vector tile: 256 threads take 128x128, 256x64, 256x128 or 128x256 bf16 tiles; "
                 "128 threads 128x128 or 64x128; 64 threads 64x128 or 128x64; 32 threads 64x64";
    return cudaErrorInvalidValue;
}

}  // namespace vec
}  // namespace tr
