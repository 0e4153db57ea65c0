// In-place transpose of square planes: data[b][j][i] <- data[b][i][j].
//
// The out-of-place kernels read one tile and write its transpose elsewhere.
// In place, the transpose of tile (ti, tj) lands where tile (tj, ti) lives, so
// one block owns each unordered pair of tiles: it reads BOTH tiles into two
// swizzled shared tiles (whole tiles by asynchronous 16-byte copies, edge
// tiles through registers), and only after the barrier writes each one's
// transpose over the other ("Shared memory and the bank conflict", "The
// barrier": nothing may be written before every thread's reads are in).  A
// diagonal tile is its own partner.  No other block reads or writes either
// tile, so blocks never race.
//
// Layout and lane mapping are those of the vectorised swizzled tile
// (tile_vec_kernel.cuh):
// a 16V x 16V tile (64x64 fp32, 128x128 bf16), chunk cc of tile row r stored at
// chunk position cc ^ ((r / V) % 8), 256 threads, 16-byte loads and stores and a
// register micro-transpose; VEC = false moves single elements (any alignment).
//
// Blocks walk the pairs (ti <= tj) of each plane's upper triangle of tiles (T
// tiles per side, T (T + 1) / 2 pairs), tile column by tile column: pair index
// tj (tj + 1) / 2 + ti.  Walking the whole T x T grid and letting the blocks
// below the diagonal exit at once costs a launch slot per skipped block:
// 8192x8192 fp32 in place runs at 6330 GB/s that way against 6427 with the
// triangle, 16384x16384 bf16 at 6331 against 6483.
#include "bounds.cuh"
#include "launch.cuh"
#include "ptx.cuh"
#include "tile_geom.cuh"
#include "tr_internal.h"
#include "vec_common.cuh"

#include <atomic>
#include <mutex>

namespace tr {
namespace {

struct InplaceGeom {
    int64_t batch, n, ld, stride;
    int64_t tiles;  // tiles per side
    int64_t pairs;  // tile pairs per plane: tiles * (tiles + 1) / 2
    int64_t total;  // batch * pairs
};

// Pair index p (< tiles * (tiles + 1) / 2) -> tiles (ti <= tj), p = tj (tj + 1) / 2 + ti.
// tj is the floor of the root of x (x + 1) / 2 = p, taken in float.  For p < 2^32
// (tj < 92682) the float root is within 0.02 of the true one, so one step up or
// down corrects it, in 32-bit arithmetic (every triangular number compared with
// p stays below 2^32; halving the even factor first keeps the product there too).
__device__ __forceinline__ uint32_t triangle32(uint32_t n) {
    return (n & 1u) ? n * ((n + 1u) >> 1) : (n >> 1) * (n + 1u);
}
__device__ __forceinline__ void split_pair32(uint32_t p, uint32_t &ti, uint32_t &tj) {
    tj = uint32_t((sqrtf(8.0f * float(p) + 1.0f) - 1.0f) * 0.5f);
    tj -= triangle32(tj) > p ? 1u : 0u;
    tj += triangle32(tj + 1u) <= p ? 1u : 0u;
    ti = p - triangle32(tj);
}
// Any size: the same root, corrected by as many steps as it takes.
__device__ __forceinline__ void split_pair64(int64_t p, int64_t &ti, int64_t &tj) {
    tj = int64_t((sqrtf(8.0f * float(p) + 1.0f) - 1.0f) * 0.5f);
    while (tj > 0 && tj * (tj + 1) / 2 > p) --tj;
    while ((tj + 1) * (tj + 2) / 2 <= p) ++tj;
    ti = p - tj * (tj + 1) / 2;
}

// Resident blocks per SM the aligned fp32 kernel is compiled for: 6 (40
// registers, 32 KiB of shared memory each); 0 leaves the others to the compiler.
template <typename T, bool VEC>
constexpr int kInplaceMinBlocks = VEC && sizeof(T) == 4 ? 6 : 0;

// BIG: more than 2^32 tile pairs in the launch (64-bit pair arithmetic, kept
// out of the common instantiations, whose registers it would raise).
template <typename T, bool VEC, bool BIG>
__global__ void __launch_bounds__(256, (kInplaceMinBlocks<T, VEC>)) k_inplace(T *__restrict__ data,
                                                                            InplaceGeom g) {
    constexpr int V = VecTraits<T>::V;
    constexpr int TILE = 16 * V;
    constexpr int LOADS = V;        // 16 tile rows per load pass, TILE rows
    extern __shared__ uint4 smem[]; // two tiles of TILE rows x 16 chunks
    uint4 *tile0 = smem, *tile1 = smem + TILE * 16;
    pdl_prologue();

    const int t = threadIdx.x;
    const int lcc = t & 15, lr = t >> 4;  // phase 1: chunk and first row
    const int A = t & 15, C = t >> 4;     // phase 2: micro-block
    // Debug builds: every load and store must touch logical elements only.
    TR_SIDE(side, data, g.batch, g.n, g.n, g.ld, g.stride, int(sizeof(T)));

    bool first = true;
    for (int64_t w = blockIdx.x; w < g.total; w += gridDim.x) {
        int64_t b, ti, tj;
        if constexpr (!BIG) {  // 32-bit arithmetic is far cheaper than 64-bit
            const uint32_t w32 = uint32_t(w), pp = uint32_t(g.pairs);
            const uint32_t bb = w32 / pp;
            uint32_t i, j;
            split_pair32(w32 - bb * pp, i, j);
            b = bb;
            ti = i;
            tj = j;
        } else {
            b = w / g.pairs;
            split_pair64(w - b * g.pairs, ti, tj);
        }
        T *plane = data + b * g.stride;
        const bool diag = ti == tj;
        const int64_t r0 = ti * TILE, c0 = tj * TILE;  // tile (ti, tj); partner at (c0, r0)
        const bool full = r0 + TILE <= g.n && c0 + TILE <= g.n;

        // Phase 1: both tiles into shared memory.  Whole tiles on a 16-byte
        // aligned side go straight from global memory into their swizzled
        // slots with asynchronous 16-byte copies, so no register holds data
        // in flight and the transpose phase sets the register budget (fp32:
        // 6 blocks/SM instead of 4 with both tiles' loads in registers).  Edge
        // tiles and misaligned sides go through registers, the second tile's
        // loads after the first tile is staged.
        if (VEC && full) {
            if (!first) __syncthreads();  // previous pair fully read from shared memory
            first = false;
#pragma unroll
            for (int k = 0; k < LOADS; ++k) {
                const int r = lr + 16 * k;
                const T *p = plane + (r0 + r) * g.ld + c0 + lcc * V;
                if (TR_LOAD_OK(side, p, 16)) ptx::cp_async_16(tile0 + r * 16 + (lcc ^ ((r / V) & 7)), p);
            }
            if (!diag) {
#pragma unroll
                for (int k = 0; k < LOADS; ++k) {
                    const int r = lr + 16 * k;
                    const T *p = plane + (c0 + r) * g.ld + r0 + lcc * V;
                    if (TR_LOAD_OK(side, p, 16)) ptx::cp_async_16(tile1 + r * 16 + (lcc ^ ((r / V) & 7)), p);
                }
            }
            ptx::cp_async_wait_all();
        } else {
            Chunk x0[LOADS];
            auto load = [&](int64_t rr0, int64_t cc0) {
                const int64_t gc = cc0 + lcc * V;
#pragma unroll
                for (int k = 0; k < LOADS; ++k) {
                    const int64_t gr = rr0 + lr + 16 * k;
                    if (VEC && gr < g.n && gc + V <= g.n) {
                        const T *p = plane + gr * g.ld + gc;
                        x0[k].v = TR_LOAD_OK(side, p, 16) ? *reinterpret_cast<const uint4 *>(p)
                                                          : make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        T e[V];
#pragma unroll
                        for (int q = 0; q < V; ++q)
                            e[q] = (gr < g.n && gc + q < g.n &&
                                    TR_LOAD_OK(side, plane + gr * g.ld + gc + q, int(sizeof(T))))
                                       ? plane[gr * g.ld + gc + q]
                                       : T(0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if constexpr (sizeof(T) == 4)
                                x0[k].w[q] = uint32_t(e[q]);
                            else
                                x0[k].w[q] = uint32_t(e[2 * q]) | (uint32_t(e[2 * q + 1]) << 16);
                        }
                    }
                }
            };
            auto stage = [&](uint4 *tile) {
#pragma unroll
                for (int k = 0; k < LOADS; ++k) {
                    const int r = lr + 16 * k;
                    tile[r * 16 + (lcc ^ ((r / V) & 7))] = x0[k].v;
                }
            };
            load(r0, c0);
            if (!first) __syncthreads();  // previous pair fully read from shared memory
            first = false;
            stage(tile0);
            if (!diag) {
                asm volatile("" ::: "memory");  // keep the second tile's loads after these stores
                load(c0, r0);
                stage(tile1);
            }
        }
        __syncthreads();  // every read of both tiles is in before any write

        // Phase 2: tile0 (at r0, c0) goes to (c0, r0); tile1 (at c0, r0) to (r0, c0).
        auto store = [&](const uint4 *tile, int64_t dr0, int64_t dc0) {
            Chunk xv[V], yv[V];
#pragma unroll
            for (int m = 0; m < V; ++m) xv[m].v = tile[(V * A + m) * 16 + (C ^ (A & 7))];
            micro_transpose(xv, yv);
            const int64_t oc = dc0 + V * A;
#pragma unroll
            for (int m = 0; m < V; ++m) {
                const int64_t orow = dr0 + V * C + m;
                if (!full && orow >= g.n) break;
                T *row = plane + orow * g.ld;
                if (VEC && (full || oc + V <= g.n)) {
                    if (TR_STORE_OK(side, row + oc, 16))
                        __stcs(reinterpret_cast<uint4 *>(row + oc), yv[m].v);  // streaming store
                } else {
#pragma unroll
                    for (int q = 0; q < V; ++q)
                        if (oc + q < g.n && TR_STORE_OK(side, row + oc + q, int(sizeof(T))))
                            row[oc + q] = elem<T>(yv[m], q);
                }
            }
        };
        store(tile0, c0, r0);
        if (!diag) store(tile1, r0, c0);
    }
}

template <typename T, bool VEC, bool BIG>
cudaError_t launch_one(T *data, const InplaceGeom &g, cudaStream_t stream) {
    constexpr int V = VecTraits<T>::V;
    constexpr size_t smem = 2 * size_t(16 * V) * 16 * 16;
    auto kern = k_inplace<T, VEC, BIG>;
    if (smem > 48 * 1024) {
        static std::atomic<bool> opted[64];  // per device, zero-initialised (static)
        static std::mutex mu;
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!opted[dev].load(std::memory_order_acquire)) {
            std::lock_guard<std::mutex> lock(mu);
            if (!opted[dev].load(std::memory_order_relaxed)) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
                if (e != cudaSuccess) return e;
                opted[dev].store(true, std::memory_order_release);
            }
        }
    }
    return launch_pdl(kern, dim3(grid_blocks(g.total)), dim3(256), smem, stream, data, g);
}

template <typename T, bool VEC>
cudaError_t launch_typed(T *data, const InplaceGeom &g, cudaStream_t stream) {
    return g.total <= 0xFFFFFFFFll ? launch_one<T, VEC, false>(data, g, stream)
                                   : launch_one<T, VEC, true>(data, g, stream);
}

}  // namespace

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_inplace)

cudaError_t launch_inplace(void *data, int esize, int64_t batch, int64_t n, int64_t ld,
                           int64_t stride, cudaStream_t stream) {
    const int V = 16 / esize;
    InplaceGeom g{batch, n, ld, stride, 0, 0, 0};
    g.tiles = (n + 16 * V - 1) / (16 * V);
    g.pairs = g.tiles * (g.tiles + 1) / 2;
    g.total = batch * g.pairs;
    const bool vec = side_aligned16(data, ld, stride, batch, esize);
    if (esize == 4)
        return vec ? launch_typed<uint32_t, true>(static_cast<uint32_t *>(data), g, stream)
                   : launch_typed<uint32_t, false>(static_cast<uint32_t *>(data), g, stream);
    return vec ? launch_typed<uint16_t, true>(static_cast<uint16_t *>(data), g, stream)
               : launch_typed<uint16_t, false>(static_cast<uint16_t *>(data), g, stream);
}

}  // namespace tr
