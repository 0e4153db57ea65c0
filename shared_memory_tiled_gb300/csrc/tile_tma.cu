// TMA transpose: tiles move between global and shared memory with
// cp.async.bulk.tensor in the hardware's 128-byte swizzle, and the threads only
// turn each tile around on chip.
//
// Tile: 16V x 16V elements with V = 16 / sizeof(T) elements per 16-byte chunk
// (64x64 fp32, 128x128 bf16).  TMA boxes are 128 bytes wide (the widest box
// the 128-byte swizzle allows), so an input tile arrives as two boxes of 16V
// rows x 8 chunks (input columns 0..8V-1 and 8V..16V-1) and the output tile
// leaves as two boxes of 16V output rows x 8 chunks (input rows 0..8V-1 and
// 8V..16V-1).  In a 1024-byte aligned box with 128-byte rows the swizzle puts
// chunk k of row r at chunk position k ^ (r % 8).
//
// Each of the 256 threads owns one V x V micro-block: tile rows V*A..V*A+V-1
// (A < 16) and chunk C (< 16).  It reads V chunks with 16-byte shared loads,
// transposes them in registers (pure renaming for fp32, byte permutes for
// bf16) and writes V chunks of the output tile.  With a = A % 8, c = C % 8:
//   read  row V*A+m, chunk c   -> position c ^ ((V*A+m) % 8)
//   write row V*C+m', chunk a  -> position a ^ ((V*C+m') % 8)
// A 16-byte shared access is served 8 lanes at a time, and is conflict-free
// when those 8 lanes hit 8 distinct positions.  The 8 lanes of one phase take
// the micro-blocks (a, c) = (x ^ s, x), x = 0..7, for one s: for bf16 both
// maps reduce to c ^ m and a ^ m' (distinct because c and a are); for fp32
// they are x ^ 4*((x^s) & 1) ^ m and x ^ s ^ 4*(x & 1) ^ m', each a bijection
// of x.  So every shared access of the kernel is conflict-free on its own.
// Nsight's bank-conflict counter still reads 7-28% extra wavefronts here: it
// also charges an LSU access for the cycles it waits while a TMA box load
// writes, or a box store reads, the same banks (the LSU's shared stores take
// the extra cycles when only the box loads run, its loads when only the box
// stores run; with neither, the kernel's own accesses cost 0-3%).
//
// Pipeline (per persistent CTA, tiles blockIdx.x, +gridDim.x, ...):
//   thread 0 keeps up to `in_stages` tile loads in flight, one mbarrier per
//   input slot (arrive.expect_tx + complete_tx);  all threads wait for the
//   slot's phase, transpose into one of two output buffers, fence the async
//   proxy and meet at one CTA barrier; thread 0 then issues the TMA store of
//   the output buffer, refills the input slot and, before the next barrier,
//   waits until the store issued two tiles ago has finished reading its
//   buffer ("Shared-memory tiling and bank conflicts", "Protect tile phases":
//   a buffer is reusable only after its readers finish).
// Every mbarrier wait is bounded; a wait that runs out sets the device fault
// flag, the CTA drains the copies it has in flight and returns.
//
// Ragged output rows: when an output row (rows elements) does not end on a
// 16-byte boundary, a TMA store writes the row's last 16-byte chunk whole and
// so would overwrite the output's pitch padding.  Tiles of the last tile row
// then bypass the output buffer: each thread stores its transposed
// micro-block with bounds-checked element stores.  Input rows need no such
// care: extra elements a load brings in land in output rows past `cols`, which
// the store clips (whole lines).
#include "bounds.cuh"
#include "launch.cuh"
#include "ptx.cuh"
#include "tr_internal.h"
#include "vec_common.cuh"

#include <atomic>
#include <cstdio>
#include <mutex>

namespace tr {

// Set when a bounded in-kernel wait ran out; read and cleared by the host.
__device__ unsigned g_fault_flag = 0;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxOutStages = 4;

struct TmaGeom {
    int64_t total;        // batch * tiles_r * tiles_c
    int32_t tiles_r, tiles_c;
    int32_t rows, cols;   // input plane (the output plane is cols x rows)
    int32_t in_stages;    // input slots (tile loads in flight)
    int32_t out_stages;   // output buffers (tile stores in flight), 2..4
    int32_t diagonal;
    // Output rows whose length (rows elements) is not a whole number of 16-byte
    // chunks: a TMA store writes its last chunk whole, which would spill into
    // the row pitch, so the last tile row is written with element stores.
    int32_t ragged_out;
    void *out;            // output base, for those element stores
    int64_t ld_out, stride_out;
};

// Global stores made with the LSU (the TMA boxes themselves are clipped to the
// tensor maps by the hardware).  Debug builds check each against the logical
// output elements first.
template <typename T>
__device__ __forceinline__ dbg::Side out_side(const TmaGeom &g) {
    return dbg::side(g.out, g.total / (int64_t(g.tiles_r) * g.tiles_c), g.cols, g.rows, g.ld_out,
                     g.stride_out, int(sizeof(T)));
}

template <typename T>
__device__ __forceinline__ void store_chunk(const TmaGeom &g, T *p, uint4 v) {
    if (TR_STORE_OK(out_side<T>(g), p, 16)) __stcs(reinterpret_cast<uint4 *>(p), v);
}

template <typename T>
struct TmaTile {
    static constexpr int V = 16 / int(sizeof(T));
    static constexpr int TILE = 16 * V;             // elements per tile side
    static constexpr int BOXC = 8 * V;              // elements per 128-byte box row
    static constexpr int BOX_BYTES = TILE * 128;    // one box: TILE rows x 128 bytes
    static constexpr int BUF_BYTES = 2 * BOX_BYTES; // one tile
};

__device__ __forceinline__ void tile_coords(const TmaGeom &g, int64_t t, int32_t &b, int32_t &tr,
                                            int32_t &tc) {
    const int64_t per_plane = int64_t(g.tiles_r) * g.tiles_c;
    const int64_t bb = t / per_plane;
    const int64_t r = t - bb * per_plane;
    int64_t r_ = r / g.tiles_c;
    int64_t c_ = r - r_ * g.tiles_c;
    if (g.diagonal) {
        c_ += r_;
        c_ %= g.tiles_c;
    }
    b = int32_t(bb);
    tr = int32_t(r_);
    tc = int32_t(c_);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
k_tma(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_out,
      TmaGeom g) {
    using L = TmaTile<T>;
    constexpr int V = L::V;
    extern __shared__ uint8_t smem_raw[];
    pdl_prologue();
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *in_buf = base;
    uint8_t *out_buf = base + size_t(g.in_stages) * L::BUF_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(out_buf + size_t(g.out_stages) * L::BUF_BYTES);

    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int quad = w >> 1;                      // which 8x8 group of micro-blocks
    const int s = (lane >> 3) + 4 * (w & 1);      // generalized diagonal of the phase
    const int c = lane & 7, a = c ^ s;
    const int A = 8 * (quad >> 1) + a, C = 8 * (quad & 1) + c;
    uint32_t roff[V], woff[V];
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const int r = V * A + m, o = V * C + m;
        roff[m] = (C >> 3) * L::BOX_BYTES + r * 128 + ((c ^ (r & 7)) << 4);
        woff[m] = (A >> 3) * L::BOX_BYTES + o * 128 + ((a ^ (o & 7)) << 4);
    }

    const int64_t n_local =
        blockIdx.x < g.total ? (g.total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int S = g.in_stages;
    const int SO = g.out_stages;

    auto issue_load = [&](int64_t k, int slot) {
        int32_t b, tr, tc;
        tile_coords(g, int64_t(blockIdx.x) + k * gridDim.x, b, tr, tc);
        uint64_t *bar = full + slot;
        ptx::mbar_arrive_expect_tx(bar, L::BUF_BYTES);
        uint8_t *dst = in_buf + size_t(slot) * L::BUF_BYTES;
        ptx::tma_load_3d(dst, &tm_in, bar, tc * L::TILE, tr * L::TILE, b);
        ptx::tma_load_3d(dst + L::BOX_BYTES, &tm_in, bar, tc * L::TILE + L::BOXC, tr * L::TILE, b);
    };

    if (t == 0) {
        ptx::prefetch_tensormap(&tm_in);
        ptx::prefetch_tensormap(&tm_out);
        for (int i = 0; i < S; ++i) ptx::mbar_init(full + i, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (t == 0)
        for (int64_t k = 0; k < n_local && k < S; ++k) issue_load(k, int(k));

    int64_t k = 0;
    bool aborted = false;
    for (; k < n_local; ++k) {
        const int slot = int(k % S);
        const uint32_t parity = uint32_t((k / S) & 1);
        const bool ok = ptx::mbar_wait_bounded(full + slot, parity);

        int32_t b, tr, tc;
        tile_coords(g, int64_t(blockIdx.x) + k * gridDim.x, b, tr, tc);
        const bool direct = g.ragged_out && tr == g.tiles_r - 1;

        const uint8_t *ib = in_buf + size_t(slot) * L::BUF_BYTES;
        uint8_t *ob = out_buf + size_t(k % SO) * L::BUF_BYTES;
        Chunk x[V], y[V];
#pragma unroll
        for (int m = 0; m < V; ++m) x[m].v = *reinterpret_cast<const uint4 *>(ib + roff[m]);
        micro_transpose(x, y);
        if (!direct) {
#pragma unroll
            for (int m = 0; m < V; ++m) *reinterpret_cast<uint4 *>(ob + woff[m]) = y[m].v;
            ptx::fence_proxy_async_smem();
        } else if (ok) {
            // Last tile row of a ragged output: bounds-checked element stores.
            T *dst = static_cast<T *>(g.out) + int64_t(b) * g.stride_out;
            const int64_t oc = int64_t(tr) * L::TILE + V * A;
#pragma unroll
            for (int m = 0; m < V; ++m) {
                const int64_t orow = int64_t(tc) * L::TILE + V * C + m;
                if (orow < g.cols) {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        if (oc + e < g.rows &&
                            TR_STORE_OK(out_side<T>(g), dst + orow * g.ld_out + oc + e, int(sizeof(T))))
                            dst[orow * g.ld_out + oc + e] = elem<T>(y[m], e);
                }
            }
        }
        // Tile k+1 goes to the buffer of the store issued for tile k+1-SO: that
        // store must have finished reading it, so at most SO-2 of the stores
        // committed so far (tiles .. k-1) may still be reading.
        if (t == 0) {
            if (SO == 2) ptx::bulk_wait_group_read<0>();
            else if (SO == 3) ptx::bulk_wait_group_read<1>();
            else ptx::bulk_wait_group_read<2>();
        }
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        if (t == 0) {
            if (!direct) {
                ptx::tma_store_3d(&tm_out, ob, tr * L::TILE, tc * L::TILE, b);
                if (tr * L::TILE + L::BOXC < g.rows)
                    ptx::tma_store_3d(&tm_out, ob + L::BOX_BYTES, tr * L::TILE + L::BOXC,
                                      tc * L::TILE, b);
            }
            // An empty group keeps the count of committed groups one per tile.
            ptx::bulk_commit_group();
            if (k + S < n_local) issue_load(k + S, slot);
        }
    }

    if (t == 0) {
        if (aborted) {
            atomicExch(&g_fault_flag, 1u);
            // Drain the loads still in flight (tiles k .. k+S-1) before the
            // shared memory they target goes away; each wait is bounded too.
            for (int64_t kk = k; kk < n_local && kk < k + S; ++kk)
                ptx::mbar_wait_bounded(full + int(kk % S), uint32_t((kk / S) & 1));
        }
        ptx::bulk_wait_group<0>();
    }
}

// ---------------------------------------------------------------------------
// Per-warp pipelines.  The CTA-wide pipeline above stalls every warp on one
// barrier per tile and leaves the loads to one thread of the block.  Here each
// warp is its own pipeline over its own tiles (warp w of the grid takes tiles
// w, w + warps, ...): lane 0 keeps `in_stages` TMA box loads in flight on the
// warp's mbarriers, the 32 lanes turn each tile around and lane 0 stores it
// with one TMA box store.  The only synchronisation is __syncwarp, so warps
// and blocks never wait for one another.
//
// Tile: one 128-byte-wide box each way, 8V x 8V elements (32x32 fp32, 64x64
// bf16), 8 x 8 micro-blocks; each lane owns two, (a, c) = (x ^ s, x) with
// x = lane % 8 and s = lane / 8 + 4p for p = 0, 1, so every 8-lane phase of a
// 16-byte shared access hits 8 distinct positions (see the analysis above).
template <typename T>
struct WarpTile {
    static constexpr int V = 16 / int(sizeof(T));
    static constexpr int TILE = 8 * V;        // elements per tile side
    static constexpr int BYTES = TILE * 128;  // one box: 4 KiB fp32, 8 KiB bf16
};

template <typename T>
__global__ void __launch_bounds__(256)
k_tma_warp(const __grid_constant__ CUtensorMap tm_in, const __grid_constant__ CUtensorMap tm_out,
           TmaGeom g) {
    using L = WarpTile<T>;
    constexpr int V = L::V;
    extern __shared__ uint8_t smem_raw[];
    pdl_prologue();
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int S = g.in_stages, SO = g.out_stages;
    const size_t per_warp = size_t(S + SO) * L::BYTES;
    uint8_t *in_buf = base + warp * per_warp;
    uint8_t *out_buf = in_buf + size_t(S) * L::BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + nwarps * per_warp) + warp * S;

    const int x = lane & 7;
    int aa[2];
    uint32_t roff[2][V], woff[2][V];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int s = (lane >> 3) + 4 * p, a = x ^ s;
        aa[p] = a;
#pragma unroll
        for (int m = 0; m < V; ++m) {
            const int r = V * a + m, o = V * x + m;
            roff[p][m] = r * 128 + ((x ^ (r & 7)) << 4);
            woff[p][m] = o * 128 + ((a ^ (o & 7)) << 4);
        }
    }

    const int64_t gw = int64_t(blockIdx.x) * nwarps + warp;
    const int64_t G = int64_t(gridDim.x) * nwarps;
    const int64_t n_local = gw < g.total ? (g.total - 1 - gw) / G + 1 : 0;

    auto issue_load = [&](int64_t k, int slot) {
        int32_t b, tr, tc;
        tile_coords(g, gw + k * G, b, tr, tc);
        ptx::mbar_arrive_expect_tx(full + slot, L::BYTES);
        ptx::tma_load_3d(in_buf + size_t(slot) * L::BYTES, &tm_in, full + slot, tc * L::TILE,
                         tr * L::TILE, b);
    };

    if (lane == 0) {
        ptx::prefetch_tensormap(&tm_in);
        ptx::prefetch_tensormap(&tm_out);
        for (int i = 0; i < S; ++i) ptx::mbar_init(full + i, 1);
        ptx::fence_barrier_init();
        for (int64_t k = 0; k < n_local && k < S; ++k) issue_load(k, int(k));
    }
    __syncwarp();

    int64_t k = 0;
    bool aborted = false;
    for (; k < n_local; ++k) {
        const int slot = int(k % S);
        const bool ok = ptx::mbar_wait_bounded(full + slot, uint32_t((k / S) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            aborted = true;
            break;
        }
        int32_t b, tr, tc;
        tile_coords(g, gw + k * G, b, tr, tc);
        const bool direct = g.ragged_out && tr == g.tiles_r - 1;
        const uint8_t *ib = in_buf + size_t(slot) * L::BYTES;
        uint8_t *ob = out_buf + size_t(k % SO) * L::BYTES;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            Chunk xv[V], yv[V];
#pragma unroll
            for (int m = 0; m < V; ++m) xv[m].v = *reinterpret_cast<const uint4 *>(ib + roff[p][m]);
            micro_transpose(xv, yv);
            if (!direct) {
#pragma unroll
                for (int m = 0; m < V; ++m) *reinterpret_cast<uint4 *>(ob + woff[p][m]) = yv[m].v;
            } else {
                // Last tile row of a ragged output: bounds-checked element stores.
                T *dst = static_cast<T *>(g.out) + int64_t(b) * g.stride_out;
                const int64_t oc = int64_t(tr) * L::TILE + V * aa[p];
#pragma unroll
                for (int m = 0; m < V; ++m) {
                    const int64_t orow = int64_t(tc) * L::TILE + V * x + m;
                    if (orow < g.cols) {
#pragma unroll
                        for (int e = 0; e < V; ++e)
                            if (oc + e < g.rows &&
                                TR_STORE_OK(out_side<T>(g), dst + orow * g.ld_out + oc + e, int(sizeof(T))))
                                dst[orow * g.ld_out + oc + e] = elem<T>(yv[m], e);
                    }
                }
            }
        }
        if (!direct) ptx::fence_proxy_async_smem();
        if (lane == 0) {
            // The next tile's output buffer was last read by the store issued
            // SO-1 tiles ago: at most SO-2 stores may still be reading.
            if (SO == 2) ptx::bulk_wait_group_read<0>();
            else if (SO == 3) ptx::bulk_wait_group_read<1>();
            else ptx::bulk_wait_group_read<2>();
        }
        __syncwarp();
        if (lane == 0) {
            if (!direct) ptx::tma_store_3d(&tm_out, ob, tr * L::TILE, tc * L::TILE, b);
            ptx::bulk_commit_group();
            if (k + S < n_local) issue_load(k + S, slot);
        }
    }
    if (lane == 0) {
        if (aborted) {
            atomicExch(&g_fault_flag, 1u);
            for (int64_t kk = k; kk < n_local && kk < k + S; ++kk)
                ptx::mbar_wait_bounded(full + int(kk % S), uint32_t((kk / S) & 1));
        }
        ptx::bulk_wait_group<0>();
    }
}

// ---------------------------------------------------------------------------
// TMA loads, register stores.  Per-warp pipelines of TMA box loads as above,
// but no output buffer and no TMA store: each lane turns its micro-blocks
// around in registers and stores them straight to global memory with 16-byte
// stores, lanes with consecutive A (same C) writing consecutive chunks of one
// output row (8 lanes = 128 contiguous bytes).  Only the input side needs the
// TMA alignment rules; the output side needs 16-byte aligned rows for the
// vector stores (the launcher checks) and edge tiles use element stores.
//
// That lane map reads 8 micro-blocks of one chunk column per phase, which on
// the 128-byte swizzle (position = chunk ^ (row % 8)) would put 8 lanes on 2
// positions (fp32) or 1 (bf16).  So lane A reads its V rows in a rotated
// order, row V*A + ((m + rot) % V) at step m with rot = A / 2 (fp32) or A
// (bf16), which makes (row % 8) distinct across the 8 lanes at every step; the
// rotation is undone in registers before the micro-transpose.
template <int V>
__device__ __forceinline__ void unrotate(Chunk (&x)[V], int rot) {
    // x[m] holds row (m + rot) % V; afterwards x[j] holds row j.
    Chunk t[V];
#pragma unroll
    for (int step = 1; step < V; step <<= 1) {
        if (rot & step) {
#pragma unroll
            for (int j = 0; j < V; ++j) t[j] = x[(j - step + V) % V];
#pragma unroll
            for (int j = 0; j < V; ++j) x[j] = t[j];
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
k_tma_ldst(const __grid_constant__ CUtensorMap tm_in, TmaGeom g) {
    using L = WarpTile<T>;
    constexpr int V = L::V;
    extern __shared__ uint8_t smem_raw[];
    pdl_prologue();
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int S = g.in_stages;
    uint8_t *in_buf = base + size_t(warp) * S * L::BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + size_t(nwarps) * S * L::BYTES) + warp * S;

    const int A = lane & 7;
    const int rot = V == 4 ? (A >> 1) : A;
    uint32_t roff[2][V];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int C = 4 * p + (lane >> 3);
#pragma unroll
        for (int m = 0; m < V; ++m) {
            const int r = V * A + ((m + rot) & (V - 1));
            roff[p][m] = r * 128 + ((C ^ (r & 7)) << 4);
        }
    }

    const int64_t gw = int64_t(blockIdx.x) * nwarps + warp;
    const int64_t G = int64_t(gridDim.x) * nwarps;
    const int64_t n_local = gw < g.total ? (g.total - 1 - gw) / G + 1 : 0;

    auto issue_load = [&](int64_t k, int slot) {
        int32_t b, tr, tc;
        tile_coords(g, gw + k * G, b, tr, tc);
        ptx::mbar_arrive_expect_tx(full + slot, L::BYTES);
        ptx::tma_load_3d(in_buf + size_t(slot) * L::BYTES, &tm_in, full + slot, tc * L::TILE,
                         tr * L::TILE, b);
    };

    if (lane == 0) {
        ptx::prefetch_tensormap(&tm_in);
        for (int i = 0; i < S; ++i) ptx::mbar_init(full + i, 1);
        ptx::fence_barrier_init();
        for (int64_t k = 0; k < n_local && k < S; ++k) issue_load(k, int(k));
    }
    __syncwarp();

    int64_t k = 0;
    bool aborted = false;
    for (; k < n_local; ++k) {
        const int slot = int(k % S);
        const bool ok = ptx::mbar_wait_bounded(full + slot, uint32_t((k / S) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            aborted = true;
            break;
        }
        int32_t b, tr, tc;
        tile_coords(g, gw + k * G, b, tr, tc);
        const uint8_t *ib = in_buf + size_t(slot) * L::BYTES;
        Chunk x[2][V];
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
            for (int m = 0; m < V; ++m) x[p][m].v = *reinterpret_cast<const uint4 *>(ib + roff[p][m]);
        __syncwarp();  // the slot is read: it may be refilled
        if (lane == 0 && k + S < n_local) issue_load(k + S, slot);

        T *dst = static_cast<T *>(g.out) + int64_t(b) * g.stride_out;
        const int64_t r0 = int64_t(tr) * L::TILE, c0 = int64_t(tc) * L::TILE;
        const bool full_tile = r0 + L::TILE <= g.rows && c0 + L::TILE <= g.cols;
        const int64_t oc = r0 + V * A;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int C = 4 * p + (lane >> 3);
            unrotate<V>(x[p], rot);
            Chunk y[V];
            micro_transpose(x[p], y);
#pragma unroll
            for (int m = 0; m < V; ++m) {
                const int64_t orow = c0 + V * C + m;
                T *row = dst + orow * g.ld_out;
                if (full_tile) {
                    store_chunk<T>(g, row + oc, y[m].v);
                } else if (orow < g.cols) {
                    if (oc + V <= g.rows) {
                        store_chunk<T>(g, row + oc, y[m].v);
                    } else {
#pragma unroll
                        for (int e = 0; e < V; ++e)
                            if (oc + e < g.rows && TR_STORE_OK(out_side<T>(g), row + oc + e, int(sizeof(T))))
                            row[oc + e] = elem<T>(y[m], e);
                    }
                }
            }
        }
    }
    if (lane == 0 && aborted) {
        atomicExch(&g_fault_flag, 1u);
        for (int64_t kk = k; kk < n_local && kk < k + S; ++kk)
            ptx::mbar_wait_bounded(full + int(kk % S), uint32_t((kk / S) & 1));
    }
}

// ---------------------------------------------------------------------------
// Warp-specialised pipeline: one producer warp and eight consumer warps per
// CTA, over the CTA-wide 16V x 16V tiles (two 128-byte boxes per tile).
//
// Each input slot has two mbarriers.  `full[slot]` completes when the TMA
// bytes of the tile have landed (the producer arms it with expect_tx);
// `empty[slot]` completes when all eight consumer warps have read the slot
// (one arrival per warp).  The producer (lane 0 of the last warp) walks the
// CTA's tiles, waits for a slot to be empty and refills it, so up to S tile
// loads are in flight while the consumers work; it never touches the data.
// The consumers wait for a slot to be full, read their micro-block, release
// the slot and store the transposed micro-block straight to global memory
// with 16-byte stores.  No consumer waits for another: the only coupling is
// through the slot barriers ("Shared-memory tiling and bank conflicts",
// "Protect tile phases": a buffer is refilled only after its readers are
// done, and read only after its writer is done).
//
// Consumer thread t (< 256) owns micro-block (A, C) = (t % 16, t / 16): tile
// rows V*A .. V*A+V-1 of chunk column C, which become output rows V*C + m,
// chunk A; sixteen lanes with consecutive A write 256 contiguous bytes of one
// output row.  The 8 lanes of a shared-load phase share C and have A = 8h ..
// 8h+7; reading row V*A + m for the same m in every lane would put them on 2
// (fp32) or 1 (bf16) swizzle positions, so lane A reads its rows rotated by
// rot = (A / 2) % 4 (fp32) or A % 8 (bf16), which makes row % 8 -- and with
// it the position chunk ^ (row % 8) -- distinct across the phase; the rotation
// is undone in registers.
constexpr int kWsConsumerWarps = 8;
constexpr int kWsThreads = 32 * (kWsConsumerWarps + 1);

template <typename T>
__global__ void __launch_bounds__(kWsThreads, 1)
k_tma_ws(const __grid_constant__ CUtensorMap tm_in, TmaGeom g) {
    using L = TmaTile<T>;
    constexpr int V = L::V;
    extern __shared__ uint8_t smem_raw[];
    pdl_prologue();
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = g.in_stages;
    uint8_t *in_buf = base;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + size_t(S) * L::BUF_BYTES);
    uint64_t *empty = full + S;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int64_t n_local =
        blockIdx.x < g.total ? (g.total - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (t == 0) {
        ptx::prefetch_tensormap(&tm_in);
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(full + i, 1);
            ptx::mbar_init(empty + i, kWsConsumerWarps);
        }
        ptx::fence_barrier_init();
    }
    __syncthreads();

    if (warp == kWsConsumerWarps) {
        // ---- producer
        if (lane != 0) return;
        int64_t k = 0;
        bool ok = true;
        for (; k < n_local; ++k) {
            const int slot = int(k % S);
            // Slot reuse: the consumers must have released the tile loaded
            // into it S tiles ago (phase k/S - 1 of its empty barrier).
            if (k >= S && !ptx::mbar_wait_bounded(empty + slot, uint32_t((k / S - 1) & 1))) {
                ok = false;
                break;
            }
            int32_t b, tr, tc;
            tile_coords(g, int64_t(blockIdx.x) + k * gridDim.x, b, tr, tc);
            uint8_t *dst = in_buf + size_t(slot) * L::BUF_BYTES;
            ptx::mbar_arrive_expect_tx(full + slot, L::BUF_BYTES);
            ptx::tma_load_3d(dst, &tm_in, full + slot, tc * L::TILE, tr * L::TILE, b);
            ptx::tma_load_3d(dst + L::BOX_BYTES, &tm_in, full + slot, tc * L::TILE + L::BOXC,
                             tr * L::TILE, b);
        }
        if (!ok) atomicExch(&g_fault_flag, 1u);
        // The last load issued into each slot lands before the CTA's shared
        // memory can go away (no later phase starts, so the parity is exact).
        for (int64_t kk = k > S ? k - S : 0; kk < k; ++kk)
            ptx::mbar_wait_bounded(full + int(kk % S), uint32_t((kk / S) & 1));
        return;
    }

    // ---- consumers
    const int A = t & 15, C = t >> 4;
    const int rot = V == 4 ? ((A >> 1) & 3) : (A & 7);
    uint32_t roff[V];
#pragma unroll
    for (int m = 0; m < V; ++m) {
        const int r = V * A + ((m + rot) & (V - 1));
        roff[m] = (C >> 3) * L::BOX_BYTES + r * 128 + (((C & 7) ^ (r & 7)) << 4);
    }
    for (int64_t k = 0; k < n_local; ++k) {
        const int slot = int(k % S);
        const bool ok = ptx::mbar_wait_bounded(full + slot, uint32_t((k / S) & 1));
        if (__any_sync(0xffffffffu, !ok)) {
            // The producer's own bounded wait for this warp's release runs out
            // in turn and drains the loads in flight.
            if (lane == 0) atomicExch(&g_fault_flag, 1u);
            break;
        }
        const uint8_t *ib = in_buf + size_t(slot) * L::BUF_BYTES;
        Chunk x[V];
#pragma unroll
        for (int m = 0; m < V; ++m) x[m].v = *reinterpret_cast<const uint4 *>(ib + roff[m]);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(empty + slot);

        int32_t b, tr, tc;
        tile_coords(g, int64_t(blockIdx.x) + k * gridDim.x, b, tr, tc);
        unrotate<V>(x, rot);
        Chunk y[V];
        micro_transpose(x, y);
        T *dst = static_cast<T *>(g.out) + int64_t(b) * g.stride_out;
        const int64_t r0 = int64_t(tr) * L::TILE, c0 = int64_t(tc) * L::TILE;
        const bool full_tile = r0 + L::TILE <= g.rows && c0 + L::TILE <= g.cols;
        const int64_t oc = r0 + V * A;
#pragma unroll
        for (int m = 0; m < V; ++m) {
            const int64_t orow = c0 + V * C + m;
            T *row = dst + orow * g.ld_out;
            if (full_tile) {
                store_chunk<T>(g, row + oc, y[m].v);
            } else if (orow < g.cols) {
                if (oc + V <= g.rows) {
                    store_chunk<T>(g, row + oc, y[m].v);
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        if (oc + e < g.rows && TR_STORE_OK(out_side<T>(g), row + oc + e, int(sizeof(T))))
                            row[oc + e] = elem<T>(y[m], e);
                }
            }
        }
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 3-D map over [planes][lines][elems] with a 128-byte-wide box of box_lines lines.
bool encode_3d(CUtensorMap *map, const void *base, int esize, int64_t elems, int64_t lines,
               int64_t planes, int64_t line_pitch, int64_t plane_pitch, int box_elems,
               int box_lines) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {cuuint64_t(elems), cuuint64_t(lines), cuuint64_t(planes)};
    const cuuint64_t strides[2] = {cuuint64_t(line_pitch) * esize,
                                   cuuint64_t(plane_pitch) * esize};
    const cuuint32_t box[3] = {cuuint32_t(box_elems), cuuint32_t(box_lines), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                          3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Per-device facts and per-configuration occupancy, computed once: the
// launch path then makes no attribute or occupancy query per call.
enum Kind { kPerBlock = 0, kPerWarp = 1, kLoadOnly = 2, kWarpSpec = 3 };

struct DeviceInfo {
    std::atomic<bool> ok{false};  // set last, after the fields below are filled
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int max_smem_optin = 0;
    // [kind][esize == 4][in_stages][out_stages]; 0 = not computed
    std::atomic<int> fit[4][2][9][kMaxOutStages + 1] = {};
};

constexpr int kMaxDevices = 64;
constexpr int kWarpsPerBlock = 1;  // per-warp pipelines: one warp per block
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

DeviceInfo &device_info() {
    static thread_local DeviceInfo failed;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
        failed.ok.store(false);
        failed.err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return failed;
    }
    DeviceInfo &info = g_dev[d];
    if (!info.ok.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        if (!info.ok.load(std::memory_order_relaxed)) {
            int sms = 0, optin = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
            if (e == cudaSuccess)
                e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
            // Opt the kernels in to the largest dynamic shared memory once.
            const void *kernels[8] = {reinterpret_cast<const void *>(k_tma<uint32_t>),
                                      reinterpret_cast<const void *>(k_tma<uint16_t>),
                                      reinterpret_cast<const void *>(k_tma_warp<uint32_t>),
                                      reinterpret_cast<const void *>(k_tma_warp<uint16_t>),
                                      reinterpret_cast<const void *>(k_tma_ldst<uint32_t>),
                                      reinterpret_cast<const void *>(k_tma_ldst<uint16_t>),
                                      reinterpret_cast<const void *>(k_tma_ws<uint32_t>),
                                      reinterpret_cast<const void *>(k_tma_ws<uint16_t>)};
            for (const void *k : kernels)
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
            if (e != cudaSuccess) {
                failed.ok.store(false);
                failed.err = e;
                return failed;
            }
            info.sms = sms;
            info.max_smem_optin = optin;
            info.ok.store(true, std::memory_order_release);
        }
    }
    return info;
}

// Dynamic shared memory: 1 KiB of slack to align the buffers to the 128-byte
// swizzle's 1 KiB pattern, the tile buffers, one 8-byte mbarrier per input slot.
template <typename T>
size_t smem_bytes(Kind kind, int in_stages, int out_stages) {
    switch (kind) {
        case kPerBlock:
            return 1024 + size_t(in_stages + out_stages) * TmaTile<T>::BUF_BYTES +
                   size_t(in_stages) * 8;
        case kPerWarp:
            return 1024 + size_t(kWarpsPerBlock) * (size_t(in_stages + out_stages) *
                                                        WarpTile<T>::BYTES + size_t(in_stages) * 8);
        case kWarpSpec:  // input slots, a full and an empty barrier per slot
            return 1024 + size_t(in_stages) * TmaTile<T>::BUF_BYTES + size_t(in_stages) * 16;
        default:
            return 1024 + size_t(kWarpsPerBlock) *
                              (size_t(in_stages) * WarpTile<T>::BYTES + size_t(in_stages) * 8);
    }
}

template <typename T>
int resident_ctas(DeviceInfo &dev, Kind kind, int in_stages, int out_stages) {
    std::atomic<int> &slot = dev.fit[kind][sizeof(T) == 4][in_stages][out_stages];
    int cached = slot.load(std::memory_order_acquire);
    if (cached == 0) {
        int fit = 0;
        const size_t smem = smem_bytes<T>(kind, in_stages, out_stages);
        cudaError_t e;
        if (kind == kPerBlock)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k_tma<T>, kThreads, smem);
        else if (kind == kPerWarp)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k_tma_warp<T>,
                                                              32 * kWarpsPerBlock, smem);
        else if (kind == kWarpSpec)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k_tma_ws<T>, kWsThreads, smem);
        else
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k_tma_ldst<T>,
                                                              32 * kWarpsPerBlock, smem);
        cached = (e != cudaSuccess || fit < 1) ? -1 : fit;
        slot.store(cached, std::memory_order_release);
    }
    return cached;
}

// Defaults, the best measured on GB300: per-warp pipeline with 6 box loads
// in flight and 2 output buffers (fp32, 4 KiB boxes) or 4 loads and 3 output
// buffers (bf16, 8 KiB boxes); CTA-wide pipeline with 2 + 2; load-only
// pipeline with 8 (fp32) or 6 (bf16) loads in flight; warp-specialised
// pipeline with 8 tile slots (fp32, one CTA per SM) or 2 (bf16).
int default_in_stages(size_t esize, Kind kind) {
    if (kind == kPerWarp) return esize == 4 ? 6 : 4;
    if (kind == kLoadOnly) return esize == 4 ? 8 : 6;
    if (kind == kWarpSpec) return esize == 4 ? 8 : 2;
    return 2;
}
int default_out_stages(size_t esize, Kind kind) {
    return (kind == kPerWarp && esize == 2) ? 3 : 2;
}

template <typename T>
cudaError_t launch_typed(const Problem &p, const TmaConfig &cfg, const char **why) {
    const Kind kind = cfg.schedule == 1   ? kPerBlock
                      : cfg.schedule == 3 ? kLoadOnly
                      : cfg.schedule == 4 ? kWarpSpec
                                          : kPerWarp;
    const bool cta_tile = kind == kPerBlock || kind == kWarpSpec;
    const int tile = cta_tile ? TmaTile<T>::TILE : WarpTile<T>::TILE;
    const int boxc = TmaTile<T>::BOXC;  // 128-byte box rows in every kind
    const int64_t two31 = int64_t(1) << 31, two40 = int64_t(1) << 40;
    if (p.rows >= two31 || p.cols >= two31 || p.batch >= two31) {
        *why = "TMA coordinates are 32-bit: a dimension is 2^31 or more";
        return cudaErrorInvalidValue;
    }
    // Plane pitches as the tensor map sees them: a single plane still needs a
    // legal third-dimension stride, and it must cover a whole plane.
    const int64_t sin = p.batch > 1 ? p.stride_in : p.rows * p.ld_in;
    const int64_t sout = p.batch > 1 ? p.stride_out : p.cols * p.ld_out;
    if (sin < p.rows * p.ld_in || sout < p.cols * p.ld_out || sin * p.esize >= two40 ||
        sout * p.esize >= two40 || p.ld_in * p.esize >= two40 || p.ld_out * p.esize >= two40) {
        *why = "TMA needs plane pitches that cover whole planes and strides below 2^40 bytes";
        return cudaErrorInvalidValue;
    }
    CUtensorMap tm_in, tm_out;
    if (!encode_3d(&tm_in, p.in, p.esize, p.cols, p.rows, p.batch, p.ld_in, sin, boxc, tile) ||
        (kind != kLoadOnly && kind != kWarpSpec &&
         !encode_3d(&tm_out, p.out, p.esize, p.rows, p.cols, p.batch, p.ld_out, sout, boxc, tile))) {
        *why = "cuTensorMapEncodeTiled rejected the tensor maps";
        return cudaErrorInvalidValue;
    }
    TmaGeom g{};
    g.tiles_r = int32_t((p.rows + tile - 1) / tile);
    g.tiles_c = int32_t((p.cols + tile - 1) / tile);
    g.total = p.batch * int64_t(g.tiles_r) * g.tiles_c;
    g.rows = int32_t(p.rows);
    g.cols = int32_t(p.cols);
    g.diagonal = cfg.tile_order == 1;
    g.ragged_out = (p.rows * p.esize) % 16 != 0;
    g.out = p.out;
    g.ld_out = p.ld_out;
    g.stride_out = sout;
    DeviceInfo &dev = device_info();
    if (!dev.ok.load(std::memory_order_acquire)) return dev.err;
    const int stages = cfg.stages > 0 ? cfg.stages : default_in_stages(sizeof(T), kind);
    const int out_stages = cfg.out_stages > 0 ? cfg.out_stages : default_out_stages(sizeof(T), kind);
    if (stages < 2 || stages > 8 || out_stages < 2 || out_stages > kMaxOutStages) {
        *why = "TMA stage counts out of range";
        return cudaErrorInvalidValue;
    }
    g.in_stages = stages;
    g.out_stages = out_stages;
    const size_t smem = smem_bytes<T>(kind, stages, out_stages);
    if (smem > size_t(dev.max_smem_optin)) {
        *why = "TMA pipeline does not fit in shared memory; lower the stage count";
        return cudaErrorInvalidValue;
    }
    const int fit = resident_ctas<T>(dev, kind, stages, out_stages);
    if (fit < 1) {
        *why = "TMA kernel cannot be resident with this configuration";
        return cudaErrorInvalidValue;
    }
    int per_sm = cfg.ctas_per_sm > 0 ? cfg.ctas_per_sm : fit;
    if (per_sm > fit) per_sm = fit;
    const int64_t units = cta_tile ? g.total : (g.total + kWarpsPerBlock - 1) / kWarpsPerBlock;
    int64_t grid = int64_t(dev.sms) * per_sm;
    if (grid > units) grid = units;
    const dim3 gd{unsigned(grid)};
    if (kind == kPerWarp)
        return launch_pdl(k_tma_warp<T>, gd, dim3(32 * kWarpsPerBlock), smem, p.stream, tm_in,
                          tm_out, g);
    if (kind == kLoadOnly)
        return launch_pdl(k_tma_ldst<T>, gd, dim3(32 * kWarpsPerBlock), smem, p.stream, tm_in, g);
    if (kind == kWarpSpec)
        return launch_pdl(k_tma_ws<T>, gd, dim3(kWsThreads), smem, p.stream, tm_in, g);
    return launch_pdl(k_tma<T>, gd, dim3(kThreads), smem, p.stream, tm_in, tm_out, g);
}

}  // namespace

cudaError_t launch_tma(const Problem &p, const TmaConfig &cfg, const char **why) {
    return p.esize == 4 ? launch_typed<uint32_t>(p, cfg, why) : launch_typed<uint16_t>(p, cfg, why);
}

namespace {

// Self-test of the bounded wait: one warp waits on an mbarrier phase that
// completes only if `arrive` is set (lane 0 arrives on it); otherwise the
// wait runs out after limit_ns and the fault flag is raised exactly as in the
// transpose kernels.  Nothing here can fault or hang: the wait is bounded.
__global__ void k_wait_selftest(int arrive, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ptx::smem_addr(&bar))
                     : "memory");
    const bool ok = ptx::mbar_wait_bounded(&bar, 0, limit_ns);
    if (__any_sync(0xffffffffu, !ok) && threadIdx.x == 0) atomicExch(&g_fault_flag, 1u);
}

}  // namespace

cudaError_t launch_wait_selftest(bool arrive, int64_t limit_ns, cudaStream_t stream) {
    k_wait_selftest<<<1, 32, 0, stream>>>(arrive ? 1 : 0, uint64_t(limit_ns));
    return cudaGetLastError();
}

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_tma)

cudaError_t read_and_clear_fault(unsigned *value) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(value, g_fault_flag, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_fault_flag, &zero, sizeof(unsigned));
}

}  // namespace tr
