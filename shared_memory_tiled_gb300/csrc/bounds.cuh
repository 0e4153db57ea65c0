// Bounds checks of a debug build (compiled in with -DTR_DEBUG=1, absent
// otherwise).
//
// A tile kernel computes every global address from run-time pitches, plane
// pitches, shifts and tile coordinates; an index that is off by one reads or
// writes a neighbour's memory and may still leave the output right ("Shared
// memory and the bank conflict", "The barrier": a fault that shows only
// sometimes).  In a debug build every such access first asks a guard whether
// its bytes belong to its side:
//   - TR_LOAD_OK: every element of the access is a logical element of the
//     input (batch planes of rows x cols at row pitch ld_in, plane pitch
//     stride_in);
//   - TR_LOAD_IN_EXTENT: the access lies between the input's first and last
//     logical element (the realigned loads read 16-byte chunks whose extra
//     bytes are neighbouring columns or pitch padding of the same input);
//   - TR_STORE_OK: every element of the access is a logical element of the
//     output.
// A refused access is skipped (never performed) and counted in a per-
// translation-unit record, which the host reads through tr_debug_bounds().
// Nothing traps.  In a release build the guards are the constant `true` and
// the declarations vanish, so the kernels compile to what they were.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tr {
namespace dbg {

// What a translation unit's kernels recorded since the host last read it.
struct Record {
    unsigned long long count;       // refused accesses
    unsigned long long first_addr;  // address of the first one recorded
    unsigned first_bytes;           // its width
    unsigned first_store;           // 1 = store, 0 = load
    unsigned taken;                 // 1 once `first_*` is set
};

// One side of a kernel: `batch` planes of rows x cols elements of `esize`
// bytes at row pitch `ld` and plane pitch `stride` (ignored for batch 1).
struct Side {
    uintptr_t base;
    int64_t batch, rows, cols, ld, stride;
    int esize;
};

__host__ __device__ inline Side side(const void *base, int64_t batch, int64_t rows, int64_t cols,
                                     int64_t ld, int64_t stride, int esize) {
    return Side{reinterpret_cast<uintptr_t>(base), batch, rows, cols, ld, stride, esize};
}

// Bytes from the first logical element to one past the last.
__host__ __device__ inline uint64_t extent_bytes(const Side &s) {
    if (s.batch <= 0 || s.rows <= 0 || s.cols <= 0) return 0;
    return uint64_t((s.batch - 1) * (s.batch > 1 ? s.stride : 0) + (s.rows - 1) * s.ld + s.cols) *
           uint64_t(s.esize);
}

// Whether element e (counted from the base) is a logical element.
__host__ __device__ inline bool logical_element(const Side &s, int64_t e) {
    if (e < 0) return false;
    const int64_t b = s.batch > 1 ? e / s.stride : 0;
    const int64_t r = e - b * (s.batch > 1 ? s.stride : 0);
    const int64_t i = r / s.ld, j = r - i * s.ld;
    return b < s.batch && i < s.rows && j < s.cols;
}

// Whether all `bytes` bytes at address a are logical elements of s.
__host__ __device__ inline bool all_logical(const Side &s, uintptr_t a, int bytes) {
    if (a < s.base || (a - s.base) % uintptr_t(s.esize) || bytes <= 0 || bytes % s.esize) return false;
    const int64_t e0 = int64_t((a - s.base) / uintptr_t(s.esize));
    for (int q = 0; q < bytes / s.esize; ++q)
        if (!logical_element(s, e0 + q)) return false;
    return true;
}

// Whether all `bytes` bytes at address a lie inside the extent of s.
__host__ __device__ inline bool in_extent(const Side &s, uintptr_t a, int bytes) {
    return a >= s.base && bytes > 0 && uint64_t(a - s.base) + uint64_t(bytes) <= extent_bytes(s);
}

#ifdef TR_DEBUG
// One record per translation unit (each unit that includes this header).  The
// checks below are out-of-line calls: inlined at every access of the unrolled
// tile loops they would multiply the code, and its compile time, many times.
static __device__ Record g_bounds;

static __device__ inline bool refuse(uintptr_t a, int bytes, bool store) {
    atomicAdd(&g_bounds.count, 1ull);
    if (atomicCAS(&g_bounds.taken, 0u, 1u) == 0u) {
        g_bounds.first_addr = a;
        g_bounds.first_bytes = unsigned(bytes);
        g_bounds.first_store = store ? 1u : 0u;
    }
    return false;
}

static __device__ __noinline__ bool load_ok(const Side &s, const void *p, int bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return all_logical(s, a, bytes) || refuse(a, bytes, false);
}

static __device__ __noinline__ bool load_in_extent(const Side &s, const void *p, int bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return in_extent(s, a, bytes) || refuse(a, bytes, false);
}

static __device__ __noinline__ bool store_ok(const Side &s, const void *p, int bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return all_logical(s, a, bytes) || refuse(a, bytes, true);
}

#define TR_SIDE(name, ...) const ::tr::dbg::Side name = ::tr::dbg::side(__VA_ARGS__)
#define TR_LOAD_OK(s, p, bytes) ::tr::dbg::load_ok((s), (p), (bytes))
#define TR_LOAD_IN_EXTENT(s, p, bytes) ::tr::dbg::load_in_extent((s), (p), (bytes))
#define TR_STORE_OK(s, p, bytes) ::tr::dbg::store_ok((s), (p), (bytes))

// Host reader of this unit's record: copies it out and clears it.
#define TR_BOUNDS_READER(fn)                                                              \
    cudaError_t fn(::tr::dbg::Record *r) {                                                \
        cudaError_t e = cudaMemcpyFromSymbol(r, ::tr::dbg::g_bounds, sizeof(*r));         \
        if (e != cudaSuccess) return e;                                                   \
        const ::tr::dbg::Record zero{};                                                   \
        return cudaMemcpyToSymbol(::tr::dbg::g_bounds, &zero, sizeof(zero));              \
    }
#else
#define TR_SIDE(name, ...)
#define TR_LOAD_OK(s, p, bytes) true
#define TR_LOAD_IN_EXTENT(s, p, bytes) true
#define TR_STORE_OK(s, p, bytes) true
#define TR_BOUNDS_READER(fn)                 \
    cudaError_t fn(::tr::dbg::Record *r) {   \
        *r = ::tr::dbg::Record{};            \
        return cudaSuccess;                  \
    }
#endif

}  // namespace dbg
}  // namespace tr
