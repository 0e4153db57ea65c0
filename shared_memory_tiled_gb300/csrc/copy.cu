// tr_copy: device-to-device copy of a byte range, the bandwidth ceiling the
// transpose is measured against ("Shared memory and the bank conflict",
// section "What to record": the transpose sits next to a copy of the same
// bytes).  Moving N bytes costs N bytes read plus N bytes written, exactly the
// algorithmic traffic of a transpose of N bytes.
#include "bounds.cuh"
#include "launch.cuh"
#include "tr_internal.h"

namespace tr {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // 16-byte vectors in flight per thread

// Body of a copy whose source and destination share their offset modulo 16:
// `head` leading bytes bring both to a 16-byte boundary, then n16 vectors,
// then `tail` bytes.  Every block copies kThreads*kUnroll vectors per turn,
// all loads issued before any store so each thread has 64 bytes in flight.
__global__ void __launch_bounds__(kThreads)
k_copy_aligned(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int head,
               int64_t n16, int tail) {
    pdl_prologue();
    // Debug builds: both ranges as one row of head + 16*n16 + tail bytes.
    TR_SIDE(in_side, in, 1, 1, head + n16 * 16 + tail, head + n16 * 16 + tail, 0, 1);
    TR_SIDE(out_side, out, 1, 1, head + n16 * 16 + tail, head + n16 * 16 + tail, 0, 1);
    auto ld = [&](const uint4 *p) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (TR_LOAD_OK(in_side, p, 16)) v = __ldcs(p);
        return v;
    };
    auto st = [&](uint4 *p, uint4 v) {
        if (TR_STORE_OK(out_side, p, 16)) __stcs(p, v);
    };
    auto move1 = [&](int64_t i) {
        if (TR_LOAD_OK(in_side, in + i, 1) && TR_STORE_OK(out_side, out + i, 1)) out[i] = in[i];
    };
    if (blockIdx.x == 0) {
        if (threadIdx.x < head) move1(threadIdx.x);
        const int64_t t0 = head + n16 * 16;
        if (threadIdx.x < tail) move1(t0 + threadIdx.x);
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(in + head);
    uint4 *dst = reinterpret_cast<uint4 *>(out + head);
    const int64_t per_turn = int64_t(kThreads) * kUnroll;
    for (int64_t base = int64_t(blockIdx.x) * per_turn; base < n16;
         base += int64_t(gridDim.x) * per_turn) {
        uint4 v[kUnroll];
        if (base + per_turn <= n16) {
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) v[k] = ld(src + base + k * kThreads + threadIdx.x);
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) st(dst + base + k * kThreads + threadIdx.x, v[k]);
        } else {
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t idx = base + k * kThreads + threadIdx.x;
                if (idx < n16) v[k] = ld(src + idx);
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t idx = base + k * kThreads + threadIdx.x;
                if (idx < n16) st(dst + idx, v[k]);
            }
        }
    }
}

// Copy for ranges whose offsets differ modulo 16: 4-byte words when the
// offsets agree modulo 4 (after a byte head), single bytes otherwise.
template <typename W>
__global__ void __launch_bounds__(kThreads)
k_copy_narrow(const uint8_t *__restrict__ in, uint8_t *__restrict__ out, int head, int64_t nw,
              int tail) {
    pdl_prologue();
    const int64_t n = head + nw * int64_t(sizeof(W)) + tail;
    TR_SIDE(in_side, in, 1, 1, n, n, 0, 1);
    TR_SIDE(out_side, out, 1, 1, n, n, 0, 1);
    auto move1 = [&](int64_t i) {
        if (TR_LOAD_OK(in_side, in + i, 1) && TR_STORE_OK(out_side, out + i, 1)) out[i] = in[i];
    };
    if (blockIdx.x == 0) {
        if (threadIdx.x < head) move1(threadIdx.x);
        const int64_t t0 = head + nw * int64_t(sizeof(W));
        if (threadIdx.x < tail) move1(t0 + threadIdx.x);
    }
    const W *src = reinterpret_cast<const W *>(in + head);
    W *dst = reinterpret_cast<W *>(out + head);
    for (int64_t idx = int64_t(blockIdx.x) * kThreads + threadIdx.x; idx < nw;
         idx += int64_t(gridDim.x) * kThreads)
        if (TR_LOAD_OK(in_side, src + idx, int(sizeof(W))) &&
            TR_STORE_OK(out_side, dst + idx, int(sizeof(W))))
            dst[idx] = src[idx];
}

int64_t grid_for(int64_t units, int64_t per_block) {
    int64_t g = (units + per_block - 1) / per_block;
    if (g < 1) g = 1;
    const int64_t cap = int64_t(sm_count()) * 64;  // grid-stride beyond this
    return g < cap ? g : cap;
}

}  // namespace

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_copy)

cudaError_t launch_copy(const void *in_, void *out_, size_t bytes, cudaStream_t stream) {
    const uint8_t *in = static_cast<const uint8_t *>(in_);
    uint8_t *out = static_cast<uint8_t *>(out_);
    const uintptr_t a = reinterpret_cast<uintptr_t>(in), b = reinterpret_cast<uintptr_t>(out);
    const int64_t n = int64_t(bytes);
    if (((a ^ b) & 15u) == 0) {
        int head = int((16 - (a & 15u)) & 15u);
        if (head > n) head = int(n);
        const int64_t n16 = (n - head) / 16;
        const int tail = int(n - head - n16 * 16);
        const int64_t grid = grid_for(n16, int64_t(kThreads) * kUnroll);
        return launch_pdl(k_copy_aligned, dim3(unsigned(grid)), dim3(kThreads), 0, stream, in, out,
                          head, n16, tail);
    } else if (((a ^ b) & 3u) == 0) {
        int head = int((4 - (a & 3u)) & 3u);
        if (head > n) head = int(n);
        const int64_t nw = (n - head) / 4;
        const int tail = int(n - head - nw * 4);
        return launch_pdl(k_copy_narrow<uint32_t>, dim3(unsigned(grid_for(nw, kThreads))),
                          dim3(kThreads), 0, stream, in, out, head, nw, tail);
    }
    return launch_pdl(k_copy_narrow<uint8_t>, dim3(unsigned(grid_for(n, kThreads))), dim3(kThreads),
                      0, stream, in, out, 0, n, 0);
}

}  // namespace tr
