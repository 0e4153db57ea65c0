// Internal declarations shared by the host API and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "transpose.h"

namespace tr {

// One validated transpose problem (sizes and pitches in elements).
struct Problem {
    const void *in;
    void *out;
    int esize;                 // 4 (fp32 bits) or 2 (bf16 bits)
    int64_t batch, rows, cols;
    int64_t ld_in, ld_out;
    int64_t stride_in, stride_out;
    cudaStream_t stream;
};

struct TmaConfig {
    int ctas_per_sm;   // 0 = as many as fit
    int stages;        // input pipeline depth, 0 = default
    int tile_order;    // 0 row-major, 1 diagonal
    int out_stages;    // output buffers, 0 = default
    int schedule;      // 0 default (per-warp), 1 CTA-wide pipeline, 2 per-warp pipelines,
                       // 3 per-warp TMA loads with register stores, 4 warp-specialised
                       // producer warp + consumer warps with register stores
};

// True when the side's base pointer, row pitch and (for batch > 1) plane pitch
// are all multiples of 16 bytes, so 16-byte vector or TMA accesses are legal.
inline bool side_aligned16(const void *base, int64_t ld, int64_t stride, int64_t batch,
                           int esize) {
    if (reinterpret_cast<uintptr_t>(base) & 15u) return false;
    if ((ld * esize) & 15) return false;
    if (batch > 1 && ((stride * esize) & 15)) return false;
    return true;
}

struct VecConfig {
    int tile_order;    // 0 row-major, 1 diagonal
    int tile_rows;     // tile shape in elements, 0 = default
    int tile_cols;
    bool prefetch;     // persistent blocks that prefetch their next tile
    int threads;       // threads per block (32, 64, 128 or 256), 0 = default
};

// Launchers: each returns the CUDA error of the launch (cudaSuccess when fine).
cudaError_t launch_naive(const Problem &p, bool read_coalesced);
cudaError_t launch_tile_pad(const Problem &p, int pad);
// `why` receives a static message when the configuration itself is refused.
cudaError_t launch_tile_vec(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                            const char **why);
// TMA path: may fail in tensor-map encoding (driver error) as well as launch.
// `why` receives a static message for non-CUDA failures.
cudaError_t launch_tma(const Problem &p, const TmaConfig &cfg, const char **why);
cudaError_t launch_copy(const void *in, void *out, size_t bytes, cudaStream_t stream);
cudaError_t launch_bank_probe(int layout, int reps, int blocks, uint32_t *result,
                              cudaStream_t stream);
cudaError_t launch_operand_tiles(const uint32_t *a, uint32_t *out, int64_t m, int64_t k,
                                 int64_t lda, int bm, int bk, int pad, cudaStream_t stream);
cudaError_t launch_inplace(void *data, int esize, int64_t batch, int64_t n, int64_t ld,
                           int64_t stride, cudaStream_t stream);

// One warp waiting on an mbarrier that completes only when `arrive` is set;
// otherwise the bounded wait runs out after limit_ns and raises the fault flag.
cudaError_t launch_wait_selftest(bool arrive, int64_t limit_ns, cudaStream_t stream);

// Device-side fault flag (bounded waits that ran out).  Reads and clears it.
cudaError_t read_and_clear_fault(unsigned *value);

// Number of SMs of the current device (cached per device).
int sm_count();

// Debug-build bounds checks (bounds.cuh): the merged record of every unit.
struct BoundsSummary {
    unsigned long long refused;     // accesses refused since the last read
    unsigned long long first_addr;  // one refused access (the first a unit recorded)
    unsigned first_bytes;
    unsigned first_store;
};
// Whether the library was compiled with the checks (TR_DEBUG).
bool bounds_checked_build();
// Synchronizes the current device, then reads and clears every unit's record.
cudaError_t read_and_clear_bounds(BoundsSummary *sum);
// The guards' self-test (debug builds; cudaErrorNotSupported otherwise):
// `base` is a made-up address the kernel never dereferences.
cudaError_t launch_bounds_selftest(uintptr_t base, cudaStream_t stream);

}  // namespace tr
