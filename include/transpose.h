/*
 * libtranspose -- out-of-place matrix transpose for GB300 (sm_103a).
 *
 * What it computes.  For every batch plane b < batch, input row i < rows and
 * input column j < cols (all sizes and pitches in ELEMENTS):
 *
 *     out[b*stride_out + j*ld_out + i] = in[b*stride_in + i*ld_in + j]
 *
 * This is the operation of "Shared memory and the bank conflict"
 * (roobli.org, kernels-from-zero 03), section "Turn the tile around on chip":
 * a block reads a tile of the input by rows, turns it around in on-chip shared
 * memory and writes it out by rows.  "Shared-memory tiling and bank
 * conflicts" (intro-to-ai-systems-performance, shared-memory chapter),
 * "Worked example", fixes that global coordinates stay logical and that any
 * padding lives only in on-chip storage, so the result is the plain transpose
 * above whatever tile layout a kernel uses.
 *
 * Conventions shared by every entry point:
 *   - Elements are moved as raw bit patterns: the fp32 entry points move
 *     32-bit words and the bf16 entry points 16-bit words, with no arithmetic
 *     on them, so NaN payloads, signed zeros and subnormals survive unchanged.
 *   - rows/cols describe the INPUT plane (rows x cols, row pitch ld_in); the
 *     output plane is cols x rows with row pitch ld_out.  Required:
 *     ld_in >= cols, ld_out >= rows.  For batched calls with batch > 1 the
 *     plane pitches must keep planes apart:
 *     stride_in >= (rows-1)*ld_in + cols and stride_out >= (cols-1)*ld_out + rows.
 *   - Only the logical output elements are written; pitch padding of the
 *     output keeps whatever it held.
 *   - `in` and `out` are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory in any call.  Each must sit on a boundary of
 *     its element size (4 bytes for fp32, 2 for bf16), else the call returns
 *     TR_ERR_UNSUPPORTED; beyond that any base address and pitch is accepted.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and do not synchronize.
 *   - The transpose and copy kernels are launched with programmatic stream
 *     serialization: one may be scheduled while the previous kernel in the
 *     stream is still draining, and it waits for that kernel to complete
 *     before touching memory, so results follow plain stream order.  They
 *     signal their dependents at start, so a kernel that the caller launches
 *     after them WITH programmatic stream serialization must itself wait
 *     (cudaGridDependencySynchronize) before reading their output; kernels
 *     launched without it are ordered as usual.
 *   - Calls can be captured into a CUDA graph and replayed.  The first call
 *     of a configuration on a device sets kernel attributes (shared-memory
 *     limits, occupancy), so make it once before capturing.
 *   - A zero dimension returns TR_OK without launching anything.  A negative
 *     dimension returns TR_ERR_BAD_DIM, a pitch below its minimum
 *     TR_ERR_BAD_LD, a NULL pointer with a nonzero size TR_ERR_NULL, and any
 *     byte overlap between the input and output extents TR_ERR_OVERLAP (the
 *     operation is out-of-place).  Argument errors are detected on the host
 *     before any CUDA call.
 *   - A CUDA launch or driver failure returns TR_ERR_CUDA; tr_last_error()
 *     then describes it (per host thread).
 *   - Every wait on an mbarrier inside a kernel is bounded.  A wait that runs
 *     out records a device-side fault flag and the kernel returns early;
 *     tr_device_status() reports it as TR_ERR_TIMEOUT.
 */
#ifndef LIBTRANSPOSE_TRANSPOSE_H
#define LIBTRANSPOSE_TRANSPOSE_H

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden symbol visibility; the declarations below
 * are the only symbols it exports. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA headers. */
typedef struct CUstream_st *tr_stream_t;

typedef enum tr_status {
    TR_OK = 0,
    TR_ERR_NULL = 1,         /* NULL pointer with a nonzero size                       */
    TR_ERR_BAD_DIM = 2,      /* negative size, or a size/extent that overflows int64   */
    TR_ERR_BAD_LD = 3,       /* row or plane pitch below its minimum                   */
    TR_ERR_OVERLAP = 4,      /* input and output byte extents overlap                  */
    TR_ERR_UNSUPPORTED = 5,  /* requested variant cannot run on these arguments        */
    TR_ERR_CUDA = 6,         /* CUDA runtime/driver error; see tr_last_error()         */
    TR_ERR_TIMEOUT = 7       /* a bounded in-kernel wait ran out (tr_device_status)    */
} tr_status;

/* Element width of a transpose. */
typedef enum tr_dtype {
    TR_DTYPE_F32 = 0,        /* 4-byte elements (fp32 bit patterns)  */
    TR_DTYPE_BF16 = 1        /* 2-byte elements (bf16 bit patterns)  */
} tr_dtype;

/* Kernel variants.  All give bit-identical results; they differ in how the
 * tile is staged.  AUTO picks the fastest one the arguments allow. */
typedef enum tr_variant {
    TR_VARIANT_AUTO = 0,
    /* One element per thread, no shared memory; reads coalesced, writes strided
     * down a column ("episode 02" of the kernels-from-zero series). */
    TR_VARIANT_NAIVE_ROW = 1,
    /* One element per thread, no shared memory; reads strided, writes coalesced. */
    TR_VARIANT_NAIVE_COL = 2,
    /* 32 x 32 tile, 32 x 8 threads, one element per access, shared row pitch of
     * 32 + pad elements ("Shared memory and the bank conflict", kernel
     * transpose_tiled; pad = 0 is its unpadded width-32 form). */
    TR_VARIANT_TILE_PAD = 3,
    /* 16-byte global loads and stores, XOR-swizzled shared tile read with
     * 16-byte accesses, register micro-transpose (4x4 fp32, 8x8 bf16). */
    TR_VARIANT_TILE_VEC = 4,
    /* TMA tile loads and stores with the hardware 128-byte swizzle, persistent
     * CTAs and an mbarrier pipeline.  Needs 16-byte aligned bases and pitches. */
    TR_VARIANT_TMA = 5
} tr_variant;

/* Tuning knobs for tr_transpose_ex.  Zero-initialise for defaults.
 * TILE_VEC tile shapes (rows x cols, elements) with 256 threads: fp32 64x64
 * (default), 128x32, 128x64, 64x128, 128x128; bf16 128x128 (default), 256x64,
 * 256x128, 128x256.  With 128 threads: fp32 64x64, 32x64, 128x64; bf16 128x128,
 * 64x128.  With 64 threads: fp32 32x64, 64x32; bf16 64x128, 128x64.  With 32
 * threads (one warp, so the tile barrier is a warp barrier): fp32 32x32,
 * bf16 64x64.  Other combinations return TR_ERR_UNSUPPORTED.  With
 * tile_rows = tile_cols = 0 the shape follows the alignment of the two sides:
 * bf16 64x128 on 128 threads when input rows do not start on 16-byte
 * boundaries (unless `threads` is set); else 128 rows x 16 chunks (fp32
 * 128x64, bf16 128x128) when output rows do not; fp32 64x128 (bf16 128x128
 * with `threads` set) when only input rows do not; the 256-thread default
 * otherwise. */
typedef struct tr_options {
    int32_t variant;      /* tr_variant                                                  */
    int32_t pad;          /* TILE_PAD: shared row pitch is 32 + pad elements, 0..8        */
    int32_t ctas_per_sm;  /* TMA: persistent CTAs per SM, 0 = as many as fit (max 8)      */
    int32_t stages;       /* TMA: input pipeline depth 2..8, 0 = default                  */
    int32_t tile_order;   /* TMA/TILE_VEC: 0 = row-major tile walk, 1 = diagonal          */
    int32_t out_stages;   /* TMA: output buffers (stores in flight) 2..4, 0 = default     */
    int32_t tile_rows;    /* TILE_VEC: tile rows in elements, 0 = default (see below)     */
    int32_t tile_cols;    /* TILE_VEC: tile columns in elements, 0 = default              */
    int32_t schedule;     /* TILE_VEC: 0 = default, 1 = one tile per block,
                           *   2 = persistent blocks that prefetch their next tile;
                           * TMA: 0 = default, 1 = one pipeline per block (64x64 fp32 /
                           *   128x128 bf16 tiles, one block barrier per tile),
                           *   2 = one pipeline per warp (32x32 fp32 / 64x64 bf16 tiles),
                           *   3 = per-warp TMA loads, register transpose and 16-byte
                           *       global stores (no output buffer, no TMA store),
                           *   4 = warp-specialised: one producer warp keeps up to
                           *       `stages` 64x64 fp32 / 128x128 bf16 tile loads in
                           *       flight on full/empty mbarriers, eight consumer warps
                           *       transpose and store with 16-byte global stores     */
    int32_t threads;      /* TILE_VEC: threads per block, 32, 64, 128 or 256, 0 = default */
} tr_options;

/* Full argument set of one (possibly batched) transpose; see the conventions
 * above.  For a single matrix set batch = 1 (stride_in/stride_out ignored). */
typedef struct tr_args {
    const void *in;
    void *out;
    int32_t dtype;        /* tr_dtype */
    int32_t reserved;     /* must be zero */
    int64_t batch, rows, cols;
    int64_t ld_in, ld_out;
    int64_t stride_in, stride_out;
    tr_stream_t stream;
} tr_args;

/* Single-matrix transpose of fp32 bit patterns: out[j*ld_out + i] = in[i*ld_in + j]
 * for i < rows, j < cols ("Shared memory and the bank conflict", "Turn the tile
 * around on chip": read a tile by rows, turn it around on chip, write it by
 * rows).  `in` is rows x cols with row pitch ld_in (>= cols), `out` is cols x
 * rows with row pitch ld_out (>= rows); both device memory owned by the caller.
 * Errors: TR_ERR_BAD_DIM, TR_ERR_BAD_LD, TR_ERR_NULL, TR_ERR_OVERLAP before any
 * launch, TR_ERR_CUDA if the launch fails (conventions at the top). */
tr_status tr_transpose_f32(const float *in, float *out, int64_t rows, int64_t cols,
                           int64_t ld_in, int64_t ld_out, tr_stream_t stream);

/* Single-matrix transpose of bf16 bit patterns (`in`/`out` point at 16-bit
 * elements, moved as raw 16-bit words -- never converted, so every NaN payload
 * survives); otherwise exactly tr_transpose_f32. */
tr_status tr_transpose_bf16(const void *in, void *out, int64_t rows, int64_t cols,
                            int64_t ld_in, int64_t ld_out, tr_stream_t stream);

/* Batched transpose [batch, rows, cols] -> [batch, cols, rows] of fp32 bit
 * patterns: each plane is transposed as in tr_transpose_f32; plane b of the
 * input starts at in + b*stride_in, of the output at out + b*stride_out
 * (elements).  For batch > 1 the plane pitches must keep planes apart
 * (stride_in >= (rows-1)*ld_in + cols, stride_out >= (cols-1)*ld_out + rows,
 * else TR_ERR_BAD_LD); no byte of the input extent may overlap the output
 * extent (TR_ERR_OVERLAP). */
tr_status tr_transpose_batched_f32(const float *in, float *out, int64_t batch, int64_t rows,
                                   int64_t cols, int64_t ld_in, int64_t ld_out,
                                   int64_t stride_in, int64_t stride_out, tr_stream_t stream);

/* Batched transpose of bf16 bit patterns; same arguments, layout and errors
 * as the fp32 form. */
tr_status tr_transpose_batched_bf16(const void *in, void *out, int64_t batch, int64_t rows,
                                    int64_t cols, int64_t ld_in, int64_t ld_out,
                                    int64_t stride_in, int64_t stride_out, tr_stream_t stream);

/* Any transpose of the forms above with an explicit variant and tuning
 * (`args` carries the element type, sizes, pitches and stream; `opts` may be
 * NULL = AUTO).  Same result and argument errors as the fixed entry points;
 * TR_ERR_UNSUPPORTED when an option is out of range or the requested variant
 * cannot run on these arguments (e.g. TMA with a pitch that is not a multiple
 * of 16 bytes, or a tile shape the variant does not have); tr_last_error()
 * then says which. */
tr_status tr_transpose_ex(const tr_args *args, const tr_options *opts);

/* In-place transpose of `batch` square n x n planes of fp32 bit patterns:
 * element (i, j) of plane b (at data + b*stride + i*ld + j) exchanges places
 * with element (j, i); the diagonal and all pitch padding stay as they were.
 * Requires ld >= n and, for batch > 1, stride >= (n-1)*ld + n (stride is
 * ignored when batch == 1).  Each pair of mirror tiles is read completely
 * before either is written, so the call is safe on one buffer; the planes
 * of one call must not overlap each other.  Same errors as above (no
 * TR_ERR_OVERLAP: aliasing is the point).  Not part of the pages' kernels:
 * it is the square special case in which the output buffer is the input. */
tr_status tr_transpose_inplace_f32(float *data, int64_t batch, int64_t n, int64_t ld,
                                   int64_t stride, tr_stream_t stream);

/* In-place transpose of square planes of bf16 bit patterns; as above. */
tr_status tr_transpose_inplace_bf16(void *data, int64_t batch, int64_t n, int64_t ld,
                                    int64_t stride, tr_stream_t stream);

/* Device-to-device copy of `bytes` bytes, the bandwidth ceiling the transpose
 * is compared against ("Shared memory and the bank conflict", section "What to
 * record": the transpose timings sit next to a copy of the same bytes).
 * Any alignment; the ranges must not overlap (TR_ERR_OVERLAP). */
tr_status tr_copy(const void *in, void *out, size_t bytes, tr_stream_t stream);

/* Transposed operand tiles: the shared-memory load stage of the padded SGEMM
 * of "Padded Shared Memory: Eliminating Bank Conflicts" on its own.  Each
 * BM x BK tile of the row-major M x K fp32 matrix `a` (row pitch lda) is
 * staged transposed in shared memory with a row pitch of BM + pad words and
 * written, unpadded, to `out`: tile (mt, kt) at out + (mt*(K/BK) + kt)*BK*BM,
 * element (k, m) at k*BM + m, i.e. out holds A[mt*BM + m][kt*BK + k].
 * BM in {64, 128}, BK in {8, 16, 32}, pad in 0..8 or negative for the page's
 * rule (32 / BK) % 8.  M and K must be multiples of BM and BK, `a` 16-byte
 * aligned, lda a multiple of 4 (float4 loads) and `out` 4-byte aligned, else
 * TR_ERR_UNSUPPORTED; `out` (M*K words) must not overlap `a` (TR_ERR_OVERLAP).  Device pointers,
 * caller-owned; asynchronous on `stream`. */
tr_status tr_operand_tiles_f32(const float *a, float *out, int64_t m, int64_t k, int64_t lda,
                               int32_t bm, int32_t bk, int32_t pad, tr_stream_t stream);

/* Column-read microbenchmark of a 32 x 32 shared tile of 4-byte words
 * ("Shared-memory tiling and bank conflicts", "Expose a shared-memory bank
 * conflict").  `blocks` blocks of 256 threads each fill one tile holding value
 * row*32 + col at logical (row, col) in the chosen layout, then lane l of warp
 * w reads logical (l, (r + w) % 32) for r < reps and folds the values
 * (acc = rotl(acc, 1) ^ value, starting from 0):
 *   layout 0: row pitch 32 (a column read is a 32-way bank conflict)
 *   layout 1: row pitch 33 (the padded tile, conflict-free)
 *   layout 2: pitch 32 with column index XOR row (swizzled, conflict-free)
 *   layout 3: pitch 32 read along rows, logical ((r + w) % 32, l) (reference)
 * `result` (device, blocks*256 words, 4-byte aligned, caller-owned) receives each thread's
 * fold, so the reads cannot be optimised away and the run is checkable.
 * Time it with events on `stream` to compare layouts. */
tr_status tr_bank_probe(int32_t layout, int32_t reps, int32_t blocks, uint32_t *result,
                        tr_stream_t stream);

/* Host-only planning: the variant tr_transpose_ex would run for these
 * arguments and options (a tr_variant value, never AUTO), or a negative
 * tr_status on invalid arguments.  Makes no CUDA call. */
int32_t tr_plan_variant(const tr_args *args, const tr_options *opts);

/* What tr_transpose_ex would launch, as tr_plan_ex reports it. */
typedef struct tr_plan {
    int32_t variant;    /* tr_variant, never AUTO                                          */
    int32_t tile_rows;  /* TILE_VEC: tile rows in elements (0 for the other variants)       */
    int32_t tile_cols;  /* TILE_VEC: tile columns in elements                               */
    int32_t threads;    /* TILE_VEC: threads per block                                     */
    int32_t schedule;   /* TILE_VEC: 0 one tile per block, 2 persistent with prefetch       */
    int32_t vec_in;     /* 1 when input rows, base and plane pitch sit on 16-byte boundaries */
    int32_t vec_out;    /* the same for the output (else TILE_VEC shifts its stores)        */
} tr_plan;

/* Host-only planning in full: fills *plan with the variant and, for the
 * vector tile, the tile shape and block size that AUTO or the options
 * request (see tr_options), and which sides allow 16-byte accesses.  Returns
 * TR_OK, TR_ERR_NULL for a NULL plan, or the argument error tr_transpose_ex
 * would return (TR_ERR_UNSUPPORTED for TMA on a misaligned side or a TMA
 * schedule on the vector tile).  A tile shape and block size that the vector
 * tile does not have (see tr_options) are reported as requested and refused
 * by tr_transpose_ex.  Makes no CUDA call. */
tr_status tr_plan_ex(const tr_args *args, const tr_options *opts, tr_plan *plan);

/* Reads and clears the device-side fault flag of the CURRENT device after
 * synchronizing it: TR_ERR_TIMEOUT if a bounded in-kernel wait ran out since
 * the last call, TR_OK otherwise (TR_ERR_CUDA if the read itself fails). */
tr_status tr_device_status(void);

/* Exercises the failure path of the bounded in-kernel waits without any
 * fault: one warp waits on an mbarrier phase that completes only when
 * `arrive` is nonzero.  With arrive == 0 the wait runs out after limit_ns
 * nanoseconds (1 ns .. 2 s, else TR_ERR_BAD_DIM), the kernel raises the same
 * device fault flag the transpose kernels raise and returns, so a following
 * tr_device_status() reports TR_ERR_TIMEOUT; with arrive != 0 it reports TR_OK.
 * Asynchronous on `stream`. */
tr_status tr_selftest_bounded_wait(int32_t arrive, int64_t limit_ns, tr_stream_t stream);

/* Record of the bounds checks of a debug build (see tr_debug_bounds). */
typedef struct tr_bounds_report {
    int64_t refused;          /* accesses refused since the last read (0 = none)           */
    uint64_t first_address;   /* device address of one refused access (the first recorded) */
    int32_t first_bytes;      /* its width in bytes                                        */
    int32_t first_store;      /* 1 = a store (output side), 0 = a load (input side)        */
} tr_bounds_report;

/* Debug builds only: the library compiled with TR_DEBUG defined checks every
 * global load and store of every kernel before making it -- loads against the
 * input's logical elements (or, for the bf16 loads that realign misaligned
 * rows on chip, against the input's extent from its first to its last
 * logical element), stores against the output's logical elements -- and
 * skips and counts any access that fails ("Shared memory and the bank
 * conflict", "The barrier": an indexing mistake can leave the result right
 * most of the time).  Nothing traps.  This call synchronizes the current
 * device, then fills *report with the accesses refused since the last call
 * and clears the record.  Returns TR_OK; TR_ERR_UNSUPPORTED (report zeroed)
 * in a release build, which makes no checks; TR_ERR_NULL for a NULL report;
 * TR_ERR_CUDA if the device cannot be read. */
tr_status tr_debug_bounds(tr_bounds_report *report);

/* Debug builds only: tests the guards themselves without touching memory.
 * One thread asks them about five accesses to a made-up side that it never
 * dereferences (2 planes of 3 x 5 fp32 elements, row pitch 8, plane pitch
 * 32, at address `base`): a logical load, a load one column past a row, a
 * load of the extent's last 16 bytes, a logical 16-byte store and a 16-byte
 * store that runs two columns past a row.  A following tr_debug_bounds then
 * reports exactly 2 refusals, the first a 4-byte load at base + 212.
 * TR_ERR_UNSUPPORTED in a release build; asynchronous on `stream`. */
tr_status tr_debug_bounds_selftest(uint64_t base, tr_stream_t stream);

/* Static description of a status code (never NULL). */
const char *tr_status_string(tr_status status);

/* Description of the last TR_ERR_CUDA / TR_ERR_UNSUPPORTED on this host
 * thread, or "" (never NULL; valid until the next call on this thread). */
const char *tr_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int32_t tr_version(void);

#ifdef __cplusplus
}
#endif

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#endif /* LIBTRANSPOSE_TRANSPOSE_H */
