// The C-ABI boundary of libtranspose: argument validation, variant choice and
// dispatch to the kernel launchers.  Everything here runs on the host; the
// validation and planning functions make no CUDA call, so argument errors are
// reported without a GPU.
#include "tr_internal.h"

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace tr {
namespace {

thread_local std::string t_last_error;

void set_error(const char *what, cudaError_t e) {
    char buf[512];
    if (e != cudaSuccess)
        std::snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e),
                      cudaGetErrorString(e));
    else
        std::snprintf(buf, sizeof buf, "%s", what);
    t_last_error = buf;
}

// a*b + c with overflow detection; all inputs non-negative.
bool mul_add(int64_t a, int64_t b, int64_t c, int64_t *r) {
    __int128 v = (__int128)a * b + c;
    if (v > INT64_MAX) return false;
    *r = int64_t(v);
    return true;
}

// Elements from the first to one past the last logical element of a side.
bool side_extent(int64_t batch, int64_t lines, int64_t elems, int64_t ld, int64_t stride,
                 int64_t *ext) {
    if (batch == 0 || lines == 0 || elems == 0) {
        *ext = 0;
        return true;
    }
    int64_t e1, e2;
    if (!mul_add(lines - 1, ld, elems, &e1)) return false;
    if (!mul_add(batch - 1, stride, e1, &e2)) return false;
    *ext = e2;
    return true;
}

// Validates the arguments and fills a Problem.  Returns TR_OK, an argument
// error, or (via *empty) that there is nothing to do.
tr_status validate(const tr_args *a, Problem *p, bool *empty) {
    if (!a) return TR_ERR_NULL;
    if (a->reserved != 0) return TR_ERR_UNSUPPORTED;
    if (a->dtype != TR_DTYPE_F32 && a->dtype != TR_DTYPE_BF16) return TR_ERR_UNSUPPORTED;
    if (a->batch < 0 || a->rows < 0 || a->cols < 0) return TR_ERR_BAD_DIM;
    const int esize = a->dtype == TR_DTYPE_F32 ? 4 : 2;
    *empty = a->batch == 0 || a->rows == 0 || a->cols == 0;
    if (*empty) return TR_OK;
    if (!a->in || !a->out) return TR_ERR_NULL;
    // Every kernel accesses whole elements: a pointer off its element
    // boundary would fault on the device.
    if ((reinterpret_cast<uintptr_t>(a->in) | reinterpret_cast<uintptr_t>(a->out)) % esize)
        return TR_ERR_UNSUPPORTED;
    if (a->ld_in < a->cols || a->ld_out < a->rows) return TR_ERR_BAD_LD;
    int64_t min_sin, min_sout;
    if (!mul_add(a->rows - 1, a->ld_in, a->cols, &min_sin) ||
        !mul_add(a->cols - 1, a->ld_out, a->rows, &min_sout))
        return TR_ERR_BAD_DIM;
    if (a->batch > 1 && (a->stride_in < min_sin || a->stride_out < min_sout)) return TR_ERR_BAD_LD;
    int64_t ext_in, ext_out, bytes_in, bytes_out;
    if (!side_extent(a->batch, a->rows, a->cols, a->ld_in, a->stride_in, &ext_in) ||
        !side_extent(a->batch, a->cols, a->rows, a->ld_out, a->stride_out, &ext_out) ||
        !mul_add(ext_in, esize, 0, &bytes_in) || !mul_add(ext_out, esize, 0, &bytes_out))
        return TR_ERR_BAD_DIM;
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(a->in);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(a->out);
    if (i0 + uintptr_t(bytes_in) < i0 || o0 + uintptr_t(bytes_out) < o0) return TR_ERR_BAD_DIM;
    if (i0 < o0 + uintptr_t(bytes_out) && o0 < i0 + uintptr_t(bytes_in)) return TR_ERR_OVERLAP;
    p->in = a->in;
    p->out = a->out;
    p->esize = esize;
    p->batch = a->batch;
    p->rows = a->rows;
    p->cols = a->cols;
    p->ld_in = a->ld_in;
    p->ld_out = a->ld_out;
    p->stride_in = a->batch > 1 ? a->stride_in : a->rows * a->ld_in;
    p->stride_out = a->batch > 1 ? a->stride_out : a->cols * a->ld_out;
    p->stream = reinterpret_cast<cudaStream_t>(a->stream);
    return TR_OK;
}

bool options_valid(const tr_options *o) {
    if (!o) return true;
    if (o->variant < TR_VARIANT_AUTO || o->variant > TR_VARIANT_TMA) return false;
    if (o->pad < 0 || o->pad > 8 || (o->pad > 4 && o->pad != 8)) return false;
    if (o->ctas_per_sm < 0 || o->ctas_per_sm > 8) return false;
    if (o->stages != 0 && (o->stages < 2 || o->stages > 8)) return false;
    if (o->tile_order < 0 || o->tile_order > 1) return false;
    if (o->out_stages != 0 && (o->out_stages < 2 || o->out_stages > 4)) return false;
    if (o->tile_rows < 0 || o->tile_cols < 0 || o->tile_rows > 256 || o->tile_cols > 256)
        return false;
    if (o->schedule < 0 || o->schedule > 4) return false;
    if (o->threads != 0 && o->threads != 32 && o->threads != 64 && o->threads != 128 &&
        o->threads != 256)
        return false;
    return true;
}

// Variant choice (host logic only).  AUTO takes the vectorised swizzled tile,
// the fastest variant measured on GB300 for every alignment class: it uses
// 16-byte accesses on each side that allows them, realigns misaligned output
// rows with warp shuffles, and reads a misaligned input as aligned 16-byte
// chunks realigned on chip (bf16) or with the widest loads each chunk's
// address allows (fp32).  TMA runs only when asked for.
int32_t choose(const Problem &p, const tr_options *o) {
    (void)p;
    const int req = o ? o->variant : TR_VARIANT_AUTO;
    if (req != TR_VARIANT_AUTO) return req;
    return TR_VARIANT_TILE_VEC;
}

// Tile shape (and, unless the caller chose one, block size) AUTO uses for the
// vectorised tile (measured on GB300).  A misaligned bf16 input (aligned
// chunks realigned on chip) takes 64x128 tiles on 128 threads: 16384x16384
// bf16 with input pitch 16385 reaches 6598 GB/s, against 5961 with 128x128 on
// 256 threads, 5848 with 128x128 on 128 and 5566 with 256x64 on 256; with the
// output pitch odd as well, 4363 against 3661 with 128x128 on 256 (4576 since
// the halo rows are realigned too).  Otherwise
// output rows that are not 16-byte aligned (shifted stores) take 128-row tiles,
// 16 chunks wide: 12289x7919 fp32 with output pitch 12289 reaches 6668 GB/s
// with 128x64 against 5849 with 64x64 and 5843 with 128x128; 16384x16384 bf16
// with output pitch 16385 5630 GB/s with 128x128 against 5070 with 256x128,
// 5612 with 64x128 on 128 threads and 5388 with 128x128 on 128.  A
// misaligned fp32 input takes tiles 16 chunks tall and 128 elements wide:
// 7919x12289 fp32 with input pitch 12289 reaches 6751 GB/s with 64x128
// against 5999 with 64x64 and 5952 / 6171 with 128x64 / 64x64 on 128 threads.
void auto_vec_shape(const Problem &p, bool in16, bool out16, VecConfig *cfg) {
    const int v = 16 / p.esize;  // elements per 16-byte chunk
    if (!in16 && p.esize == 2 && cfg->threads == 0) {
        cfg->tile_rows = 64;
        cfg->tile_cols = 128;
        cfg->threads = 128;
    } else if (!out16) {
        cfg->tile_rows = 128;
        cfg->tile_cols = 16 * v;
    } else if (!in16) {
        cfg->tile_rows = 16 * v;
        cfg->tile_cols = 128;
    } else {
        cfg->tile_rows = cfg->tile_cols = 0;  // kernel default: 64x64 fp32, 128x128 bf16
    }
}

// The vector tile's configuration for these options: the caller's tile
// shape, block size, tile order and schedule, with AUTO's shape and block
// size (auto_vec_shape) where no tile shape is given.
VecConfig vec_config(const Problem &p, const tr_options *o, bool in16, bool out16) {
    VecConfig cfg{o ? o->tile_order : 0, o ? o->tile_rows : 0, o ? o->tile_cols : 0,
                  o && o->schedule == 2, o ? o->threads : 0};
    if (cfg.tile_rows == 0 && cfg.tile_cols == 0) auto_vec_shape(p, in16, out16, &cfg);
    return cfg;
}

tr_status run(const tr_args *a, const tr_options *o) {
    Problem p{};
    bool empty = false;
    if (!options_valid(o)) return TR_ERR_UNSUPPORTED;
    tr_status st = validate(a, &p, &empty);
    if (st != TR_OK || empty) return st;
    const int32_t v = choose(p, o);
    const bool in16 = side_aligned16(p.in, p.ld_in, p.stride_in, p.batch, p.esize);
    const bool out16 = side_aligned16(p.out, p.ld_out, p.stride_out, p.batch, p.esize);
    cudaError_t e = cudaSuccess;
    switch (v) {
        case TR_VARIANT_NAIVE_ROW: e = launch_naive(p, true); break;
        case TR_VARIANT_NAIVE_COL: e = launch_naive(p, false); break;
        case TR_VARIANT_TILE_PAD: e = launch_tile_pad(p, o ? o->pad : 1); break;
        case TR_VARIANT_TILE_VEC: {
            if (o && o->schedule >= 3) {
                set_error("schedules 3 and 4 (TMA load pipelines) belong to the TMA variant",
                          cudaSuccess);
                return TR_ERR_UNSUPPORTED;
            }
            const VecConfig cfg = vec_config(p, o, in16, out16);
            const char *why = nullptr;
            e = launch_tile_vec(p, in16, out16, cfg, &why);
            if (e != cudaSuccess && why) {
                set_error(why, cudaSuccess);
                return TR_ERR_UNSUPPORTED;
            }
            break;
        }
        case TR_VARIANT_TMA: {
            if (!in16 || !out16) {
                set_error("TMA needs 16-byte aligned base pointers and pitches on both sides",
                          cudaSuccess);
                return TR_ERR_UNSUPPORTED;
            }
            TmaConfig cfg{o ? o->ctas_per_sm : 0, o ? o->stages : 0, o ? o->tile_order : 0,
                          o ? o->out_stages : 0, o ? o->schedule : 0};
            const char *why = nullptr;
            e = launch_tma(p, cfg, &why);
            if (e != cudaSuccess && why) {
                // e.g. a plane pitch the tensor map cannot describe
                set_error(why, cudaSuccess);
                return TR_ERR_UNSUPPORTED;
            }
            break;
        }
        default: return TR_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) {
        set_error("kernel launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

tr_args make_args(const void *in, void *out, tr_dtype dt, int64_t batch, int64_t rows,
                  int64_t cols, int64_t ld_in, int64_t ld_out, int64_t stride_in,
                  int64_t stride_out, tr_stream_t stream) {
    tr_args a{};
    a.in = in;
    a.out = out;
    a.dtype = dt;
    a.batch = batch;
    a.rows = rows;
    a.cols = cols;
    a.ld_in = ld_in;
    a.ld_out = ld_out;
    a.stride_in = stride_in;
    a.stride_out = stride_out;
    a.stream = stream;
    return a;
}

tr_status run_inplace(void *data, int esize, int64_t batch, int64_t n, int64_t ld,
                      int64_t stride, tr_stream_t stream) {
    if (batch < 0 || n < 0) return TR_ERR_BAD_DIM;
    if (batch == 0 || n == 0) return TR_OK;
    if (!data) return TR_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(data) % esize) return TR_ERR_UNSUPPORTED;
    if (ld < n) return TR_ERR_BAD_LD;
    int64_t plane, ext, bytes;
    if (!mul_add(n - 1, ld, n, &plane)) return TR_ERR_BAD_DIM;
    if (batch > 1 && stride < plane) return TR_ERR_BAD_LD;
    if (!side_extent(batch, n, n, ld, stride, &ext) || !mul_add(ext, esize, 0, &bytes))
        return TR_ERR_BAD_DIM;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(data);
    if (d0 + uintptr_t(bytes) < d0) return TR_ERR_BAD_DIM;
    const cudaError_t e = launch_inplace(data, esize, batch, n, ld, batch > 1 ? stride : n * ld,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_error("in-place transpose launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

}  // namespace

int sm_count() {
    static std::atomic<int> cache[64];  // 0 = not queried yet (zero-initialised: static)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev < 0 || dev >= 64) dev = 0;
    int n = cache[dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        cache[dev].store(n, std::memory_order_release);
    }
    return n;
}

}  // namespace tr

extern "C" {

tr_status tr_transpose_f32(const float *in, float *out, int64_t rows, int64_t cols, int64_t ld_in,
                           int64_t ld_out, tr_stream_t stream) {
    const tr_args a = tr::make_args(in, out, TR_DTYPE_F32, 1, rows, cols, ld_in, ld_out, 0, 0, stream);
    return tr::run(&a, nullptr);
}

tr_status tr_transpose_bf16(const void *in, void *out, int64_t rows, int64_t cols, int64_t ld_in,
                            int64_t ld_out, tr_stream_t stream) {
    const tr_args a = tr::make_args(in, out, TR_DTYPE_BF16, 1, rows, cols, ld_in, ld_out, 0, 0, stream);
    return tr::run(&a, nullptr);
}

tr_status tr_transpose_batched_f32(const float *in, float *out, int64_t batch, int64_t rows,
                                   int64_t cols, int64_t ld_in, int64_t ld_out, int64_t stride_in,
                                   int64_t stride_out, tr_stream_t stream) {
    const tr_args a = tr::make_args(in, out, TR_DTYPE_F32, batch, rows, cols, ld_in, ld_out,
                                    stride_in, stride_out, stream);
    return tr::run(&a, nullptr);
}

tr_status tr_transpose_batched_bf16(const void *in, void *out, int64_t batch, int64_t rows,
                                    int64_t cols, int64_t ld_in, int64_t ld_out, int64_t stride_in,
                                    int64_t stride_out, tr_stream_t stream) {
    const tr_args a = tr::make_args(in, out, TR_DTYPE_BF16, batch, rows, cols, ld_in, ld_out,
                                    stride_in, stride_out, stream);
    return tr::run(&a, nullptr);
}

tr_status tr_transpose_ex(const tr_args *args, const tr_options *opts) {
    return tr::run(args, opts);
}

tr_status tr_transpose_inplace_f32(float *data, int64_t batch, int64_t n, int64_t ld,
                                   int64_t stride, tr_stream_t stream) {
    return tr::run_inplace(data, 4, batch, n, ld, stride, stream);
}

tr_status tr_transpose_inplace_bf16(void *data, int64_t batch, int64_t n, int64_t ld,
                                    int64_t stride, tr_stream_t stream) {
    return tr::run_inplace(data, 2, batch, n, ld, stride, stream);
}

tr_status tr_copy(const void *in, void *out, size_t bytes, tr_stream_t stream) {
    if (bytes == 0) return TR_OK;
    if (!in || !out) return TR_ERR_NULL;
    if (bytes > size_t(INT64_MAX)) return TR_ERR_BAD_DIM;
    const uintptr_t i0 = reinterpret_cast<uintptr_t>(in), o0 = reinterpret_cast<uintptr_t>(out);
    if (i0 + bytes < i0 || o0 + bytes < o0) return TR_ERR_BAD_DIM;
    if (i0 < o0 + bytes && o0 < i0 + bytes) return TR_ERR_OVERLAP;
    const cudaError_t e = tr::launch_copy(in, out, bytes, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tr::set_error("copy launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

tr_status tr_operand_tiles_f32(const float *a, float *out, int64_t m, int64_t k, int64_t lda,
                               int32_t bm, int32_t bk, int32_t pad, tr_stream_t stream) {
    if (m < 0 || k < 0) return TR_ERR_BAD_DIM;
    const bool shape_ok = (bm == 64 || bm == 128) && (bk == 8 || bk == 16 || bk == 32);
    if (!shape_ok || pad > 8) return TR_ERR_UNSUPPORTED;
    if (pad < 0) pad = (32 / bk) % 8;  // the page's padding rule
    if (m == 0 || k == 0) return TR_OK;
    if (!a || !out) return TR_ERR_NULL;
    if (lda < k) return TR_ERR_BAD_LD;
    if (m % bm || k % bk) return TR_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(a) & 15u) || (lda & 3)) return TR_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(out) & 3u) return TR_ERR_UNSUPPORTED;
    int64_t ext_a, bytes_a, bytes_out;
    if (!tr::mul_add(m - 1, lda, k, &ext_a) || !tr::mul_add(ext_a, 4, 0, &bytes_a) ||
        !tr::mul_add(m, k * 4, 0, &bytes_out))
        return TR_ERR_BAD_DIM;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), o0 = reinterpret_cast<uintptr_t>(out);
    if (a0 + uintptr_t(bytes_a) < a0 || o0 + uintptr_t(bytes_out) < o0) return TR_ERR_BAD_DIM;
    if (a0 < o0 + uintptr_t(bytes_out) && o0 < a0 + uintptr_t(bytes_a)) return TR_ERR_OVERLAP;
    const cudaError_t e = tr::launch_operand_tiles(
        reinterpret_cast<const uint32_t *>(a), reinterpret_cast<uint32_t *>(out), m, k, lda, bm, bk,
        pad, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tr::set_error("operand tile launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

tr_status tr_bank_probe(int32_t layout, int32_t reps, int32_t blocks, uint32_t *result,
                        tr_stream_t stream) {
    if (layout < 0 || layout > 3) return TR_ERR_UNSUPPORTED;
    if (reps < 0 || blocks < 0) return TR_ERR_BAD_DIM;
    if (blocks == 0) return TR_OK;
    if (!result) return TR_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(result) & 3u) return TR_ERR_UNSUPPORTED;
    const cudaError_t e = tr::launch_bank_probe(layout, reps, blocks, result,
                                                reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tr::set_error("bank probe launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

tr_status tr_plan_ex(const tr_args *args, const tr_options *opts, tr_plan *plan) {
    if (!plan) return TR_ERR_NULL;
    *plan = tr_plan{};
    tr::Problem p{};
    bool empty = false;
    if (!tr::options_valid(opts)) return TR_ERR_UNSUPPORTED;
    const tr_status st = tr::validate(args, &p, &empty);
    if (st != TR_OK) return st;
    if (empty) {
        p = tr::Problem{args->in, args->out, args->dtype == TR_DTYPE_F32 ? 4 : 2, args->batch,
                        args->rows, args->cols, args->ld_in, args->ld_out, args->stride_in,
                        args->stride_out, nullptr};
    }
    plan->variant = tr::choose(p, opts);
    const bool in16 = tr::side_aligned16(p.in, p.ld_in, p.stride_in, p.batch, p.esize);
    const bool out16 = tr::side_aligned16(p.out, p.ld_out, p.stride_out, p.batch, p.esize);
    plan->vec_in = in16;
    plan->vec_out = out16;
    if (plan->variant == TR_VARIANT_TILE_VEC) {
        if (opts && opts->schedule >= 3) return TR_ERR_UNSUPPORTED;
        const tr::VecConfig cfg = tr::vec_config(p, opts, in16, out16);
        const int v = 16 / p.esize;  // 16 x 16 chunks when a dimension is left to the kernel
        plan->tile_rows = cfg.tile_rows ? cfg.tile_rows : 16 * v;
        plan->tile_cols = cfg.tile_cols ? cfg.tile_cols : 16 * v;
        plan->threads = cfg.threads ? cfg.threads : 256;
        plan->schedule = cfg.prefetch ? 2 : 0;
    } else if (plan->variant == TR_VARIANT_TMA && !(in16 && out16)) {
        return TR_ERR_UNSUPPORTED;
    }
    return TR_OK;
}

int32_t tr_plan_variant(const tr_args *args, const tr_options *opts) {
    tr::Problem p{};
    bool empty = false;
    if (!tr::options_valid(opts)) return -int32_t(TR_ERR_UNSUPPORTED);
    const tr_status st = tr::validate(args, &p, &empty);
    if (st != TR_OK) return -int32_t(st);
    if (empty) {
        // Nothing would launch; report the choice for the same pointers and pitches.
        p = tr::Problem{args->in, args->out, args->dtype == TR_DTYPE_F32 ? 4 : 2, args->batch,
                        args->rows, args->cols, args->ld_in, args->ld_out, args->stride_in,
                        args->stride_out, nullptr};
    }
    return tr::choose(p, opts);
}

tr_status tr_selftest_bounded_wait(int32_t arrive, int64_t limit_ns, tr_stream_t stream) {
    if (limit_ns <= 0 || limit_ns > 2000000000LL) return TR_ERR_BAD_DIM;
    const cudaError_t e =
        tr::launch_wait_selftest(arrive != 0, limit_ns, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tr::set_error("self-test launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

tr_status tr_device_status(void) {
    unsigned v = 0;
    const cudaError_t e = tr::read_and_clear_fault(&v);
    if (e != cudaSuccess) {
        tr::set_error("reading the device fault flag failed", e);
        return TR_ERR_CUDA;
    }
    return v ? TR_ERR_TIMEOUT : TR_OK;
}

tr_status tr_debug_bounds(tr_bounds_report *report) {
    if (!report) return TR_ERR_NULL;
    *report = tr_bounds_report{};
    if (!tr::bounds_checked_build()) {
        tr::set_error("the library was built without bounds checks (TR_DEBUG)", cudaSuccess);
        return TR_ERR_UNSUPPORTED;
    }
    tr::BoundsSummary sum{};
    const cudaError_t e = tr::read_and_clear_bounds(&sum);
    if (e != cudaSuccess) {
        tr::set_error("reading the bounds-check records failed", e);
        return TR_ERR_CUDA;
    }
    report->refused = int64_t(sum.refused);
    report->first_address = sum.first_addr;
    report->first_bytes = int32_t(sum.first_bytes);
    report->first_store = int32_t(sum.first_store);
    return TR_OK;
}

tr_status tr_debug_bounds_selftest(uint64_t base, tr_stream_t stream) {
    if (!tr::bounds_checked_build()) {
        tr::set_error("the library was built without bounds checks (TR_DEBUG)", cudaSuccess);
        return TR_ERR_UNSUPPORTED;
    }
    const cudaError_t e =
        tr::launch_bounds_selftest(uintptr_t(base), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        tr::set_error("bounds self-test launch failed", e);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

const char *tr_status_string(tr_status s) {
    switch (s) {
        case TR_OK: return "success";
        case TR_ERR_NULL: return "NULL pointer with a nonzero size";
        case TR_ERR_BAD_DIM: return "negative or overflowing dimension";
        case TR_ERR_BAD_LD: return "row or plane pitch below its minimum";
        case TR_ERR_OVERLAP: return "input and output ranges overlap";
        case TR_ERR_UNSUPPORTED: return "variant or option not supported for these arguments";
        case TR_ERR_CUDA: return "CUDA error (see tr_last_error)";
        case TR_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    }
    return "unknown status";
}

const char *tr_last_error(void) { return tr::t_last_error.c_str(); }

int32_t tr_version(void) { return 1 * 10000 + 0 * 100 + 0; }

}  // extern "C"
