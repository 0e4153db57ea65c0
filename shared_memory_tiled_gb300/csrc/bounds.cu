// Debug-build bounds checks: the host side that gathers every translation
// unit's record of refused accesses, and a self-test of the guards that
// touches no memory.  In a release build the records are always empty and
// the self-test is not available.
#include "bounds.cuh"
#include "tr_internal.h"

namespace tr {

// One reader per unit whose kernels make guarded accesses.
cudaError_t read_bounds_vec_u32(dbg::Record *r);
cudaError_t read_bounds_vec_u32_prefetch(dbg::Record *r);
cudaError_t read_bounds_vec_u16(dbg::Record *r);
cudaError_t read_bounds_vec_u16_prefetch(dbg::Record *r);
cudaError_t read_bounds_lsu(dbg::Record *r);
cudaError_t read_bounds_tma(dbg::Record *r);
cudaError_t read_bounds_inplace(dbg::Record *r);
cudaError_t read_bounds_copy(dbg::Record *r);
cudaError_t read_bounds_operand_tiles(dbg::Record *r);
cudaError_t read_bounds_bank_probe(dbg::Record *r);

namespace {

// The self-test's record lives in this unit.
TR_BOUNDS_READER(read_bounds_selftest)

#ifdef TR_DEBUG
// One thread asks the guards about five accesses to a side that is never
// dereferenced (the guards only compute): 2 planes of 3 x 5 four-byte
// elements, row pitch 8, plane pitch 32, at a made-up base.  Expected:
//   load  element (1, 2, 4), 4 bytes           -> accepted (logical)
//   load  element (1, 2, 5), 4 bytes           -> refused (column 5 of 5)
//   load  the extent's last 16 bytes           -> accepted (in the extent)
//   store elements (0, 1, 0..3), 16 bytes      -> accepted (logical)
//   store elements (0, 0, 3..6), 16 bytes      -> refused (columns 5, 6)
// so the record holds 2 refusals, the first at element (1, 2, 5).
__global__ void k_bounds_selftest(uintptr_t base) {
    const dbg::Side s = dbg::side(reinterpret_cast<const void *>(base), 2, 3, 5, 8, 32, 4);
    const uint64_t ext = dbg::extent_bytes(s);
    auto at = [&](int64_t e) { return reinterpret_cast<const void *>(base + uintptr_t(e) * 4); };
    dbg::load_ok(s, at(32 + 2 * 8 + 4), 4);
    dbg::load_ok(s, at(32 + 2 * 8 + 5), 4);
    dbg::load_in_extent(s, reinterpret_cast<const void *>(base + ext - 16), 16);
    dbg::store_ok(s, at(8), 16);
    dbg::store_ok(s, at(3), 16);
}
#endif

}  // namespace

bool bounds_checked_build() {
#ifdef TR_DEBUG
    return true;
#else
    return false;
#endif
}

cudaError_t launch_bounds_selftest(uintptr_t base, cudaStream_t stream) {
#ifdef TR_DEBUG
    k_bounds_selftest<<<1, 1, 0, stream>>>(base);
    return cudaGetLastError();
#else
    (void)base;
    (void)stream;
    return cudaErrorNotSupported;
#endif
}

cudaError_t read_and_clear_bounds(BoundsSummary *sum) {
    *sum = BoundsSummary{};
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    cudaError_t (*const readers[])(dbg::Record *) = {
        read_bounds_vec_u32, read_bounds_vec_u32_prefetch, read_bounds_vec_u16,
        read_bounds_vec_u16_prefetch, read_bounds_lsu, read_bounds_tma, read_bounds_inplace,
        read_bounds_copy, read_bounds_operand_tiles, read_bounds_bank_probe,
        read_bounds_selftest};
    for (auto read : readers) {
        dbg::Record r{};
        e = read(&r);
        if (e != cudaSuccess) return e;
        if (r.count && !sum->refused) {
            sum->first_addr = r.first_addr;
            sum->first_bytes = r.first_bytes;
            sum->first_store = r.first_store;
        }
        sum->refused += r.count;
    }
    return cudaSuccess;
}

}  // namespace tr
