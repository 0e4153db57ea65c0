/* Host-side entry points to the bounds-checked build's guard predicates
 * (csrc/bounds.cuh), so a CPU test can compare them with an independent
 * enumeration of each side's logical elements.  Built as a host-only shared
 * library by tests/test_bounds_guard.py; no device code runs. */
#include "bounds.cuh"

extern "C" {

int guard_all_logical(unsigned long long base, long long batch, long long rows, long long cols,
                      long long ld, long long stride, int esize, unsigned long long addr,
                      int bytes) {
    const tr::dbg::Side s = tr::dbg::side(reinterpret_cast<const void *>(base), batch, rows, cols,
                                          ld, stride, esize);
    return tr::dbg::all_logical(s, uintptr_t(addr), bytes) ? 1 : 0;
}

int guard_in_extent(unsigned long long base, long long batch, long long rows, long long cols,
                    long long ld, long long stride, int esize, unsigned long long addr, int bytes) {
    const tr::dbg::Side s = tr::dbg::side(reinterpret_cast<const void *>(base), batch, rows, cols,
                                          ld, stride, esize);
    return tr::dbg::in_extent(s, uintptr_t(addr), bytes) ? 1 : 0;
}

}  // extern "C"
