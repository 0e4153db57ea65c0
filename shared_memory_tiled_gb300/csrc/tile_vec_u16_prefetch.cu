// Instantiations of the vectorised swizzled tile: bf16 persistent prefetching blocks.
#include "tile_vec_kernel.cuh"

namespace tr {

cudaError_t launch_vec_u16_prefetch(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                           const char **why) {
    return vec::launch_typed<uint16_t, true>(p, vec_in, vec_out, cfg, why);
}

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_vec_u16_prefetch)

}  // namespace tr
