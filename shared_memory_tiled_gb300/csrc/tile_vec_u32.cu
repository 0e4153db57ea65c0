// Instantiations of the vectorised swizzled tile: fp32 one tile per block.
#include "tile_vec_kernel.cuh"

namespace tr {

cudaError_t launch_vec_u32(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                           const char **why) {
    return vec::launch_typed<uint32_t, false>(p, vec_in, vec_out, cfg, why);
}

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_vec_u32)

}  // namespace tr
