// Instantiations of the vectorised swizzled tile: bf16 one tile per block.
#include "tile_vec_kernel.cuh"

namespace tr {

cudaError_t launch_vec_u16(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                           const char **why) {
    return vec::launch_typed<uint16_t, false>(p, vec_in, vec_out, cfg, why);
}

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_vec_u16)

}  // namespace tr
