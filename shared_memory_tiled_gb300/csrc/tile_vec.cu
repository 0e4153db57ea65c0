// Dispatch of the vectorised swizzled tile (kernel in tile_vec_kernel.cuh)
// to its per-type, per-schedule instantiation units.
#include "tr_internal.h"

namespace tr {

cudaError_t launch_vec_u32(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                           const char **why);
cudaError_t launch_vec_u32_prefetch(const Problem &p, bool vec_in, bool vec_out,
                                    const VecConfig &cfg, const char **why);
cudaError_t launch_vec_u16(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                           const char **why);
cudaError_t launch_vec_u16_prefetch(const Problem &p, bool vec_in, bool vec_out,
                                    const VecConfig &cfg, const char **why);

cudaError_t launch_tile_vec(const Problem &p, bool vec_in, bool vec_out, const VecConfig &cfg,
                            const char **why) {
    if (p.esize == 4)
        return cfg.prefetch ? launch_vec_u32_prefetch(p, vec_in, vec_out, cfg, why)
                            : launch_vec_u32(p, vec_in, vec_out, cfg, why);
    return cfg.prefetch ? launch_vec_u16_prefetch(p, vec_in, vec_out, cfg, why)
                        : launch_vec_u16(p, vec_in, vec_out, cfg, why);
}

}  // namespace tr
