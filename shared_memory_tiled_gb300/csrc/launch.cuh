// Programmatic dependent launch for the transpose and copy kernels.
//
// Back-to-back kernels in one stream normally leave a gap: the next grid is
// launched only after the previous one has completed, and its blocks then
// ramp up from an empty machine.  Launched with programmatic stream
// serialization, a kernel may be scheduled as soon as every block of the
// previous kernel has signalled `griddepcontrol.launch_dependents` (or
// exited), so its blocks become resident while the previous kernel's last
// blocks drain.  Each kernel begins with `griddepcontrol.wait`, which blocks
// until the previous grid has completed and its memory operations are
// visible: nothing is read or written before that, so the result is the same
// as with plain stream order whatever ran before (a kernel that never
// signals simply lets the next one launch when it completes).  A dependent
// grid is launched only after all blocks of the previous one have started, so
// waiting blocks never hold back a block they depend on.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace tr {

// First statement of every kernel launched through launch_pdl.
__device__ __forceinline__ void pdl_prologue() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename... KernelArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    // The error goes back through the return value; leave no stale per-thread
    // error behind for the next launch's cudaGetLastError().
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e;
}

}  // namespace tr
