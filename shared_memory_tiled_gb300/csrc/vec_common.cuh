// Pieces shared by the kernels that move 16-byte chunks through an
// XOR-swizzled shared tile: the chunk type, the register micro-transposes and
// element access inside a chunk.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tr {

// V = elements per 16-byte chunk.
template <typename T>
struct VecTraits;
template <>
struct VecTraits<uint32_t> {
    static constexpr int V = 4;
};
template <>
struct VecTraits<uint16_t> {
    static constexpr int V = 8;
};

union Chunk {
    uint4 v;
    uint32_t w[4];
};

__device__ __forceinline__ void micro_transpose(const Chunk (&x)[4], Chunk (&y)[4]) {
#pragma unroll
    for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int k = 0; k < 4; ++k) y[m].w[k] = x[k].w[m];
}

// 8x8 of 16-bit elements: output row m takes half (m & 1) of word (m >> 1)
// from every input row; output word w pairs input rows 2w (low) and 2w+1 (high).
__device__ __forceinline__ void micro_transpose(const Chunk (&x)[8], Chunk (&y)[8]) {
#pragma unroll
    for (int m = 0; m < 8; ++m)
#pragma unroll
        for (int w = 0; w < 4; ++w)
            y[m].w[w] = __byte_perm(x[2 * w].w[m >> 1], x[2 * w + 1].w[m >> 1],
                                    (m & 1) ? 0x7632 : 0x5410);
}

template <typename T>
__device__ __forceinline__ T elem(const Chunk &c, int q) {
    if (sizeof(T) == 4) return T(c.w[q]);
    return T(c.w[q >> 1] >> ((q & 1) * 16));
}


}  // namespace tr
