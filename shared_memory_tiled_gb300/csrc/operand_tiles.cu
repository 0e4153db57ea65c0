// Transposed operand tiles: the shared-memory load stage of the padded SGEMM
// ("Padded Shared Memory: Eliminating Bank Conflicts") run on its own.
//
// A block of 128 threads stages one BM x BK tile of the row-major M x K
// matrix A transposed, As[k][m] = A[m][k], as the page's kernel does: thread t
// loads one 16-byte float4 of A (row t / (BK/4), columns 4*(t % (BK/4)) ..
// +3) per pass of 512/BK rows, and writes its four words down four rows of
// As ("How Shared Memory Is Addressed").  As has a row pitch of
// A_STRIDE = BM + pad words.  With pad = 0 the pitch is a multiple of 32, so a
// store's bank depends only on the tile row its lane carries: a warp's 32
// lanes carry 32/(BK/4) rows, BK/4 lanes each, a (BK/4)-way conflict (4-way
// at BK = 16, 2-way at BK = 8).  With the page's pad = (32 / BK) % 8 the
// column term comes back into the bank and the 32 lanes land on 32 distinct
// banks ("The Fix Is One Constant").  After the barrier the block writes As
// without its padding to the blocked output, tile (mt, kt) at
// ((mt * K/BK) + kt) * BK*BM, element (k, m) at k*BM + m, with consecutive
// threads on consecutive words.
//
// The output exists so the stage has a checkable result and so its shared
// stores can be measured (bank-conflict counters) apart from any arithmetic.
#include "bounds.cuh"
#include "tile_geom.cuh"
#include "tr_internal.h"

namespace tr {
namespace {

constexpr int kThreads = 128;

template <int BM, int BK>
__global__ void __launch_bounds__(kThreads)
k_operand_tiles(const uint32_t *__restrict__ a, uint32_t *__restrict__ out, int64_t m_tiles,
                int64_t k_tiles, int64_t lda, int a_stride) {
    extern __shared__ uint32_t as[];  // BK rows of a_stride words
    constexpr int COLS4 = BK / 4;                 // float4s per tile row
    constexpr int ROW_STRIDE = kThreads * 4 / BK; // tile rows per load pass
    static_assert(BM % ROW_STRIDE == 0, "tile rows must be a multiple of the pass height");
    const int t = threadIdx.x;
    const int inner_row = t / COLS4, inner_col = t % COLS4;
    const int64_t total = m_tiles * k_tiles;
    // Debug builds: A is M x K at pitch lda; the output holds M*K words.
    TR_SIDE(in_side, a, 1, m_tiles * BM, k_tiles * BK, lda, 0, 4);
    TR_SIDE(out_side, out, 1, 1, total * BM * BK, total * BM * BK, 0, 4);
    for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int64_t mt = tile / k_tiles, kt = tile - mt * k_tiles;
        const uint32_t *src = a + (mt * BM) * lda + kt * BK + inner_col * 4;
        if (tile != blockIdx.x) __syncthreads();  // previous tile written out
#pragma unroll
        for (int off = 0; off < BM; off += ROW_STRIDE) {
            const uint32_t *p = src + (inner_row + off) * lda;
            const uint4 v = TR_LOAD_OK(in_side, p, 16) ? *reinterpret_cast<const uint4 *>(p)
                                                       : make_uint4(0u, 0u, 0u, 0u);
            uint32_t *col = as + (inner_col * 4) * a_stride + inner_row + off;
            col[0] = v.x;
            col[a_stride] = v.y;
            col[2 * a_stride] = v.z;
            col[3 * a_stride] = v.w;
        }
        __syncthreads();
        uint32_t *dst = out + tile * (BM * BK);
#pragma unroll 4
        for (int w = t; w < BM * BK; w += kThreads)
            if (TR_STORE_OK(out_side, dst + w, 4)) dst[w] = as[(w / BM) * a_stride + (w % BM)];
    }
}

template <int BM, int BK>
cudaError_t launch_shape(const uint32_t *a, uint32_t *out, int64_t m, int64_t k, int64_t lda,
                         int pad, cudaStream_t stream) {
    const int a_stride = BM + pad;
    const size_t smem = size_t(BK) * a_stride * 4;
    const int64_t m_tiles = m / BM, k_tiles = k / BK;
    k_operand_tiles<BM, BK><<<grid_blocks(m_tiles * k_tiles), kThreads, smem, stream>>>(
        a, out, m_tiles, k_tiles, lda, a_stride);
    return cudaGetLastError();
}

}  // namespace

// Debug builds: this unit's record of refused accesses.
TR_BOUNDS_READER(read_bounds_operand_tiles)

cudaError_t launch_operand_tiles(const uint32_t *a, uint32_t *out, int64_t m, int64_t k,
                                 int64_t lda, int bm, int bk, int pad, cudaStream_t stream) {
#define TR_OPERAND_CASE(BM_, BK_) \
    if (bm == BM_ && bk == BK_) return launch_shape<BM_, BK_>(a, out, m, k, lda, pad, stream);
    TR_OPERAND_CASE(128, 8)
    TR_OPERAND_CASE(128, 16)
    TR_OPERAND_CASE(128, 32)
    TR_OPERAND_CASE(64, 8)
    TR_OPERAND_CASE(64, 16)
    TR_OPERAND_CASE(64, 32)
#undef TR_OPERAND_CASE
    return cudaErrorInvalidValue;
}

}  // namespace tr
