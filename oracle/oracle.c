/*
 * Oracle for the out-of-place matrix transpose -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously correct CPU statement of what the
 * GPU library computes.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it; the product path never does.
 * It shares no code, header, constant or helper with the CUDA library.
 *
 * What it follows:
 *   - "Shared memory and the bank conflict" (roobli.org, kernels-from-zero 03),
 *     section "Turn the tile around on chip": the element read from input row
 *     y, column x is written to output row x, column y.  The tile there is only
 *     a staging device; the result it produces is the plain transpose.
 *   - "Shared-memory tiling and bank conflicts" (intro-to-ai-systems-performance,
 *     shared-memory chapter), "Worked example": global coordinates stay logical,
 *     padding exists only in on-chip storage, and the logical contents are
 *     unchanged by the staging.
 *
 * Definition, for b < batch, i < rows, j < cols (all sizes in elements):
 *
 *     out[b*stride_out + j*ld_out + i] = in[b*stride_in + i*ld_in + j]
 *
 * Elements are moved as raw bit patterns (uint32_t for fp32, uint16_t for
 * bf16): no floating-point load or store ever touches them, so NaN payloads,
 * signed zeros and subnormals pass through unchanged.  Nothing outside the
 * logical output region is written.
 *
 * Two loop orders are given.  The gather form visits the output in memory
 * order and is the definition above written out.  The scatter form visits the
 * input in memory order.  They must agree on every input; the tests use the
 * pair as one cross-check among several (closed forms, numpy's own transpose,
 * involution, permutation and sentinel invariants).
 *
 * Parity status: pinned (see the oracle tests).
 */
#include <stdint.h>
#include <stddef.h>

/* ---- gather form: loop over output elements in memory order ---------- */

void oracle_transpose_u32(const uint32_t *in, uint32_t *out,
                          int64_t batch, int64_t rows, int64_t cols,
                          int64_t ld_in, int64_t ld_out,
                          int64_t stride_in, int64_t stride_out)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t j = 0; j < cols; ++j)          /* output row    */
            for (int64_t i = 0; i < rows; ++i)      /* output column */
                out[b * stride_out + j * ld_out + i] =
                    in[b * stride_in + i * ld_in + j];
}

void oracle_transpose_u16(const uint16_t *in, uint16_t *out,
                          int64_t batch, int64_t rows, int64_t cols,
                          int64_t ld_in, int64_t ld_out,
                          int64_t stride_in, int64_t stride_out)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t j = 0; j < cols; ++j)
            for (int64_t i = 0; i < rows; ++i)
                out[b * stride_out + j * ld_out + i] =
                    in[b * stride_in + i * ld_in + j];
}

/* ---- scatter form: loop over input elements in memory order ---------- */

void oracle_transpose_scatter_u32(const uint32_t *in, uint32_t *out,
                                  int64_t batch, int64_t rows, int64_t cols,
                                  int64_t ld_in, int64_t ld_out,
                                  int64_t stride_in, int64_t stride_out)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < rows; ++i)          /* input row    */
            for (int64_t j = 0; j < cols; ++j)      /* input column */
                out[b * stride_out + j * ld_out + i] =
                    in[b * stride_in + i * ld_in + j];
}

void oracle_transpose_scatter_u16(const uint16_t *in, uint16_t *out,
                                  int64_t batch, int64_t rows, int64_t cols,
                                  int64_t ld_in, int64_t ld_out,
                                  int64_t stride_in, int64_t stride_out)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < rows; ++i)
            for (int64_t j = 0; j < cols; ++j)
                out[b * stride_out + j * ld_out + i] =
                    in[b * stride_in + i * ld_in + j];
}

/* ---- the copy the transpose is measured against ----------------------
 * "Shared memory and the bank conflict", section "What to record": the
 * transpose timings sit next to a plain copy of the same bytes.  Its result is
 * out[k] = in[k] for every byte k < bytes.                                  */

void oracle_copy_bytes(const uint8_t *in, uint8_t *out, int64_t bytes)
{
    for (int64_t k = 0; k < bytes; ++k)
        out[k] = in[k];
}

/* ---- in-place transpose of square planes -------------------------------
 * The same result written over the input: plane b of an n x n matrix with
 * row pitch ld becomes its transpose, element (i, j) exchanging places with
 * element (j, i) for every i < j; diagonal and padding elements stay put.   */

void oracle_transpose_inplace_u32(uint32_t *data, int64_t batch, int64_t n, int64_t ld,
                                  int64_t stride)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = i + 1; j < n; ++j) {
                uint32_t *p = data + b * stride + i * ld + j;
                uint32_t *q = data + b * stride + j * ld + i;
                uint32_t tmp = *p;
                *p = *q;
                *q = tmp;
            }
}

void oracle_transpose_inplace_u16(uint16_t *data, int64_t batch, int64_t n, int64_t ld,
                                  int64_t stride)
{
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = i + 1; j < n; ++j) {
                uint16_t *p = data + b * stride + i * ld + j;
                uint16_t *q = data + b * stride + j * ld + i;
                uint16_t tmp = *p;
                *p = *q;
                *q = tmp;
            }
}

/* ---- transposed operand tiles ------------------------------------------
 * "Padded Shared Memory: Eliminating Bank Conflicts", sections "How Shared
 * Memory Is Addressed" and "The Fix Is One Constant": the SGEMM kernel loads
 * a BM x BK tile of A (rows m, columns k of a row-major M x K matrix with row
 * pitch lda) and stores it transposed in shared memory, As[k][m] = A[m][k]
 * (the padding of the As row pitch changes only where the words sit, never
 * their values).  The stage on its own writes every tile's As, unpadded, to
 * a blocked output: tile (mt, kt) at ((mt * K/BK) + kt) * BK*BM, element
 * (k, m) at k*BM + m.  M and K are multiples of BM and BK.                 */

void oracle_operand_tiles_u32(const uint32_t *a, uint32_t *out, int64_t m_rows, int64_t k_cols,
                              int64_t lda, int64_t bm, int64_t bk)
{
    const int64_t tiles_k = k_cols / bk;
    for (int64_t mt = 0; mt < m_rows / bm; ++mt)
        for (int64_t kt = 0; kt < tiles_k; ++kt) {
            uint32_t *as = out + (mt * tiles_k + kt) * bk * bm;
            for (int64_t k = 0; k < bk; ++k)
                for (int64_t m = 0; m < bm; ++m)
                    as[k * bm + m] = a[(mt * bm + m) * lda + kt * bk + k];
        }
}
