/* The C ABI driven from plain C on a GPU: device buffers from the CUDA
 * runtime, results compared byte for byte with the CPU oracle (liboracle),
 * output pitch padding included. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "transpose.h"

/* The oracle's entry points (oracle/oracle.c). */
void oracle_transpose_u32(const uint32_t *in, uint32_t *out, int64_t batch, int64_t rows,
                          int64_t cols, int64_t ld_in, int64_t ld_out, int64_t stride_in,
                          int64_t stride_out);
void oracle_transpose_u16(const uint16_t *in, uint16_t *out, int64_t batch, int64_t rows,
                          int64_t cols, int64_t ld_in, int64_t ld_out, int64_t stride_in,
                          int64_t stride_out);
void oracle_transpose_inplace_u32(uint32_t *data, int64_t batch, int64_t n, int64_t ld,
                                  int64_t stride);
void oracle_copy_bytes(const uint8_t *in, uint8_t *out, int64_t bytes);

static int failures = 0;

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t next_u32(void) { /* xorshift64* */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (uint32_t)((rng_state * 2685821657736338717ull) >> 32);
}

static void fill(void *p, size_t bytes) {
    uint8_t *b = (uint8_t *)p;
    for (size_t i = 0; i < bytes; ++i) b[i] = (uint8_t)next_u32();
}

static void check_cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        printf("FAIL: %s: %s\n", what, cudaGetErrorString(e));
        exit(2);
    }
}

/* Device copy of a host buffer. */
static void *to_device(const void *h, size_t bytes) {
    void *d = NULL;
    check_cuda(cudaMalloc(&d, bytes ? bytes : 1), "cudaMalloc");
    check_cuda(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice), "upload");
    return d;
}

static void compare(const void *d, const void *want, size_t bytes, const char *what) {
    void *got = malloc(bytes ? bytes : 1);
    check_cuda(cudaMemcpy(got, d, bytes, cudaMemcpyDeviceToHost), "download");
    if (memcmp(got, want, bytes) != 0) {
        printf("FAIL: %s differs from the oracle\n", what);
        ++failures;
    }
    free(got);
}

/* fp32 or bf16 (esize 4 or 2), optionally batched, through the plain entry points. */
static void case_transpose(int esize, int64_t batch, int64_t rows, int64_t cols, int64_t ld_in,
                           int64_t ld_out, int64_t stride_in, int64_t stride_out,
                           cudaStream_t stream, const char *what) {
    const int64_t sin = batch > 1 ? stride_in : rows * ld_in;
    const int64_t sout = batch > 1 ? stride_out : cols * ld_out;
    const size_t in_bytes = (size_t)(batch * sin) * esize, out_bytes = (size_t)(batch * sout) * esize;
    void *h_in = malloc(in_bytes), *want = malloc(out_bytes);
    fill(h_in, in_bytes);
    fill(want, out_bytes); /* prefill: padding must keep it */
    void *d_in = to_device(h_in, in_bytes), *d_out = to_device(want, out_bytes);
    tr_status st;
    if (esize == 4) {
        oracle_transpose_u32((const uint32_t *)h_in, (uint32_t *)want, batch, rows, cols, ld_in,
                             ld_out, sin, sout);
        st = batch > 1 ? tr_transpose_batched_f32((const float *)d_in, (float *)d_out, batch, rows,
                                                  cols, ld_in, ld_out, sin, sout, stream)
                       : tr_transpose_f32((const float *)d_in, (float *)d_out, rows, cols, ld_in,
                                          ld_out, stream);
    } else {
        oracle_transpose_u16((const uint16_t *)h_in, (uint16_t *)want, batch, rows, cols, ld_in,
                             ld_out, sin, sout);
        st = batch > 1 ? tr_transpose_batched_bf16(d_in, d_out, batch, rows, cols, ld_in, ld_out,
                                                   sin, sout, stream)
                       : tr_transpose_bf16(d_in, d_out, rows, cols, ld_in, ld_out, stream);
    }
    if (st != TR_OK) {
        printf("FAIL: %s: %s (%s)\n", what, tr_status_string(st), tr_last_error());
        ++failures;
    }
    check_cuda(cudaStreamSynchronize(stream), "sync");
    compare(d_out, want, out_bytes, what);
    cudaFree(d_in);
    cudaFree(d_out);
    free(h_in);
    free(want);
}

int main(void) {
    cudaStream_t stream;
    check_cuda(cudaStreamCreate(&stream), "cudaStreamCreate");

    case_transpose(4, 1, 2048, 2048, 2048, 2048, 0, 0, stream, "fp32 2048x2048");
    case_transpose(4, 1, 1000, 777, 800, 1003, 0, 0, stream, "fp32 1000x777, output pitch 1003");
    case_transpose(4, 1, 999, 1201, 1203, 1000, 0, 0, NULL, "fp32 999x1201, input pitch 1203");
    case_transpose(2, 3, 513, 1030, 1040, 520, 513 * 1040 + 16, 1030 * 520 + 8, stream,
                   "bf16 3x513x1030 with plane gaps");
    case_transpose(2, 1, 640, 384, 385, 641, 0, 0, stream, "bf16 640x384, odd pitches");

    { /* in place, square, with row pitch padding */
        const int64_t n = 1000, ld = 1008;
        const size_t bytes = (size_t)(n * ld) * 4;
        uint32_t *h = (uint32_t *)malloc(bytes);
        fill(h, bytes);
        void *d = to_device(h, bytes);
        oracle_transpose_inplace_u32(h, 1, n, ld, n * ld);
        tr_status st = tr_transpose_inplace_f32((float *)d, 1, n, ld, n * ld, stream);
        if (st != TR_OK) {
            printf("FAIL: in place: %s\n", tr_status_string(st));
            ++failures;
        }
        check_cuda(cudaStreamSynchronize(stream), "sync");
        compare(d, h, bytes, "fp32 in place 1000 (pitch 1008)");
        cudaFree(d);
        free(h);
    }
    { /* copy with an odd length between differently aligned addresses */
        const size_t bytes = 1000003;
        uint8_t *h = (uint8_t *)malloc(bytes + 16), *want = (uint8_t *)malloc(bytes + 16);
        fill(h, bytes + 16);
        fill(want, bytes + 16);
        uint8_t *d_in = (uint8_t *)to_device(h, bytes + 16);
        uint8_t *d_out = (uint8_t *)to_device(want, bytes + 16);
        oracle_copy_bytes(h + 3, want + 5, (int64_t)bytes);
        tr_status st = tr_copy(d_in + 3, d_out + 5, bytes, stream);
        if (st != TR_OK) {
            printf("FAIL: copy: %s\n", tr_status_string(st));
            ++failures;
        }
        check_cuda(cudaStreamSynchronize(stream), "sync");
        compare(d_out, want, bytes + 16, "copy of 1000003 bytes, offsets 3 -> 5");
        cudaFree(d_in);
        cudaFree(d_out);
        free(h);
        free(want);
    }
    if (tr_device_status() != TR_OK) {
        printf("FAIL: a bounded in-kernel wait ran out\n");
        ++failures;
    }
    cudaStreamDestroy(stream);
    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
