/* Host-only use of the C ABI from plain C: the header compiles as C99, the
 * library links, and argument errors come back before any CUDA call. */
#include <stdio.h>
#include <string.h>

#include "transpose.h"

static int failures = 0;

static void expect(int cond, const char *what) {
    if (!cond) {
        printf("FAIL: %s\n", what);
        ++failures;
    }
}

int main(void) {
    /* Addresses that are never dereferenced: every call below is refused (or
     * planned) on the host. */
    float *in = (float *)(size_t)0x10000, *out = (float *)(size_t)0x80000000;
    tr_args a;
    tr_options o;

    expect(tr_version() > 0, "tr_version");
    expect(strlen(tr_status_string(TR_ERR_BAD_DIM)) > 0, "tr_status_string");
    expect(tr_transpose_f32(in, out, -1, 4, 4, 4, NULL) == TR_ERR_BAD_DIM, "negative rows");
    expect(tr_transpose_f32(in, out, 4, 4, 3, 4, NULL) == TR_ERR_BAD_LD, "ld_in < cols");
    expect(tr_transpose_f32(NULL, out, 4, 4, 4, 4, NULL) == TR_ERR_NULL, "NULL input");
    expect(tr_transpose_f32(in, in + 1, 4, 4, 4, 4, NULL) == TR_ERR_OVERLAP, "overlap");
    expect(tr_transpose_f32(in, out, 0, 4, 4, 4, NULL) == TR_OK, "empty problem");
    expect(tr_transpose_batched_bf16(in, out, 2, 4, 4, 4, 4, 15, 16, NULL) == TR_ERR_BAD_LD,
           "overlapping planes");

    memset(&a, 0, sizeof a);
    memset(&o, 0, sizeof o);
    a.in = in;
    a.out = out;
    a.dtype = TR_DTYPE_F32;
    a.batch = 1;
    a.rows = 8192;
    a.cols = 8192;
    a.ld_in = 8192;
    a.ld_out = 8192;
    expect(tr_plan_variant(&a, NULL) == TR_VARIANT_TILE_VEC, "AUTO plans the vector tile");
    {
        tr_plan plan;
        expect(tr_plan_ex(&a, NULL, &plan) == TR_OK && plan.variant == TR_VARIANT_TILE_VEC &&
                   plan.tile_rows == 64 && plan.tile_cols == 64 && plan.threads == 256 &&
                   plan.vec_in == 1 && plan.vec_out == 1,
               "AUTO's tile for the aligned 8192 x 8192 fp32 case");
        a.ld_out = 8193;
        expect(tr_plan_ex(&a, NULL, &plan) == TR_OK && plan.tile_rows == 128 &&
                   plan.tile_cols == 64 && plan.vec_out == 0,
               "AUTO's tile for an odd output pitch");
        a.ld_out = 8192;
        expect(tr_plan_ex(&a, NULL, NULL) == TR_ERR_NULL, "NULL plan");
    }
    o.variant = TR_VARIANT_TMA;
    expect(tr_plan_variant(&a, &o) == TR_VARIANT_TMA, "explicit TMA honoured");
    o.stages = 1;
    expect(tr_plan_variant(&a, &o) == -TR_ERR_UNSUPPORTED, "bad stage count refused");
    o.stages = 0;
    o.variant = TR_VARIANT_TILE_VEC;
    o.schedule = 4;
    expect(tr_transpose_ex(&a, &o) == TR_ERR_UNSUPPORTED, "TMA schedule on the LSU tile");
    expect(strlen(tr_last_error()) > 0, "tr_last_error describes it");

    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
