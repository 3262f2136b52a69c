/*
 * abi_client.c -- a plain C99 client of libtl_permute.so: includes only
 * include/tl_permute.h, links only the library, and calls the host-side entry
 * points on the worked examples of the TVM pages.  Prints one line per check and
 * exits non-zero on the first failure (tests/test_host_abi.py compiles and runs it;
 * no GPU is needed).
 *
 *   - "permute_layout", "Algorithm" step 1 / "Demonstration program": the float32
 *     SF transpose (pipe=2, high=1, 4, 32), strides (128,128,32,1) -> (128,128,1,4),
 *     canonicalises to extent (2, 4, 32), src (128, 32, 1), dst (128, 1, 4).
 *   - "permute_layout", "Algorithm" step 2: the warp tile (4, 32) of that transpose
 *     picks k = 2, shift = 3, mask = 3.
 *   - "copy_async -> dsmem", "Algorithm" step 1: a 128x64 float16 tile copied to
 *     the same layout is one contiguous chunk of 8192 elements (16384 bytes).
 *   - tl_plan on the same SF transpose chooses the warp path.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "tl_permute.h"

static int failures = 0;

static void expect(int ok, const char *what) {
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok) ++failures;
}

static tl_layout layout(int n, const int64_t *shape, const int64_t *stride) {
    tl_layout l;
    memset(&l, 0, sizeof l);
    l.ndim = n;
    for (int i = 0; i < n; ++i) {
        l.shape[i] = shape[i];
        l.stride[i] = stride[i];
    }
    return l;
}

int main(void) {
    expect(tl_version() == 2, "tl_version is 2");
    expect(strcmp(tl_status_string(TL_OK), "ok") == 0, "tl_status_string(TL_OK)");

    /* the SF transpose of the permute_layout page */
    const int64_t sf_shape[4] = {2, 1, 4, 32};
    const int64_t sf_src[4] = {128, 128, 32, 1};
    const int64_t sf_dst[4] = {128, 128, 1, 4};
    tl_layout s = layout(4, sf_shape, sf_src), d = layout(4, sf_shape, sf_dst);
    tl_layout cs, cd;
    int64_t chunk = -1;
    int rc = tl_layout_canon(&s, &d, NULL, NULL, &cs, &cd, &chunk);
    expect(rc == TL_OK, "tl_layout_canon on the SF transpose");
    expect(cs.ndim == 3 && cs.shape[0] == 2 && cs.shape[1] == 4 && cs.shape[2] == 32,
           "canonical extent (2, 4, 32)");
    expect(cs.stride[0] == 128 && cs.stride[1] == 32 && cs.stride[2] == 1,
           "canonical src strides (128, 32, 1)");
    expect(cd.stride[0] == 128 && cd.stride[1] == 1 && cd.stride[2] == 4,
           "canonical dst strides (128, 1, 4)");
    expect(chunk == 0, "no common contiguous chunk");

    const int64_t wt_ext[2] = {4, 32}, wt_src[2] = {32, 1}, wt_dst[2] = {1, 4};
    int k = -1, shift = -1, mask = -1;
    rc = tl_choose_xor_k(2, wt_ext, wt_src, wt_dst, 4, &k, &shift, &mask);
    expect(rc == TL_OK && k == 2 && shift == 3 && mask == 3, "tl_choose_xor_k -> (2, 3, 3)");

    /* the 128x64 float16 tile of the copy_async -> dsmem page, same layout both sides */
    const int64_t t_shape[2] = {128, 64}, t_str[2] = {64, 1};
    s = layout(2, t_shape, t_str);
    rc = tl_layout_canon(&s, &s, NULL, NULL, &cs, &cd, &chunk);
    expect(rc == TL_OK && chunk == 8192 && chunk * 2 == 16384, "one chunk of 16384 bytes");

    /* a region that leaves the shape */
    const int64_t begin[2] = {100, 0}, extent[2] = {64, 64};
    rc = tl_layout_canon(&s, &s, begin, extent, &cs, &cd, &chunk);
    expect(rc == TL_ERR_RANGE, "region outside the shape -> TL_ERR_RANGE");

    /* the planner (pointers only for their alignment) */
    tl_plan_info info;
    rc = tl_plan((const void *)(uintptr_t)(1u << 20), (const void *)(uintptr_t)(1u << 24), 4,
                 sf_shape, sf_src, sf_dst, 4, NULL, &info);
    expect(rc == TL_OK && info.path == (int32_t)TL_PATH_WARP, "tl_plan chooses the warp path");
    expect(info.k == 2 && info.shift == 3 && info.mask == 3, "tl_plan reports the swizzle");

    /* a high-rank permute of short axes: 10^8 reversed, 4-byte elements; the short
       src-contiguous axis is merged with the next src axis (dense across the two) */
    {
        int64_t shp[8], ss8[8], ds8[8];
        for (int i = 0; i < 8; ++i) {
            int64_t st = 1;
            for (int j = i + 1; j < 8; ++j) st *= 10;
            shp[i] = 10;
            ss8[i] = st;                   /* row-major */
            int64_t dt = 1;
            for (int j = 0; j < i; ++j) dt *= 10;
            ds8[i] = dt;                   /* axes reversed */
        }
        rc = tl_plan((const void *)(uintptr_t)(1u << 20), (const void *)((uintptr_t)1 << 36), 8,
                     shp, ss8, ds8, 4, NULL, &info);
        expect(rc == TL_OK && info.path == (int32_t)TL_PATH_PANEL && info.panel_a1 == 10,
               "tl_plan merges the short a axis (panel_a1 = 10)");
    }

    /* validation launches nothing and needs no device */
    rc = tl_permute(NULL, NULL, 4, sf_shape, sf_src, sf_dst, 3, NULL);
    expect(rc == TL_ERR_ELEM_BYTES, "elem_bytes 3 -> TL_ERR_ELEM_BYTES");

    printf("%d failure(s)\n", failures);
    return failures ? 1 : 0;
}
