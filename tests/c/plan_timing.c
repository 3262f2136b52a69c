/*
 * plan_timing.c -- host cost of a repeated tl_plan call (a plan-cache hit), timed
 * in C so that no binding overhead is counted.  Prints the best of five rounds in
 * nanoseconds per call (tests/test_host_abi.py compiles and runs it; no GPU).
 */
#define _POSIX_C_SOURCE 199309L
#include <stdint.h>
#include <stdio.h>
#include <time.h>

#include "tl_permute.h"

static double now_ns(void) {
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return (double)t.tv_sec * 1e9 + (double)t.tv_nsec;
}

int main(void) {
    /* the SF transpose of the permute_layout page, and a batched tile transpose */
    const int64_t sf_shape[4] = {2, 1, 4, 32}, sf_src[4] = {128, 128, 32, 1},
                  sf_dst[4] = {128, 128, 1, 4};
    const int64_t t_shape[3] = {65536, 128, 64}, t_src[3] = {8192, 64, 1},
                  t_dst[3] = {8192, 1, 128};
    const void *src = (const void *)(uintptr_t)0x100000000ull;
    const void *dst = (const void *)(uintptr_t)0x200000000ull;
    tl_plan_info info;
    double best = 1e30;
    if (tl_plan(src, (void *)dst, 4, sf_shape, sf_src, sf_dst, 4, NULL, &info) != TL_OK) return 1;
    if (tl_plan(src, (void *)dst, 3, t_shape, t_src, t_dst, 2, NULL, &info) != TL_OK) return 1;
    const uint64_t h0 = tl_plan_cache_hits();
    const int n = 100000;
    for (int round = 0; round < 5; ++round) {
        const double t0 = now_ns();
        for (int i = 0; i < n; ++i) {
            if (i & 1)
                tl_plan(src, (void *)dst, 4, sf_shape, sf_src, sf_dst, 4, NULL, &info);
            else
                tl_plan(src, (void *)dst, 3, t_shape, t_src, t_dst, 2, NULL, &info);
        }
        const double per = (now_ns() - t0) / n;
        if (per < best) best = per;
    }
    printf("hits %llu of %d calls\n", (unsigned long long)(tl_plan_cache_hits() - h0), 5 * n);
    printf("ns per call %.1f\n", best);
    return 0;
}
