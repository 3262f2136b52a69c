/*
 * oracle/permute_ref.c -- plain CPU oracle for a strided layout permutation.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline / reference arm may load this library.  It
 * shares no code, header, table or helper with the CUDA library: it is the
 * definition written out so that a reader can check it by eye.
 *
 * What it computes (TVM docs, "Buffers and memory", section "Declaring
 * buffers"): a buffer is a pointer plus a layout, and the element at logical
 * coordinate c lives at  data + elem_offset + layout.apply(c), where apply is
 * the sum over axes of c[i] * stride[i].  A layout permutation is therefore:
 * for every coordinate c of `shape`,
 *
 *     dst[ sum_i c[i] * dst_strides[i] ] = src[ sum_i c[i] * src_strides[i] ]
 *
 * with elements moved as raw bytes (so NaN payloads survive).  The warp
 * permute on the TVM "permute_layout" page reads every element before it
 * writes any ("Algorithm", step 3), so for non-aliasing buffers the result is
 * exactly this definition; an aliased (in-place) call equals this definition
 * applied to a copy of the input.
 *
 * The coordinates are visited with a row-major odometer (last axis fastest),
 * 64-bit offsets throughout.  `nthreads` > 1 splits the flat coordinate range
 * into contiguous pieces that run the same loop on separate OpenMP threads;
 * nothing else about the loop changes.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_DIMS 8

/* Offset of one coordinate under a layout: sum of coordinate times stride. */
static int64_t apply_layout(int ndim, const int64_t *coord, const int64_t *stride)
{
    int64_t off = 0;
    for (int i = 0; i < ndim; ++i)
        off += coord[i] * stride[i];
    return off;
}

/* Copy the elements whose row-major flat index lies in [first, last). */
static void permute_range(const unsigned char *src, unsigned char *dst, int ndim,
                          const int64_t *shape, const int64_t *src_strides,
                          const int64_t *dst_strides, int elem_bytes,
                          int64_t first, int64_t last)
{
    int64_t coord[ORACLE_MAX_DIMS];
    int64_t rem = first;
    for (int i = ndim - 1; i >= 0; --i) {
        coord[i] = rem % shape[i];
        rem /= shape[i];
    }
    for (int64_t n = first; n < last; ++n) {
        int64_t s = apply_layout(ndim, coord, src_strides);
        int64_t d = apply_layout(ndim, coord, dst_strides);
        memcpy(dst + d * elem_bytes, src + s * elem_bytes, (size_t)elem_bytes);
        for (int i = ndim - 1; i >= 0; --i) {      /* odometer step */
            if (++coord[i] < shape[i])
                break;
            coord[i] = 0;
        }
    }
}

/* Number of OpenMP threads the compiled oracle can use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Permute `shape` from src to dst.  Strides are in elements; elem_bytes is
 * one of 1, 2, 4, 8, 16 (the byte widths the permute_layout page admits).
 * Returns 0, or -1 for arguments outside that contract.  The caller guarantees
 * that every offset stays inside its buffers.
 */
int oracle_permute(const void *src, void *dst, int ndim, const int64_t *shape,
                   const int64_t *src_strides, const int64_t *dst_strides,
                   int elem_bytes, int nthreads)
{
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8 &&
        elem_bytes != 16)
        return -1;
    if (ndim < 0 || ndim > ORACLE_MAX_DIMS)
        return -1;
    int64_t total = 1;
    for (int i = 0; i < ndim; ++i) {
        if (shape[i] < 0)
            return -1;
        total *= shape[i];
    }
    if (total == 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads == 1 || total < 4096) {
        permute_range((const unsigned char *)src, (unsigned char *)dst, ndim, shape,
                      src_strides, dst_strides, elem_bytes, 0, total);
        return 0;
    }
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(static, 1)
#endif
    for (int t = 0; t < nthreads; ++t) {
        int64_t first = total / nthreads * t + (t < total % nthreads ? t : total % nthreads);
        int64_t count = total / nthreads + (t < total % nthreads ? 1 : 0);
        permute_range((const unsigned char *)src, (unsigned char *)dst, ndim, shape,
                      src_strides, dst_strides, elem_bytes, first, first + count);
    }
    return 0;
}
