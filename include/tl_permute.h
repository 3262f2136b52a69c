/*
 * tl_permute.h -- C ABI of the GB300 (sm_103a) tensor layout-permute library.
 *
 * A layout is a shape with per-axis element strides; the element at logical
 * coordinate c of a buffer lives at  data + offset + sum_i c[i] * stride[i]
 * (TVM docs, "Buffers and memory", section "Declaring buffers": a buffer is a
 * pointer plus a layout, and indexing resolves to that address arithmetic).
 * Permuting a layout means materialising, for every coordinate c of the shape,
 *
 *     dst[sum_i c[i] * dst_strides[i]] = src[sum_i c[i] * src_strides[i]]
 *
 * with elements of 1, 2, 4, 8 or 16 bytes moved as raw bits (NaN payloads and
 * signed zeros survive).  This covers warp-sized transposes such as the 4x32
 * scale-factor transpose of the TVM "permute_layout" page, batched whole-tile
 * transposes, and general N-D axis permutes.
 *
 * Conventions for every entry point
 *   - Strides, offsets and extents are counted in ELEMENTS, never bytes.
 *   - Pointers passed as src/dst are DEVICE pointers (cudaMalloc / PyTorch CUDA
 *     storage) unless stated otherwise; the caller owns every buffer.  The
 *     library allocates no device memory and keeps no per-call state; it caches
 *     device properties and a driver entry point on first use.
 *   - Return value: TL_OK (0) or a negative tl_status.  Argument errors are
 *     reported synchronously and launch nothing.  tl_permute* is asynchronous
 *     and stream-ordered: a kernel fault surfaces later through the CUDA runtime.
 *   - Thread safety: all entry points may be called from several host threads.
 */
#ifndef TL_PERMUTE_H
#define TL_PERMUTE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TL_MAX_DIMS 8
#define TL_VERSION 2

#if defined(__GNUC__)
#define TL_API __attribute__((visibility("default")))
#else
#define TL_API
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *tl_stream_t;

/* Status codes.  The first group mirrors the reasons the TVM permute_layout
 * dispatch gives for declining ("permute_layout", section "What it accepts"). */
typedef enum tl_status {
    TL_OK = 0,
    TL_ERR_ARG = -1,          /* NULL pointer, rank outside 0..8, negative extent or stride */
    TL_ERR_ELEM_BYTES = -2,   /* element width not one of 1, 2, 4, 8, 16 */
    TL_ERR_EXTENT = -3,       /* extents not a whole number of warp iterations (32 x P) */
    TL_ERR_NO_VALID_K = -4,   /* no XOR swizzle leaves both phases bank-conflict-free */
    TL_ERR_CHUNK = -5,        /* reserved: contiguous chunk under 16 B / not a multiple of 16 */
    TL_ERR_DST_OVERLAP = -6,  /* two coordinates may land on one dst element */
    TL_ERR_ALIAS = -7,        /* src and dst byte ranges intersect (outside the in-place case) */
    TL_ERR_ALIGN = -8,        /* src or dst not aligned to its element width */
    TL_ERR_PATH = -9,         /* the path forced through tl_permute_opts.flags does not apply */
    TL_ERR_RANGE = -10,       /* an offset overflows 64 bits, or a region leaves its layout */
    TL_ERR_CUDA = -11,        /* a CUDA runtime / driver call failed */
    TL_ERR_TIMEOUT = -12,     /* device side: a bounded wait expired (written to dev_status) */
    TL_ERR_BOUNDS = -13       /* a layout reaches outside the buffer size given in opts */
} tl_status;

/* A layout over `ndim` axes: element offset = offset + sum shape-coordinate * stride. */
typedef struct tl_layout {
    int32_t ndim;
    int32_t reserved;
    int64_t shape[TL_MAX_DIMS];
    int64_t stride[TL_MAX_DIMS];
    int64_t offset;
} tl_layout;

/*
 * tl_layout_canon -- slice a pair of layouts to a region, canonicalise them and
 * regroup src to dst's shape (TVM "permute_layout", "Algorithm" step 1; the
 * contiguous-chunk walk of "copy_async -> dsmem", "Algorithm" step 1).
 *
 *   src, dst     layouts of equal ndim and shape (host structs, read only)
 *   begin,extent region box per axis (host arrays of ndim); begin NULL = all
 *                zeros, extent NULL = shape - begin
 *   src_out,
 *   dst_out      receive the canonical pair: one shared shape (extent-1 axes
 *                dropped; adjacent axes merged, order kept, where BOTH sides are
 *                contiguous across them), per-side strides, and offsets moved to
 *                the region's first element
 *   chunk_elems  (nullable) length of the common stride-1 chain at the
 *                innermost end: the last extent when both last strides are 1,
 *                else 0; 1 for a single-element region, 0 for an empty one.
 *                A bulk copy needs chunk_elems * elem_bytes >= 16 and % 16 == 0.
 * Returns TL_OK, TL_ERR_ARG (NULL, ndim mismatch, negative extent) or
 * TL_ERR_RANGE (region outside the shape).
 */
TL_API int tl_layout_canon(const tl_layout *src, const tl_layout *dst, const int64_t *begin,
                    const int64_t *extent, tl_layout *src_out, tl_layout *dst_out,
                    int64_t *chunk_elems);

/*
 * tl_choose_xor_k -- host-side shared-memory bank simulator of the warp
 * register-staged permute (TVM "permute_layout", "Algorithm" steps 2 and 3).
 *
 * Each of the 32 lanes stages P = prod(extent)/32 elements; in iteration r a
 * lane handles iteration index j = r ^ ((lane >> shift) & mask), at coordinates
 * decompose(lane + 32*j, extent) (row-major).  The simulator checks, for every r,
 * the read phase (src_str) and the write phase (dst_str) against 32 banks of
 * 4 bytes, wavefronts of 128 bytes (32 lanes for widths <= 4, 16 for 8-byte, 8
 * for 16-byte), counting lanes that touch one bank -- even within one word -- as
 * a conflict.  It returns the first conflict-free candidate in the order
 * k = 0..log2(P) (k = 0 only if P is not a power of two), shift = 0..5-k.
 *
 *   ndim, extent, src_str, dst_str  host arrays, ndim 1..8, element units
 *   elem_bytes                      1, 2, 4, 8 or 16
 *   k, shift, mask                  outputs (mask = 2^k - 1); untouched on error
 * Returns TL_OK, TL_ERR_ARG, TL_ERR_ELEM_BYTES, TL_ERR_EXTENT (prod(extent) is
 * 0 or not a multiple of 32, or P > 1024) or TL_ERR_NO_VALID_K.
 */
TL_API int tl_choose_xor_k(int ndim, const int64_t *extent, const int64_t *src_str,
                    const int64_t *dst_str, int elem_bytes, int *k, int *shift, int *mask);

/*
 * tl_bank_conflicts -- the simulator's worst bank-conflict degree for one
 * warp-wide shared-memory access: lane_offsets[l] is the element offset lane l
 * touches (n_lanes <= 32, negative = idle lane).  model 0 = the conservative
 * rule above; model 1 = hardware rule (lanes reading one word share it).
 * Returns the degree (1 = conflict-free, 0 = no active lane) or a tl_status < 0.
 */
TL_API int tl_bank_conflicts(int n_lanes, const int64_t *lane_offsets, int elem_bytes, int model);

/*
 * tl_permute -- materialise the permutation on the GPU (the hot path): for every
 * coordinate c of shape, the element at src + sum(c_i * src_strides_i) is copied to
 * dst + sum(c_i * dst_strides_i) (TVM "Buffers and memory", section "Declaring
 * buffers": an element's address is the data pointer plus the element offset plus
 * the layout's offset of its coordinate; `B.permute` of "Buffer APIs" is this copy
 * with dst strides of the permuted row-major layout), as raw bits of one of the
 * widths "permute_layout" admits ("What it accepts").
 *
 *   src          device pointer to the source's element at coordinate 0
 *   dst          device pointer to the destination's element at coordinate 0
 *   ndim         0..8 (0 = one element)
 *   shape        host array of ndim extents (0 allowed: the call is a no-op)
 *   src_strides,
 *   dst_strides  host arrays of ndim element strides, each >= 0
 *   elem_bytes   1, 2, 4, 8 or 16; src and dst must be aligned to
 *                min(elem_bytes, 16) bytes
 *   stream       stream to launch on
 * dst must be non-overlapping (no two coordinates on one element; the check is
 * the sorted-stride sufficient test).  src may overlap itself.  src and dst byte
 * ranges must be disjoint, except for the in-place case of the warp path
 * (identical pointers and per-tile footprints), where every tile is read in
 * full before it is written.  Kernels are chosen by the planner (generic
 * strided, contiguous-chunk copy, TMA-staged tile transpose, cp.async-staged panel
 * transpose for planes TMA cannot describe, small-row register transpose, warp
 * XOR-swizzle transpose).
 */
TL_API int tl_permute(const void *src, void *dst, int ndim, const int64_t *shape,
               const int64_t *src_strides, const int64_t *dst_strides, int elem_bytes,
               tl_stream_t stream);

/* Kernel paths (low 4 bits of tl_permute_opts.flags). */
#define TL_PATH_AUTO 0u     /* planner's choice */
#define TL_PATH_GENERIC 1u  /* any layout: one element per step, coordinates decoded */
#define TL_PATH_CHUNK 2u    /* common contiguous innermost chain, widest aligned vector */
#define TL_PATH_TILE 3u     /* 2-D/batched transpose: TMA tile into 128B-swizzled smem */
#define TL_PATH_WARP 4u     /* warp register-staged XOR-swizzle transpose (in-place safe) */
#define TL_PATH_ROWS 5u     /* short dst runs (<= 16 B): 16 B row loads, register transpose */
#define TL_PATH_CLUSTER 6u  /* TILE with a 2-CTA cluster handing tiles over through DSMEM */
#define TL_PATH_PANEL 7u    /* plane transpose staged in smem by cp.async of the 16-byte
                               blocks covering each src row: any element alignment, up
                               to 6 batch axes, tiny extents */
#define TL_PATH_COLS 8u     /* short src runs (interleaved channels -> planes, pixels of
                               2..16 elements, <= 24 bytes): 16-byte pixel loads, register
                               transpose, one 16-byte store per plane */
#define TL_PATH_BLOCK 9u    /* a tile of up to four axes that is a few long contiguous runs
                               on both sides (high-rank permutes of short axes): each src
                               run one bulk copy into smem, stores along the dst runs */
#define TL_PATH_MASK 0xFu
/* Test hook for the cluster path (the producer CTA skips its DSMEM hand-off), for
 * panel tiles loaded by TMA phase maps (the loading thread skips one phase load of its
 * first tile) and for the block path (the producer warp skips the first src-run copy
 * of its first tile): the bounded wait (50 ms under the hook) must expire and report
 * TL_ERR_TIMEOUT in dev_status; the kernel returns without a fault. */
#define TL_FLAG_TEST_DROP_HANDOFF (1u << 8)
/* Launch without programmatic dependent launch (by default a permute may be scheduled
 * while the previous kernel of the stream drains; it waits for that kernel to complete
 * before touching global memory, so stream order is unchanged either way). */
#define TL_FLAG_NO_PDL (1u << 9)
/* Checked run (a sanitizer stand-in): the generic kernel moves every element after
 * checking its src and dst byte ranges against opts.src_bytes / opts.dst_bytes (a
 * side given as 0 is not checked); an element outside is skipped and
 * TL_ERR_BOUNDS written to dev_status.  Forces the generic path (another forced path
 * returns TL_ERR_PATH).  The host-side layout check still runs first. */
#define TL_FLAG_DEBUG_CHECKS (1u << 10)
/* Test hook, only with TL_FLAG_DEBUG_CHECKS (else TL_ERR_ARG): skip the host-side
 * TL_ERR_BOUNDS check so that a test can show the device-side one. */
#define TL_FLAG_TEST_SKIP_HOST_BOUNDS (1u << 11)
/* Panel path: store the tile element by element even where its dst rows would take
 * 16-byte runs (tuning and comparison; the result is the same). */
#define TL_FLAG_PANEL_ELEMENT_STORES (1u << 12)

/* Fused permute + cast (tl_permute_opts.cast): a widening of the equal-dtype rule of
 * "permute_layout" ("What it accepts"), each element converted as IEEE 754 does,
 * rounding to nearest with ties to even; a NaN keeps its sign and upper payload bits
 * when narrowed (the lowest payload bit set if those are all zero) and its payload
 * when widened. */
#define TL_CAST_NONE 0
#define TL_CAST_F32_TO_BF16 1   /* float32 -> bfloat16 */
#define TL_CAST_F32_TO_F16 2    /* float32 -> float16 */
#define TL_CAST_BF16_TO_F32 3   /* bfloat16 -> float32 (exact) */
#define TL_CAST_F16_TO_F32 4    /* float16 -> float32 (exact) */

/* Options of tl_permute_ex.  Zero-initialise, then set what you need. */
typedef struct tl_permute_opts {
    uint32_t flags;       /* TL_PATH_* | TL_FLAG_* */
    int32_t max_ctas;     /* > 0: cap on the persistent grid (tuning); 0 = planner */
    int32_t *dev_status;  /* nullable DEVICE int32: a kernel whose bounded wait expires
                             writes TL_ERR_TIMEOUT here (it is never cleared by the
                             library; the caller zeroes it).  NULL = not reported. */
    int64_t src_bytes;    /* > 0: bytes addressable from src; the layout must fit */
    int64_t dst_bytes;    /* > 0: bytes addressable from dst */
    /* Tuning of the tile, cluster and panel paths; 0 selects the planner's default
     * for each, as do values outside the ranges given. */
    int32_t tile_group;   /* tile rows visited together (tile and panel visit order;
                             default: the whole extent) */
    int32_t tile_stages;  /* shared-memory ring depth: 2..12 (tile, 128-row tiles),
                             2..6 (tile, 256-row tiles); cluster: staging ring, 1..8;
                             panel skew walk (panel_vec 4): 1 or 2 stages per CTA */
    int32_t tile_ctas_per_sm;  /* resident CTAs per SM the grid is sized for (block
                                  path: at most this many, 1..4) */
    int32_t tile_l2_promotion; /* L2 fill size of the TMA loads (tile path, panel phase
                                  maps): 64, 128, 256, or -1 = none */
    int32_t tile_rows;    /* tile height in rows of the dst-contiguous axis: 128 or 256
                             on the tile path, 16..1024 on the panel path (where both
                             plane extents exceed 16); other values select the default */
    int32_t cluster_recv_stages; /* cluster: receive ring depth, 1..8 (staging + receive
                                    slots at most 12) */
    int32_t cluster_consumer_warps; /* cluster: consumer warps per CTA, 4 or 8; block:
                                       this many, 1..17, as far as the SM's registers
                                       allow at the CTAs per SM its shared memory holds
                                       (by default 8, or 4 for tiles of 48 src runs or
                                       more) */
    int32_t panel_tile_kib;       /* panel path: tile size, 4..48 KiB (default 32, or 24
                                     with an extent of 16 or less; the skew walk: 256 x
                                     256 elements, 128 x 256 at 32 KiB or less); block
                                     path: its tile's bytes */
    int32_t cast;         /* TL_CAST_*: convert every element on the way (elem_bytes
                             and src_strides are the source type's, dst_strides the
                             destination type's); the tile, chunk, block and generic
                             paths take casts, a forced other path returns
                             TL_ERR_PATH */
    uint64_t *cta_times;  /* nullable DEVICE array (measurement): the tile, rows, panel
                             and block kernels write each CTA's start and finish time
                             (%globaltimer, ns) to cta_times[2 * b] and [2 * b + 1] for
                             CTA b of the grid tl_plan reports */
} tl_permute_opts;

/* tl_permute with options (path forcing, status word, buffer bounds): the same
 * operation ("Buffers and memory", "Declaring buffers"; "permute_layout", "What it
 * accepts").  Forcing a path is the dispatch choice "permute_layout" describes as a
 * variant that accepts or declines a call ("What it accepts"): a forced path that
 * does not apply returns TL_ERR_PATH and launches nothing, as a declined variant
 * does.  The status word reports the bounded waits of the mbarrier completions
 * ("copy_async -> dsmem", "Algorithm"; the wait_until pull request, "The
 * operation").  opts may be NULL (same as tl_permute). */
TL_API int tl_permute_ex(const void *src, void *dst, int ndim, const int64_t *shape,
                  const int64_t *src_strides, const int64_t *dst_strides, int elem_bytes,
                  tl_stream_t stream, const tl_permute_opts *opts);

/* What the planner would do for a call (host only; pointers are used for their
 * alignment only and never dereferenced; no GPU needed except for grid sizing,
 * which reports 0 when no device is present). */
typedef struct tl_plan_info {
    int32_t path;                  /* TL_PATH_* chosen */
    int32_t ndim;                  /* canonical rank (sorted by dst stride, merged) */
    int64_t extent[TL_MAX_DIMS];
    int64_t src_str[TL_MAX_DIMS];
    int64_t dst_str[TL_MAX_DIMS];
    int32_t vec_bytes;             /* vector width of global accesses */
    int32_t in_place;              /* 1 when src == dst and the warp path runs in place */
    int32_t k, shift, mask;        /* warp path swizzle (else 0) */
    int32_t tile_rows, tile_cols;  /* tile/panel path: rows (b) x columns (a) per tile,
                                      in elements; cols path: pixels per 16-byte piece x
                                      elements per pixel; block path: the dst run x the
                                      src run of a tile, in elements */
    int64_t tiles;                 /* work units (tiles, rows, warps...) */
    int32_t grid, block;           /* launch shape (0 without a device) */
    int32_t smem_bytes;            /* dynamic shared memory per CTA */
    int32_t pitch;                 /* panel path: shared-memory bytes per tile row;
                                      block path: between neighbouring src runs */
    int32_t panel_mode;            /* panel path: 0 rows of 16-byte blocks, 1 one run,
                                      2 rows loaded by TMA phase maps into a phase-major
                                      stage (a row pitch off the 16-byte grid), 3 the
                                      same stage filled by cp.async */
    int32_t panel_b1;              /* panel path: > 0 when the dst-contiguous axis (extent
                                      panel_b1) and the next dst axis are walked as one */
    int32_t panel_vec;             /* panel path store mode: 1 tiles stored as 16-byte dst
                                      runs along their rows, 2 as 16-byte pieces of the
                                      single dst run of a tile (a short dst-contiguous
                                      axis), 3 as 4-byte words per dst row (1-byte block
                                      rows off the 16-byte grid), 4 as 16-byte pieces of
                                      dst rows at an odd pitch (1-byte elements, the skew
                                      walk), 0 element by element
                                      (4-byte words for packed rows of 1- and 2-byte
                                      elements) */
    int32_t panel_wrot;            /* panel path, modes stored as 4-byte words: the lanes'
                                      read rotation, shift | multiplier << 8 */
    int32_t panel_a1;              /* panel path: > 0 when a short src-contiguous axis a
                                      was merged with the next src axis (src dense across
                                      the two); the inner extent, each tile row's dst
                                      offset then splits a into its two axes */
    int32_t block_runs;            /* block path: dst runs a warp of the store walk covers
                                      at once (1: consecutive elements in dst order, on
                                      into the next run; 2 .. 32: as many runs, an equal
                                      share of consecutive pieces in each) */
} tl_plan_info;

TL_API int tl_plan(const void *src, const void *dst, int ndim, const int64_t *shape,
            const int64_t *src_strides, const int64_t *dst_strides, int elem_bytes,
            const tl_permute_opts *opts, tl_plan_info *out);

/*
 * tl_thread_axis_check -- validate a warp's thread-axis layout (TVM "Buffers and
 * memory", "Buffer APIs", "Registers -- local": S[(32, 8) : (1 @ laneid, 1)] with
 * R.local(8) puts element (l, j) in register j of lane l) and count the registers
 * each lane holds.  Host only; the device side is tl_dev::ThreadAxisLayout with
 * warp_load_lanes / warp_store_lanes in tl_permute_device.cuh.
 *
 *   ndim        1..4
 *   extent      host array of ndim extents (>= 1)
 *   lane_str    host array: the "s @ laneid" stride of each axis, 0 if the axis is
 *               a register axis
 *   reg_str     host array: the register stride of each axis, 0 if the axis is a
 *               lane axis
 *   registers   out: registers per lane (P)
 * Returns TL_OK when every axis is on exactly one side and the coordinates fall on
 * 32 lanes x P registers once each; TL_ERR_EXTENT otherwise; TL_ERR_ARG for null
 * pointers or ndim out of range.
 */
TL_API int tl_thread_axis_check(int ndim, const int64_t *extent, const int64_t *lane_str,
                                const int64_t *reg_str, int *registers);

/* Human-readable text of a status code (static storage).  The decline reasons
 * are worded after the reasons the permute_layout dispatch gives ("permute_layout",
 * "What it accepts"); the others name this library's own errors. */
TL_API const char *tl_status_string(int status);

/* Number of kernels this library has launched in this process. */
TL_API uint64_t tl_launch_count(void);

/*
 * Number of tl_permute / tl_permute_ex / tl_plan calls served from the plan cache.
 * The library keeps the plans of recent calls (256 slots, process-wide, guarded by
 * a mutex): a call whose layout, element width, flags, tuning options, device and
 * base-address offsets within 16 bytes match an earlier call's reuses its plan and
 * launch shape.  The checks that depend on the pointers themselves (null pointers,
 * caller-given bounds, overlap of the two byte ranges) still run on every call, and
 * calls whose ranges meet (in place, or rejected as aliased) are planned afresh.
 */
TL_API uint64_t tl_plan_cache_hits(void);

/* TL_VERSION of the loaded library. */
TL_API int tl_version(void);

/*
 * tl_permute_tile_noalloc -- the TMA tile transpose (TL_PATH_TILE) for callers
 * that cannot allocate device memory.  The TVM pages have no counterpart: it
 * exists for integration, not for the method.
 *
 * Who needs it: plug-ins living inside a framework whose caching allocator
 * already owns the device's memory budget (a cudaMalloc of their own would
 * compete with it), code on latency-critical paths where cudaMalloc's implicit
 * device synchronisation is not acceptable, and fixed-memory or real-time
 * deployments whose policy forbids allocating after start-up.  Such callers
 * cannot provide the status word that tl_permute_ex takes in opts.dev_status.
 *
 * What it does: the same launch as tl_permute_ex with TL_PATH_TILE, except that
 * the kernel's only scratch -- the 4-byte status word it writes when a bounded
 * wait expires -- lives in a file-scope device array of
 * TL_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that loads
 * the library keeps until the process exits.  The call zeroes that word on
 * `stream`, launches, and, if host_status is not NULL, copies the word into
 * *host_status on the same stream (0 = ok, TL_ERR_TIMEOUT = a wait expired;
 * valid once the stream has reached that point; pass pinned host memory to keep
 * the call asynchronous).  It calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 *   src, dst, ndim, shape, src_strides, dst_strides, elem_bytes, stream:
 *       as tl_permute; the layout must admit the tile path
 *   host_status  nullable host pointer (see above)
 * Returns TL_OK; TL_ERR_PATH if the tile path does not apply; TL_ERR_BOUNDS if
 * the launch would need more scratch than TL_NOALLOC_SCRATCH_BYTES; otherwise
 * the errors of tl_permute.
 *
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture begins.  All
 * calls share the one array and it keeps the last call's contents: calls whose
 * work overlaps on the GPU (other streams, other host threads) race on the
 * status word, so one call's report may be cleared or overwritten by another's.
 * The looked-up address is kept for the life of the process: after a
 * cudaDeviceReset of a device, do not call this entry point on it again.
 */
#define TL_NOALLOC_SCRATCH_BYTES 256
TL_API int tl_permute_tile_noalloc(const void *src, void *dst, int ndim, const int64_t *shape,
                                   const int64_t *src_strides, const int64_t *dst_strides,
                                   int elem_bytes, tl_stream_t stream, int32_t *host_status);

#ifdef __cplusplus
}
#endif

#endif /* TL_PERMUTE_H */
