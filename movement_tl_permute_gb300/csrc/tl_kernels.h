// tl_kernels.h -- kernel argument blocks and launch wrappers (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tl_permute.h"
#include "tl_device.cuh"
#include "tl_internal.h"

#include <utility>

namespace tl {

// Launches `kernel` on `st`, with programmatic stream serialization when `pdl`
// (the kernels call dev::grid_dependency_wait before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- generic
struct GenericArgs {
    const uint8_t* src;
    uint8_t* dst;
    int32_t n;
    int32_t use32;               // 1: flat index and extents fit in 32 bits
    int64_t total;               // steps: elements, or 16-byte groups (vmode 1, 2)
    // vmode 1: a step is 16/EB consecutive dst elements (one 16-byte store, loads
    // vstep apart in src).  The innermost axis below is then counted in groups (its
    // extent divided, its strides multiplied, by 16/EB).
    int32_t vmode;
    int32_t checked;             // 1: TL_FLAG_DEBUG_CHECKS (bounds below, status word)
    int64_t vstep;
    int64_t src_bytes, dst_bytes;    // checked run: addressable bytes (0 = unchecked)
    int32_t* status;
    int64_t ext[TL_MAX_DIMS];
    int64_t ss[TL_MAX_DIMS];     // elements
    int64_t ds[TL_MAX_DIMS];
    dev::DivU32 div[TL_MAX_DIMS];
};
template <int EB>
cudaError_t launch_generic(const GenericArgs& a, int grid, int block, cudaStream_t st, bool pdl);
// the generic kernel converting every element (TL_CAST_*; dst offsets in dst elements)
cudaError_t launch_generic_cast(int cast, const GenericArgs& a, int grid, int block,
                               cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- chunk
struct ChunkArgs {
    const uint8_t* src;
    uint8_t* dst;
    int64_t rows;                // rows of contiguous bytes
    int64_t vpr;                 // vectors per row
    int32_t n;                   // outer axes
    int32_t log2g;               // lanes per row group = 1 << log2g
    int32_t use32;
    int32_t pad;
    int64_t ext[TL_MAX_DIMS];
    int64_t ss[TL_MAX_DIMS];     // BYTES
    int64_t ds[TL_MAX_DIMS];     // BYTES
    dev::DivU32 div[TL_MAX_DIMS];
};
template <int VB>
cudaError_t launch_chunk(const ChunkArgs& a, int grid, int block, cudaStream_t st, bool pdl);
// the chunk kernel converting every element: vb = source vector bytes (4, 2 or 1
// elements), ss in source bytes, ds in destination bytes
cudaError_t launch_chunk_cast(int cast, int vb, const ChunkArgs& a, int grid, int block,
                              cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- tile (TMA)
constexpr int kMaxClusterStages = 8;   // ring depth limit of each cluster ring
constexpr int kMaxClusterSlots = 12;   // staging + receive slots of one cluster CTA
constexpr int kMaxTileStages = 12;     // ring depth limit of the single-CTA tile kernel
constexpr int kTileThreads = 9 * 32;   // 8 consumer warps + 1 producer warp
// block of the cluster variant: ncw consumer warps + loader, pusher and watcher warps
__host__ __device__ constexpr int cluster_threads(int ncw) { return (ncw + 3) * 32; }
struct TileArgs {
    uint8_t* dst;
    int32_t* status;
    uint64_t* cta_times;                 // measurement: per-CTA start / finish (or null)
    int64_t ext_a, ext_b, ds_a;          // elements
    int64_t tiles_a, tiles_b, tiles, group_b;
    int32_t nbatch, rank, vec_store;
    int32_t drop_handoff;                // test hook of the cluster variant
    int64_t bext[3];
    int64_t bds[3];                      // dst strides of the batch axes, elements
    uint64_t timeout_ns;
    // 32-bit tile decode (use32 = 1 when tile indices fit in 32 bits)
    int32_t use32;
    int32_t stages;                      // ring depth (cluster: staging ring)
    int32_t recv_stages;                 // cluster: receive ring depth
    dev::DivU32 d_item;                  // tiles per batch item
    dev::DivU32 d_grp;                   // tiles per group of group_b tile rows
    dev::DivU32 d_gfull, d_glast;        // full / last group height
    dev::DivU32 d_bext[3];
};
// dynamic shared memory of the tile kernel: `stages` tiles of `rows` x 128 bytes
int tile_smem_bytes(int stages, int rows);
constexpr int kTileRingBytes = kMaxTileStages * 128 * 128;   // ring bound for any tile height
template <int EB, int TB>
const void* tile_kernel();
template <int EB, int TB>
cudaError_t launch_tile(const CUtensorMap& map, const TileArgs& a, int grid, cudaStream_t st,
                        bool pdl);

// the converting tile kernels (TL_CAST_*, 128-row tiles)
cudaError_t launch_tile_cast(int cast, const CUtensorMap& map, const TileArgs& a, int grid,
                             cudaStream_t st, bool pdl);
const void* tile_cast_kernel(int cast);

// tile path with a 2-CTA cluster and a DSMEM hand-off (k_cluster.cu)
int cluster_smem_bytes(int slots);   // staging + receive slots
const void* cluster_kernel(int eb, int ncw);   // ncw = consumer warps, 8 or 4
cudaError_t launch_cluster(int eb, int ncw, const CUtensorMap& map, const TileArgs& a, int grid,
                           cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- rows
struct RowsArgs {
    const uint8_t* src;
    uint8_t* dst;
    uint64_t* cta_times;         // measurement: per-CTA start / finish (or null)
    int64_t units;               // 16-byte source columns over all batch items
    int64_t upr;                 // units per plane (ext_a * EB / 16)
    int64_t ss_b;                // src stride of b, elements
    int32_t n;                   // batch axes
    int32_t use32;               // 1: unit index and extents fit in 32 bits
    int64_t ext[TL_MAX_DIMS];
    int64_t ss[TL_MAX_DIMS];     // elements
    int64_t ds[TL_MAX_DIMS];
    dev::DivU32 div_upr;
    dev::DivU32 div[TL_MAX_DIMS];
};
cudaError_t launch_rows(int eb, int r, const RowsArgs& a, int grid, int block, cudaStream_t st,
                        bool pdl);

// ---------------------------------------------------------------- cols
// Short src runs (pixels of A elements, A * eb <= 32 bytes, dense in src) -> one dst
// plane per a; a unit is one 16-byte piece (n_px = 16 / eb pixels) of every plane.
constexpr int kColsThreads = 256;
struct ColsArgs {
    const uint8_t* src;
    uint8_t* dst;
    int64_t units;               // pieces over all planes' b and batch items
    int64_t upp;                 // units per batch item (ext_b / n_px)
    int64_t ds_a;                // dst stride of a (elements): plane to plane
    int32_t A, n_px;             // elements per pixel, pixels per piece
    int32_t n;                   // batch axes
    int32_t use32;               // 1: unit index and extents fit in 32 bits
    int64_t ext[TL_MAX_DIMS];
    int64_t ss[TL_MAX_DIMS];     // elements
    int64_t ds[TL_MAX_DIMS];
    dev::DivU32 div_upp;
    dev::DivU32 div[TL_MAX_DIMS];
};
cudaError_t launch_cols(int eb, const ColsArgs& a, int grid, cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- panel
// Transpose of (ta x tb)-element tiles of the plane through shared memory: the
// 16-byte blocks covering each tile row are copied asynchronously (cp.async) into
// a ring of stages, then stored in dst order; any element alignment, up to 6 batch
// axes, tiny extents.
constexpr int kPanelThreads = 256;
enum PanelMode : int32_t {
    kPanelRows = 0,    // row b copied as the 16-byte blocks covering it, at byte
                       // b * pitch; element a at byte (row address mod 16) + a * eb
    kPanelFlat = 1,    // src rows packed back to back (ss_b == ta == ext_a): the tile's
                       // src bytes are one run; element (a, b) at mis + (b*ta + a)*eb
};
struct PanelArgs {
    const uint8_t* src;
    uint8_t* dst;
    int64_t ext_a, ext_b;        // plane: a src-contiguous, b dst-contiguous
    int64_t ss_b, ds_a;          // src stride of b, dst stride of a (elements)
    // b may be two axes merged because dst is dense across them: b = hi * b1 + lo,
    // src offset lo * ss_b + hi * ss_b2 (b1 >= ext_b when nothing is merged)
    int64_t b1, ss_b2;
    int32_t ta, tb;              // tile: ta elements of a x tb elements of b
    int32_t pitch;               // kPanelRows: shared-memory bytes per row (multiple of 16)
    int32_t mode;                // PanelMode
    int32_t nblk;                // kPanelRows: 16-byte blocks copied per row (at most)
    int32_t stage_bytes;         // shared memory of one stage (multiple of 16)
    int32_t nb;                  // batch axes (innermost first)
    int32_t use32;               // tile indices fit in 32 bits
    int64_t tiles_a, tiles_b, tiles;
    int64_t group_b;             // tile rows visited together (b fastest inside a group)
    int64_t bext[TL_MAX_DIMS], bss[TL_MAX_DIMS], bds[TL_MAX_DIMS];
    dev::DivU32 d_tb, d_nblk;    // divisors of the per-tile walks
    dev::DivU32 d_b1;            // b -> (hi, lo) when two axes are merged (b fits 32 bits)
    int32_t merged;              // 1 when b is two merged axes
    int32_t aligned;             // kPanelRows: every src row starts on a 16-byte boundary
    dev::DivU32 d_item, d_grp, d_gfull, d_glast;
    dev::DivU32 d_bext[TL_MAX_DIMS];
    // 16-byte dst runs (vec = 1): dst rows of every tile 16-byte aligned and tb * eb a
    // multiple of 128.  Row b of a stage starts at
    // b * vpitch + (vskew ? 16 * (b / (16 / eb)) : 0) + ((mis0 + b * vdelta) & 15).
    int32_t vec, vpitch, vdelta, vskew;
    int32_t qb8;                 // 8-block groups of one dst row of a tile (tb * eb / 128)
    // packed rows of 1- and 2-byte elements stored as words: lane l reads the k-th
    // element of its word as (k + wrot_m * (l >> wrot_s)) mod (4 / eb)
    int32_t wrot_s, wrot_m;
    // the tile's dst is one run (tb == ext_b <= 16, ds_a == tb): stored as 16-byte pieces
    int32_t run;
    // block rows of 1- and 2-byte elements stored as 4-byte words per dst row (rotation
    // in wrot_s / wrot_m, indexed by the word)
    int32_t words;
    // phase-major stages (phase = 1): tile row b sits in the block of phase
    // b % 2^phi_lg (phase_bytes apart), at row b >> phi_lg of pitch bytes; filled by
    // TMA phase maps (k_panel_tma, tma = 1) or by cp.async
    int32_t tma, phase, phi_lg, phase_bytes, tma_rank;
    int32_t drop_load;           // test hook: skip one phase load of the first tile
    // a may be two src-contiguous axes merged (amerged = 1): a = hi * a1 + lo, dst
    // offset lo * ds_a + hi * ds_a2 (a fits 32 bits)
    int32_t amerged;
    int32_t skew;                // the skew walk's kernel (k_panel_skew) is launched
    int64_t ds_a2;
    dev::DivU32 d_a1;
    int64_t timeout_ns;
    int32_t* status;
    uint64_t* cta_times;         // measurement: per-CTA start / finish (or null)
};
// The phase maps of k_panel_tma: map j covers the src rows b = j mod phi of the
// plane (stride phi * row pitch), its base aligned down to 16 bytes.
struct PanelMaps {
    CUtensorMap m[16];
};
cudaError_t launch_panel_tma(int eb, const PanelArgs& a, const PanelMaps& maps, int grid,
                             int smem, cudaStream_t st, bool pdl);
const void* panel_tma_kernel(int eb);
// vec: the 16-byte dst run kernel; am: a is two merged axes (two-level dst offsets)
const void* panel_kernel(int eb, bool vec, bool am);
cudaError_t launch_panel(int eb, const PanelArgs& a, int grid, int smem, cudaStream_t st,
                         bool pdl);
// The skew walk (1-byte elements, dst row pitch odd): one kernel per dst row pitch
// modulo 16 (`delta` = -pitch mod 16, odd) and ring depth (1 or 2 stages), 32 columns
// of a per warp of `block`.
const void* panel_skew_kernel(int delta, int stages);
cudaError_t launch_panel_skew(const PanelArgs& a, int stages, int grid, int block, int smem,
                              cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- block
// A tile of up to four axes (T) that is a few long contiguous runs on both sides.
// Every axis of T has a shared-memory byte stride (a src-run axis its src byte
// stride; a src-run index axis one congruent to its src byte stride modulo 16), so
// that each src run is one bulk copy of its 16-byte blocks and per-CTA tables (built
// once in shared memory) give the stage offset of the element at dst-run position i
// of dst run j as TA[i] + TB[j], and its dst offset as dof + dst_j + i.
// A pipeline is cw consumer warps and one producer warp with its own ring; a CTA runs
// one pipeline, or two side by side that share the tables and take the CTA's tiles from
// a shared counter (where two rings fit an SM: one CTA per SM then, so that no CTA's
// warps are favoured over another's by the schedulers).  The launch bounds (at most 18
// warps, two CTAs per SM) hold a thread to 56 registers, so an SM keeps 36 warps:
// four CTAs of 8 consumer warps, three of 11 or two of 17, by the CTAs its shared
// memory holds.
constexpr int kBlockMaxWarps = 18;
constexpr int kBlockSmWarps = 36;
constexpr int kBlockDefaultWarps = 9;       // 8 consumer warps (4 for tiles of many runs)
constexpr int kBlockStages = 3;
constexpr int kBlockMaxGroups = 2;
constexpr int kBlockCtasPerSm = 4;
constexpr int kBlockMaxSmem = 226 * 1024;   // stages of at most 48 KiB + the tables
struct BlockArgs {
    const uint8_t* src;
    uint8_t* dst;
    uint64_t* cta_times;         // measurement: per-CTA start / finish (or null)
    int32_t* status;             // first error of the launch (or null)
    uint64_t timeout_ns;         // bound of every mbarrier wait
    int32_t drop_load;           // test hook: the first copy of the first tile is skipped
    // the axes whose digits make i (dst-run axes), j (dst-run index axes) and r
    // (src-run index axes), innermost first, with the tile's extents and each axis's
    // shared-memory byte stride; (j) dst strides, (r) src byte strides
    int32_t nd, nj, nr;
    int32_t dext[4], jext[4], rext[4];
    uint32_t dsq[4], jsq[4], rsq[4];
    int64_t jds[4], rsb[4];
    int32_t jck, rck;            // index of the chunked axis in the j / r lists (-1: none)
    int32_t ld_chunk, ls_chunk;  // the chunked axis is the dst run's / src run's last axis
    int32_t Ld, Rd, Rs, Ls;      // run lengths and counts of a full tile
    int32_t ld_inner, ls_inner;  // run lengths without the chunked axis
    int32_t V, W;                // store pieces: V elements, W per dst run
    // a consumer warp-step: a group of 32 >> r_lg pieces in each of 1 << r_lg dst runs;
    // GW x GR groups per tile
    int32_t r_lg, GW, GR;
    int32_t cw;                  // consumer warps of a pipeline (cw + 1 warps each)
    int32_t groups;              // pipelines of the CTA (1 or 2)
    int32_t cast;                // TL_CAST_*: every element converted on the way
    int32_t stage_bytes;
    int32_t ring_bytes;          // one pipeline's stages, on a 128-byte boundary (the same
                                 // bank phase for every pipeline)
    int32_t table_off;           // byte offset of the tables in dynamic shared memory
    // the chunked axis: extent, tile extent, chunks, strides
    int64_t c_ext, c_ss, c_ds, nc;
    int32_t c_k, use32;
    // tiles: chunk index fastest, then the batch axes (smallest src stride first)
    int32_t nb;
    int64_t tiles;
    int64_t bext[TL_MAX_DIMS], bss[TL_MAX_DIMS], bds[TL_MAX_DIMS];
    dev::DivU32 d_nc;
    dev::DivU32 d_bext[TL_MAX_DIMS];
};
int block_smem_bytes(const BlockArgs& a);
// the kernel for elem_bytes eb storing v dst elements per step (v in 1 .. 16 / dst
// element bytes), converting under `cast` (TL_CAST_*)
const void* block_kernel(int eb, int v, int cast = TL_CAST_NONE);
cudaError_t launch_block(int eb, const BlockArgs& a, int grid, cudaStream_t st, bool pdl);

// ---------------------------------------------------------------- warp
struct WarpArgs {
    const uint8_t* src;
    uint8_t* dst;
    int32_t tn, bn;              // tile axes, batch axes
    int32_t shift, mask;
    int64_t items;               // batch items (one warp tile each)
    int64_t text[4], tss[4], tds[4];
    int64_t bext[TL_MAX_DIMS], bss[TL_MAX_DIMS], bds[TL_MAX_DIMS];
};
cudaError_t launch_warp(int eb, int P, const WarpArgs& a, int grid, int block, cudaStream_t st,
                        bool pdl);

}  // namespace tl
