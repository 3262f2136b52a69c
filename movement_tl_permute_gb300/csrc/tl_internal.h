// tl_internal.h -- plan structures shared by the host planner (tl_host.cpp) and
// the launch code (tl_launch.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>

#include "../../include/tl_permute.h"

namespace tl {

constexpr int kMaxDims = TL_MAX_DIMS;
constexpr int kMaxBatch = 6;       // batch axes of the transpose paths
constexpr int kMaxTmaBatch = 3;    // a TMA tensor map has at most 5 dims: a, b + 3 batch
constexpr int kMaxWarpTileDims = 4;
constexpr int kWarpMaxRegBytes = 128;  // P * elem_bytes a lane may stage in registers
constexpr int64_t kWarpAutoMaxElems = 8192;  // tensors the planner gives the warp path

// A list of axes with per-side element strides.
struct Axes {
    int n = 0;
    int64_t ext[kMaxDims] = {};
    int64_t ss[kMaxDims] = {};
    int64_t ds[kMaxDims] = {};
};

// BLOCK path: a tile of up to kBlockAxes axes (T) that is a few long contiguous runs
// on both sides.  The src run is the longest chain of T's axes, from the one of src
// stride 1, each of src stride the product of the extents before it; the axes of T
// outside it index the src runs.  The dst run and its index axes likewise, from the
// axis of dst stride 1.  At most one axis of T is split into chunks (the last axis
// of each run it belongs to), so both runs stay dense.
constexpr int kBlockAxes = 4;
constexpr int kBlockMaxLd = 2048;     // dst run positions (per-CTA table entries)
constexpr int kBlockMaxRuns = 512;    // src runs and dst runs of a tile
struct BlockPlan {
    int nt = 0;                        // axes of T
    int idx[kBlockAxes] = {};          // their positions in the sorted canonical axes
    int64_t ext[kBlockAxes] = {}, ss[kBlockAxes] = {}, ds[kBlockAxes] = {};
    int64_t tile[kBlockAxes] = {};     // extent of the tile along each axis of T
    int chunk = -1;                    // the axis of T split into chunks (-1: none)
    int ns = 0, sax[kBlockAxes] = {};  // src-run axes (innermost first)
    int nd = 0, dax[kBlockAxes] = {};  // dst-run axes (innermost first)
    int nr = 0, rax[kBlockAxes] = {};  // src-run index axes
    int nj = 0, jax[kBlockAxes] = {};  // dst-run index axes
    int64_t Ls = 0, Rs = 0, Ld = 0, Rd = 0;   // run lengths and counts of a full tile
    int64_t sq[kBlockAxes] = {};       // shared-memory byte stride of each axis of T
    int64_t stage = 0;                 // shared-memory bytes of one ring stage
    int pitch = 0;                     // sq of the innermost src-run index axis (the
                                       // distance between neighbouring src runs)
    int vec = 1;                       // dst elements per store (dst runs permitting)
    int r_lg = 0;                      // a store warp-step covers 1 << r_lg dst runs
    Axes batch;                        // the axes outside T (dst order, outermost first)
};

struct Plan {
    int path = 0;          // TL_PATH_*; 0 with total == 0 means "nothing to do"
    int eb = 0;            // element bytes (of the source under a cast)
    int cast = 0;          // TL_CAST_*
    int deb = 0;           // destination element bytes
    int64_t total = 0;     // elements
    int64_t sbytes = 0, dbytes = 0;   // bytes each layout reaches from its base
    Axes sorted;           // unit axes dropped, sorted by dst stride (descending), merged
    Axes kept;             // unit axes dropped, order kept, merged (the page's canon)

    // CHUNK: rows of row_elems contiguous elements on both sides.
    int64_t row_elems = 0;
    int vec_bytes = 0;
    Axes outer;            // axes outside the row, dst order
    int64_t rows = 0;

    // TILE / ROWS / CLUSTER: plane (b: dst-contiguous, a: src-contiguous) + batch.
    int64_t ext_a = 0, ext_b = 0, ss_b = 0, ds_a = 0;
    Axes batch;            // batch axes (outermost first)
    int64_t batch_total = 1;
    bool vec_store = false;  // 16-byte aligned dst runs
    int tile_rows = 0, tile_cols = 0;   // TILE: 128 x 128/eb; PANEL: tb x ta elements
    int pitch = 0;                      // PANEL: shared-memory bytes per tile row
    int panel_mode = 0;                 // PANEL: PanelMode (block rows, one block run)
    int panel_nblk = 0;                 // PANEL: 16-byte blocks copied per row (at most)
    int panel_stage = 0;                // PANEL: shared-memory bytes of one ring stage
    int64_t panel_b1 = 0;               // PANEL: inner extent of b when two axes are merged
    int64_t panel_ss_b2 = 0;            // PANEL: src stride of the outer merged axis
    int64_t panel_a1 = 0;               // PANEL: inner extent of a when two axes are merged
    int64_t panel_ds_a2 = 0;            // PANEL: dst stride of the outer merged a axis
    bool panel_aligned = false;         // PANEL: every src row starts on a 16-byte boundary
    bool panel_vec = false;             // PANEL: tiles stored as 16-byte dst runs
    bool panel_elem_stores = false;     // PANEL: 16-byte dst runs declined by the caller
    int64_t src_mis16 = 0, dst_mis16 = 0;   // base addresses mod 16
    int panel_wrot_s = 0, panel_wrot_m = 0; // PANEL: word-store rotation (packed rows, eb < 4)
    bool panel_run = false;             // PANEL: each tile's dst is one run, stored in 16-byte pieces
    bool panel_words = false;           // PANEL: block rows of 1-/2-byte elements stored as words
    bool panel_tma = false;             // PANEL: stages filled by TMA phase maps
    bool panel_phase = false;           // PANEL: phase-major stages (TMA or cp.async)
    int panel_phi_lg = 0;               // PANEL (TMA): log2 of the phase count phi
    int panel_phase_bytes = 0;          // PANEL (TMA): shared-memory bytes of one phase block
    bool panel_skew = false;            // PANEL: the skew walk (1-byte, odd dst row pitch)
    int panel_skew_warps = 0;           // PANEL (skew): warps per CTA, 32 columns of a each
    int64_t tiles = 0;
    BlockPlan blk;                      // BLOCK

    // WARP: tile (innermost suffix of `kept`) + batch of the outer `kept` axes.
    Axes wtile;
    Axes wbatch;
    int P = 0, k = 0, shift = 0, mask = 0;
    bool in_place = false;
};

// Validates the call and fills `plan`.  Pure host code, no CUDA calls.
int make_plan(const void* src, const void* dst, int ndim, const int64_t* shape,
              const int64_t* src_strides, const int64_t* dst_strides, int elem_bytes,
              uint32_t flags, int64_t src_bytes, int64_t dst_bytes, Plan* plan,
              int cast = TL_CAST_NONE);

// Panel ring: stages per CTA and the dynamic shared memory the kernels are set up
// for; plan_panel shrinks a tile until its ring fits.
constexpr int kPanelStages = 3;
constexpr int kPanelMaxSmem = 160 * 1024;

// The panel path's skew walk (1-byte elements whose dst rows sit at an odd pitch):
// tiles of 32 * warps columns of a by kSkewRows rows of b, each staged with up to 15
// rows and 15 columns past it, in a ring of kSkewStages stages.  Stage row r holds
// the 16-byte blocks around the row's src bytes at r * pitch + 16 * (r / 16), pitch =
// columns + 32 bytes.
constexpr int kSkewRows = 256;
constexpr int kSkewStages = 2;     // the most stages a CTA holds
constexpr int skew_pitch(int ta) { return ta + 32; }
constexpr int skew_stage_bytes(int ta) {
    return ((kSkewRows + 15) * skew_pitch(ta) + 16 * (kSkewRows / 16 + 1) + 127) / 128 * 128;
}
static_assert(kSkewStages * skew_stage_bytes(256) <= kPanelMaxSmem, "skew ring too large");

// Tile shape and shared-memory layout of the panel path for tiles of about
// tile_bytes (0: the default size; tuning options may redo it).  Measured on
// GB300: 32 KiB tiles for planes with two long extents, 24 KiB when one extent is
// 16 or less (interleaved channels: 5.5-6.1 TB/s against 4.8-5.5 with 16 KiB).
// rows > 0 asks for that many rows of b per tile when both extents exceed 16.
void plan_panel(Plan* p, int tile_bytes, int rows = 0);

// BLOCK path: the tile of up to four axes whose shorter run (src or dst) is longest;
// fills p->blk and p->tiles.  Returns the shorter run in bytes, 0 if none applies.
int64_t plan_block(Plan* p, int64_t tile_bytes = 0);

// The bank simulator: worst conflict degree of one warp-wide access.
int bank_degree(int n_lanes, const int64_t* lane_offsets, int elem_bytes, bool hardware);

// XOR swizzle search of the warp path; returns TL_OK or a tl_status.
int choose_xor(int n, const int64_t* ext, const int64_t* ss, const int64_t* ds, int eb,
               int* k, int* shift, int* mask);

}  // namespace tl
