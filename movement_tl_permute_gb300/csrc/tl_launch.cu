// tl_launch.cu -- C ABI entry points that touch the GPU: tl_permute,
// tl_permute_ex and tl_plan.  Validates and plans on the host (tl_host.cpp),
// encodes the TMA tensor map for the tile path, sizes persistent grids from the
// device's SM count and occupancy, and launches one kernel on the caller's stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "tl_internal.h"
#include "tl_kernels.h"

namespace tl {

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s per bounded wait
constexpr uint64_t kTestTimeoutNs = 50000000ull;        // 50 ms under the test hook

struct DevInfo {
    bool ready = false;
    int sms = 0;
    int tile_occ[5][2][kMaxTileStages + 1] = {};  // CTAs per SM of k_tile<EB, 128|256> by depth
    int cluster_occ[5][2][kMaxClusterSlots + 1] = {}; // by consumer warps (8|4), slots
};

// Tile-path tuning.  The defaults were measured on GB300 over the batched 128x64
// tile transpose and the 2-D transposes of every element width: about 600-700
// tiles (10-11 MB) in flight GPU-wide (ring depth and grid: tile_defaults) beat
// deeper rings and denser grids on every workload, and visiting every tile row of
// a column block before the next block (the whole b extent as one group) beat
// groups of 16 to 128 rows: the CTAs then write dst front to back as one
// sequential stream while their reads stay 128-byte rows.  256-row tiles were
// slower than 128-row tiles on every workload.
struct TileTuning {
    int group = 0;          // tile rows visited together (0 = the whole b extent)
    int rows = 128;         // tile height (128 or 256)
    int stages = 0;         // ring depth (0 = by element width, tile_defaults)
    int grid_per_152 = 0;   // tile grid per 152 SMs (0 = one CTA per SM)
    int ctas_per_sm = 0;    // resident CTAs the grid is sized for (0 = path default)
    int promotion = 256;    // L2 fill size of the TMA loads (0 = none)
    int cluster_stages = 2; // staging ring depth of the cluster variant
    int cluster_recv = 0;   // its receive ring depth (0 = by layout, cluster_defaults)
    int cluster_warps = 4;  // its consumer warps (8 or 4)
    int cluster_ctas = 0;   // its CTAs per SM (0 = by layout; tile_ctas_per_sm overrides)
    int block_warps = 0;    // block path: consumer warps at most (0 = as many as fit)
    int skew_stages = 0;    // panel skew walk: stages per CTA (0 = default)
};

// Tile-path ring depth and grid by element width.  Throughput against the tiles in
// flight is not smooth (a sweep of 3-6 stages x 96-152 CTAs on GB300 moved by up to
// 25 % between neighbouring points, repeatably); the best measured point was one CTA
// per SM with 4 stages for 1-, 4-, 8- and 16-byte elements and 136 CTAs with 5
// stages for 2-byte elements (batched 128x64 tiles 6.75 -> 6.83 TB/s, 2-D 6.58 ->
// 6.70 TB/s, repeated on separate boxes).  Explicit options replace both.
void tile_defaults(const Plan& p, const tl_permute_opts* o, TileTuning& t) {
    const bool user = o && o->tile_stages >= 2 && o->tile_stages <= kMaxTileStages;
    if (user) return;
    // Narrowing casts (fp32 -> 16-bit) run two CTAs per SM with 3 stages each: measured
    // on GB300, fp32 -> bf16 4.54 -> 5.32 TB/s and fp32 -> f16 4.85 -> 5.50 against one CTA
    // of 4 stages (their consumers, converting 4-byte words, pace the ring; the widening
    // casts keep one CTA: 6.19 against 5.17).
    const bool narrow = p.cast == TL_CAST_F32_TO_BF16 || p.cast == TL_CAST_F32_TO_F16;
    if (narrow && p.path == TL_PATH_TILE) {
        t.stages = 3;
        if (!(o && (o->tile_ctas_per_sm > 0 || o->max_ctas > 0))) t.ctas_per_sm = 2;
        return;
    }
    if (p.eb == 2 && t.rows == 128) {
        t.stages = 5;
        if (!(o && (o->tile_ctas_per_sm > 0 || o->max_ctas > 0))) t.grid_per_152 = 136;
    } else {
        t.stages = 4;
    }
    const int max_stages = kTileRingBytes / (t.rows * 128);
    if (t.stages > max_stages) t.stages = max_stages;
}

// The cluster variant, with its slot hand-backs released at CTA scope, is paced by
// the loads it keeps in flight GPU-wide, like the single-CTA kernel (throughput
// falls off a cliff past about 600-700 strided tiles).  Measured on GB300 with 4
// consumer warps and a 2-deep staging ring: tiles that are one contiguous 16 KiB
// run of src (the batched tile transpose) do best with 2 receive slots at 3 CTAs
// per SM (about 900 tiles in flight, 6.72 TB/s); strided tiles (2-D transposes)
// with 1 receive slot at 2 CTAs per SM (about 600, 5.8-6.1 TB/s).
void cluster_defaults(const Plan& p, TileTuning& t) {
    const bool contiguous = p.ext_a * p.eb == 128 && p.ss_b * p.eb == 128;
    if (t.cluster_recv == 0) t.cluster_recv = contiguous ? 2 : 1;
    if (t.cluster_stages + t.cluster_recv > kMaxClusterSlots)
        t.cluster_recv = kMaxClusterSlots - t.cluster_stages;
    if (t.cluster_ctas == 0) t.cluster_ctas = contiguous ? 0 : 2;
}

// Stages per CTA of the panel skew walk (tile_stages 1 or 2 overrides): one, two CTAs
// per SM.  Measured on GB300 against one CTA of two stages (8 warps an SM either way at
// two stages): odd-pitch u8 transposes 4.98 -> 5.02 (32767 x 32769), 4.54 -> 4.83
// (16385 x 16383), 4.76 -> 4.97 (32769 x 32767), 4.88 -> 5.20 TB/s (20000 x 30001):
// sixteen warps an SM hide more of the walk's latency than one CTA's own overlap of
// copies and stores.
int skew_stages(const TileTuning& t) { return t.skew_stages > 0 ? t.skew_stages : 1; }

TileTuning tile_tuning(const tl_permute_opts* o) {
    TileTuning t;
    if (!o) return t;
    if (o->tile_group > 0) t.group = o->tile_group;
    if (o->tile_stages >= 2 && o->tile_stages <= kMaxTileStages) t.stages = o->tile_stages;
    if (o->tile_stages >= 1 && o->tile_stages <= kMaxClusterStages)
        t.cluster_stages = o->tile_stages;
    if (o->cluster_recv_stages >= 1 && o->cluster_recv_stages <= kMaxClusterStages)
        t.cluster_recv = o->cluster_recv_stages;
    if (o->cluster_consumer_warps == 4 || o->cluster_consumer_warps == 8)
        t.cluster_warps = o->cluster_consumer_warps;
    if (o->cluster_consumer_warps >= 1 && o->cluster_consumer_warps < kBlockMaxWarps)
        t.block_warps = o->cluster_consumer_warps;
    if (o->tile_ctas_per_sm > 0) t.ctas_per_sm = o->tile_ctas_per_sm;
    if (o->tile_stages == 1 || o->tile_stages == 2) t.skew_stages = o->tile_stages;
    if (o->tile_rows == 256) t.rows = 256;
    const int max_stages = kTileRingBytes / (t.rows * 128);
    if (t.stages > max_stages) t.stages = max_stages;
    if (o->tile_l2_promotion == 64 || o->tile_l2_promotion == 128 ||
        o->tile_l2_promotion == 256)
        t.promotion = o->tile_l2_promotion;
    else if (o->tile_l2_promotion < 0)
        t.promotion = 0;
    return t;
}
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int log2i(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

int get_device_info(DevInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TL_ERR_CUDA;
        const void* kt[5][2] = {{tile_kernel<1, 128>(), tile_kernel<1, 256>()},
                                {tile_kernel<2, 128>(), tile_kernel<2, 256>()},
                                {tile_kernel<4, 128>(), tile_kernel<4, 256>()},
                                {tile_kernel<8, 128>(), tile_kernel<8, 256>()},
                                {tile_kernel<16, 128>(), tile_kernel<16, 256>()}};
        for (int i = 0; i < 5; ++i) {
            for (int h = 0; h < 2; ++h) {
                const int rows = 128 << h, max_st = kTileRingBytes / (rows * 128);
                if (cudaFuncSetAttribute(kt[i][h], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tile_smem_bytes(max_st, rows)) != cudaSuccess)
                    return TL_ERR_CUDA;
                for (int st = 2; st <= max_st; ++st)
                    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                            &d.tile_occ[i][h][st], kt[i][h], kTileThreads,
                            tile_smem_bytes(st, rows)) != cudaSuccess)
                        return TL_ERR_CUDA;
            }
            for (int v = 0; v < 4; ++v)
                if (cudaFuncSetAttribute(panel_kernel(1 << i, (v & 1) != 0, (v & 2) != 0),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kPanelMaxSmem) != cudaSuccess)
                    return TL_ERR_CUDA;
            if (i < 4 && cudaFuncSetAttribute(tile_cast_kernel(i + 1),
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              tile_smem_bytes(kTileRingBytes / (128 * 128),
                                                              128)) != cudaSuccess)
                return TL_ERR_CUDA;
            for (int v = 1; v <= (16 >> i); v <<= 1)
                if (cudaFuncSetAttribute(block_kernel(1 << i, v),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kBlockMaxSmem) != cudaSuccess)
                    return TL_ERR_CUDA;
            // the converting block kernels (fp32 -> 16-bit: pieces of up to 8, 16-bit ->
            // fp32: up to 4)
            if (i < 4)
                for (int v = 1; v <= (i < 2 ? 8 : 4); v <<= 1)
                    if (cudaFuncSetAttribute(block_kernel(i < 2 ? 4 : 2, v, i + 1),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kBlockMaxSmem) != cudaSuccess)
                        return TL_ERR_CUDA;
            for (int delta = 1; i == 0 && delta < 16; delta += 2)
                for (int stages = 1; stages <= kSkewStages; ++stages)
                    if (cudaFuncSetAttribute(panel_skew_kernel(delta, stages),
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kPanelMaxSmem) != cudaSuccess)
                        return TL_ERR_CUDA;
            if (panel_tma_kernel(1 << i) &&
                cudaFuncSetAttribute(panel_tma_kernel(1 << i),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPanelMaxSmem + 128) != cudaSuccess)
                return TL_ERR_CUDA;
            // The cluster variant is optional: if its set-up fails it is sized
            // conservatively (one CTA per SM) and the error is cleared.
            for (int h = 0; h < 2; ++h) {
                const int ncw = h ? 4 : 8;
                const void* kc = cluster_kernel(1 << i, ncw);
                const bool attr_ok =
                    cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         cluster_smem_bytes(kMaxClusterSlots)) == cudaSuccess;
                for (int st = 2; st <= kMaxClusterSlots; ++st) {
                    int& occ = d.cluster_occ[i][h][st];
                    if (!attr_ok || cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                        &occ, kc, cluster_threads(ncw), cluster_smem_bytes(st)) !=
                                        cudaSuccess ||
                        occ < 1) {
                        cudaGetLastError();
                        occ = 1;
                    }
                }
            }
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return TL_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = d;
    return TL_OK;
}

// Batch axes of the plane, innermost (smallest dst stride) first.
void batch_inner_first(const Plan& p, int64_t* ext, int64_t* ss, int64_t* ds) {
    for (int i = 0; i < p.batch.n; ++i) {
        const int j = p.batch.n - 1 - i;
        ext[i] = p.batch.ext[j];
        ss[i] = p.batch.ss[j];
        ds[i] = p.batch.ds[j];
    }
}

// Tensor map over the source plane: dim 0 = a in BYTES (raw bits, type UINT8),
// dim 1 = b, dims 2.. = batch.  Box = 128 bytes x p.tile_rows rows, 128-byte swizzle.
int encode_tile_map(const Plan& p, const void* src, int promotion, CUtensorMap* map,
                    int* rank) {
    if (!g_encode) return TL_ERR_CUDA;
    const int eb = p.eb;
    cuuint64_t dims[5];
    cuuint64_t strides[4];
    cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
    int64_t bext[3] = {1, 1, 1}, bss[3] = {0, 0, 0}, bds[3] = {0, 0, 0};
    batch_inner_first(p, bext, bss, bds);
    dims[0] = (cuuint64_t)(p.ext_a * eb);
    dims[1] = (cuuint64_t)p.ext_b;
    strides[0] = (cuuint64_t)(p.ss_b * eb);
    box[0] = 128;
    box[1] = (cuuint32_t)p.tile_rows;
    for (int i = 0; i < p.batch.n; ++i) {
        dims[2 + i] = (cuuint64_t)bext[i];
        strides[1 + i] = (cuuint64_t)(bss[i] * eb);
        box[2 + i] = 1;
    }
    *rank = 2 + p.batch.n;
    const CUtensorMapL2promotion promo =
        promotion == 64    ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
        : promotion == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
        : promotion == 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                           : CU_TENSOR_MAP_L2_PROMOTION_NONE;
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)*rank,
                          const_cast<void*>(src), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? TL_OK : TL_ERR_CUDA;
}

// The phase maps of the TMA panel kernel: map j covers the src rows b = j mod phi
// of the plane, base aligned down to 16 bytes, element type of the element width;
// dim 0 = a (elements, from the aligned base), dim 1 = b / phi (stride phi * pitch),
// dims 2.. = batch (innermost first).  Box = (ta + 16 / eb) x (tb / phi), no swizzle.
int encode_panel_maps(const Plan& p, const uint8_t* src, int promotion, PanelMaps* maps,
                      int* rank) {
    if (!g_encode) return TL_ERR_CUDA;
    const int eb = p.eb;
    const int phi = 1 << p.panel_phi_lg;
    const int64_t P = p.ss_b * eb;
    const CUtensorMapDataType type = eb == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                     : eb == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                               : CU_TENSOR_MAP_DATA_TYPE_UINT64;
    int64_t bext[3] = {1, 1, 1}, bss[3] = {0, 0, 0}, bds[3] = {0, 0, 0};
    batch_inner_first(p, bext, bss, bds);
    *rank = 2 + p.batch.n;
    for (int j = 0; j < phi; ++j) {
        const uintptr_t row0 = reinterpret_cast<uintptr_t>(src) + (uintptr_t)(j * P);
        const uintptr_t base = row0 & ~uintptr_t(15);
        const int64_t shift = (int64_t)(row0 - base) / eb;     // elements before a = 0
        cuuint64_t dims[5], strides[4];
        cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
        dims[0] = (cuuint64_t)(p.ext_a + shift);
        dims[1] = (cuuint64_t)((p.ext_b - j + phi - 1) / phi);
        strides[0] = (cuuint64_t)(phi * P);
        box[0] = (cuuint32_t)(p.tile_cols + 16 / eb);
        box[1] = (cuuint32_t)(p.tile_rows / phi);
        for (int i = 0; i < p.batch.n; ++i) {
            dims[2 + i] = (cuuint64_t)bext[i];
            strides[1 + i] = (cuuint64_t)(bss[i] * eb);
            box[2 + i] = 1;
        }
        const CUtensorMapL2promotion promo =
            promotion == 64    ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
            : promotion == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
            : promotion == 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                               : CU_TENSOR_MAP_L2_PROMOTION_NONE;
        const CUresult r =
            g_encode(&maps->m[j], type, (cuuint32_t)*rank, reinterpret_cast<void*>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return TL_ERR_CUDA;
    }
    return TL_OK;
}

// Lanes per row group of the chunk kernel: each lane moves two vectors of a
// row, so a group has the power of two covering half the row (at most a warp).
int chunk_group_lanes(int64_t vpr) {
    int g = 1;
    while (g < 32 && 2 * g < vpr) g <<= 1;
    return g;
}

int cap_grid(int64_t want, int64_t cap, int32_t max_ctas) {
    int64_t g = want < cap ? want : cap;
    if (max_ctas > 0 && g > max_ctas) g = max_ctas;
    return (int)(g < 1 ? 1 : g);
}

struct Launch {
    int grid = 0, block = 0, smem = 0;
};

// The block kernel's arguments from the plan (pointers left null): the tables' axes,
// the chunked axis, the batch axes innermost first, and the shared-memory layout.
// Resident rings (pipelines) per SM of the block path: as many single-pipeline CTAs as
// the shared memory holds (228 KiB per SM, 1 KiB reserved per CTA, plus the barriers
// and tile records), at most four, or the tuning option's count; where exactly two fit
// (and the option asks nothing) one CTA runs both pipelines.
int block_ring_sms(const Plan& p, const TileTuning& tt, int* groups) {
    const BlockPlan& b = p.blk;
    const int64_t tables = 4 * ((b.Ld + 3) & ~3) + 16 * b.Rd + 16 * b.Rs;
    const int64_t one = ((kBlockStages * b.stage + 127) & ~int64_t(127)) + tables;
    int per_sm = (int)(233472 / (one + 1024 + 256));
    per_sm = per_sm < 1 ? 1 : per_sm > kBlockCtasPerSm ? kBlockCtasPerSm : per_sm;
    *groups = 1;
    if (tt.ctas_per_sm > 0) {
        if (tt.ctas_per_sm < per_sm) per_sm = tt.ctas_per_sm;
    } else if (per_sm == 2) {
        *groups = 2;
    }
    return per_sm;
}

int block_ctas_per_sm(const Plan& p, const TileTuning& tt) {
    int groups;
    const int rings = block_ring_sms(p, tt, &groups);
    return rings / groups;
}

BlockArgs block_args(const Plan& p, const TileTuning& tt) {
    const BlockPlan& b = p.blk;
    const int eb = p.eb;
    BlockArgs a{};
    auto in_list = [](const int* l, int n, int q) {
        for (int k = 0; k < n; ++k)
            if (l[k] == q) return true;
        return false;
    };
    a.nd = b.nd;
    a.nj = b.nj;
    a.nr = b.nr;
    a.jck = a.rck = -1;
    for (int k = 0; k < b.nd; ++k) {
        const int q = b.dax[k];
        a.dext[k] = (int32_t)b.tile[q];
        a.dsq[k] = (uint32_t)b.sq[q];
    }
    for (int k = 0; k < b.nj; ++k) {
        const int q = b.jax[k];
        a.jext[k] = (int32_t)b.tile[q];
        a.jsq[k] = (uint32_t)b.sq[q];
        a.jds[k] = b.ds[q];
        if (q == b.chunk) a.jck = k;
    }
    for (int k = 0; k < b.nr; ++k) {
        const int q = b.rax[k];
        a.rext[k] = (int32_t)b.tile[q];
        a.rsq[k] = (uint32_t)b.sq[q];
        a.rsb[k] = b.ss[q] * eb;
        if (q == b.chunk) a.rck = k;
    }
    a.Ld = (int32_t)b.Ld;
    a.Rd = (int32_t)b.Rd;
    a.Rs = (int32_t)b.Rs;
    a.Ls = (int32_t)b.Ls;
    a.ld_chunk = b.chunk >= 0 && in_list(b.dax, b.nd, b.chunk) ? 1 : 0;
    a.ls_chunk = b.chunk >= 0 && in_list(b.sax, b.ns, b.chunk) ? 1 : 0;
    a.ld_inner = a.ld_chunk ? (int32_t)(b.Ld / b.tile[b.chunk]) : a.Ld;
    a.ls_inner = a.ls_chunk ? (int32_t)(b.Ls / b.tile[b.chunk]) : a.Ls;
    a.cast = p.cast;
    a.V = b.vec;
    a.W = a.Ld / a.V;
    a.r_lg = b.r_lg;
    a.GW = (a.W + (32 >> a.r_lg) - 1) / (32 >> a.r_lg);
    a.GR = (a.Rd + (1 << a.r_lg) - 1) >> a.r_lg;
    a.stage_bytes = (int32_t)b.stage;
    // pipelines and consumer warps: 8 consumer warps, 4 for tiles of 48 src runs or more
    // at two rings per SM or more (measured on GB300, ten layouts: 8 against 4 ran
    // 1.08-1.17x on tiles of 9 and 36 runs -- 9^8 fp32, 12^7 and 12^8 u16 --, 4 ran
    // 1.04-1.09x on tiles of 64-100 runs -- other 9^8 orders, reversed 8^8 and 10^8,
    // 12^8 u8 -- and equal at 24 and 48; 17 ran slower everywhere but one); an SM keeps
    // 36 warps at most, a CTA 18
    int groups;
    const int rings = block_ring_sms(p, tt, &groups);
    a.groups = groups;
    int warps = (b.Rs >= 48 && rings >= 2) ? 5 : kBlockDefaultWarps;
    if (tt.block_warps > 0) warps = tt.block_warps + 1;
    warps = std::min(warps, std::min(kBlockSmWarps / rings, kBlockMaxWarps / groups));
    a.cw = warps - 1;
    a.ring_bytes = (kBlockStages * a.stage_bytes + 127) & ~127;
    a.table_off = groups * a.ring_bytes;
    if (b.chunk >= 0) {
        const int q = b.chunk;
        a.c_ext = b.ext[q];
        a.c_k = (int32_t)b.tile[q];
        a.c_ss = b.ss[q];
        a.c_ds = b.ds[q];
        a.nc = (b.ext[q] + b.tile[q] - 1) / b.tile[q];
    } else {
        a.c_ext = 1;
        a.c_k = 1;
        a.nc = 1;
    }
    // the batch axes innermost first by src stride: tiles reading neighbouring src runs
    // (which share DRAM blocks at the run ends) are then in flight together (measured on
    // GB300, against dst order: 12^8 u16 in the interleaved order read 1.27x -> 1.00x its
    // bytes, 12^8 fp32 1.10x -> 1.04x and 7 % less time, 9^8 fp32 unchanged)
    a.nb = b.batch.n;
    {
        int ord[TL_MAX_DIMS];
        for (int i = 0; i < a.nb; ++i) ord[i] = i;
        std::sort(ord, ord + a.nb, [&](int x, int y) { return b.batch.ss[x] < b.batch.ss[y]; });
        for (int i = 0; i < a.nb; ++i) {
            const int j = ord[i];
            a.bext[i] = b.batch.ext[j];
            a.bss[i] = b.batch.ss[j];
            a.bds[i] = b.batch.ds[j];
        }
    }
    a.tiles = p.tiles;
    a.use32 = p.tiles < (1LL << 32) ? 1 : 0;
    a.d_nc = dev::make_divu32((uint32_t)a.nc);
    if (a.use32)
        for (int i = 0; i < a.nb; ++i) a.d_bext[i] = dev::make_divu32((uint32_t)a.bext[i]);
    return a;
}

// Launch shape of each path (grid 0 when the device is unknown).
Launch launch_shape(const Plan& p, const DevInfo* d, int32_t max_ctas, const TileTuning& tt) {
    Launch l;
    const int64_t sms = d ? d->sms : 0;
    switch (p.path) {
    case TL_PATH_GENERIC:
        l.block = 256;
        if (sms) l.grid = cap_grid((p.total + 255) / 256, sms * 8, max_ctas);
        break;
    case TL_PATH_CHUNK: {
        l.block = 256;
        const int64_t vpr = p.row_elems * p.eb / p.vec_bytes;
        const int g = chunk_group_lanes(vpr);
        const int64_t groups = 256 / g;
        // 6 CTAs of 256 threads per SM measured best on GB300 (attention permute)
        if (sms) l.grid = cap_grid((p.rows + groups * 4 - 1) / (groups * 4), sms * 6, max_ctas);
        break;
    }
    case TL_PATH_TILE:
        l.block = kTileThreads;
        l.smem = tile_smem_bytes(tt.stages, p.tile_rows);
        if (sms) {
            int per_sm = d->tile_occ[log2i(p.eb)][p.tile_rows == 256 ? 1 : 0][tt.stages];
            const int want = tt.ctas_per_sm > 0 ? tt.ctas_per_sm : 1;
            if (want < per_sm) per_sm = want;
            int64_t cap = sms * (per_sm < 1 ? 1 : per_sm);
            if (tt.grid_per_152 > 0) cap = (sms * tt.grid_per_152 + 151) / 152;
            l.grid = cap_grid(p.tiles, cap, max_ctas);
        }
        break;
    case TL_PATH_CLUSTER:
        l.block = cluster_threads(tt.cluster_warps);
        l.smem = cluster_smem_bytes(tt.cluster_stages + tt.cluster_recv);
        if (sms) {
            // as many clusters as fit
            int per_sm = d->cluster_occ[log2i(p.eb)][tt.cluster_warps == 4 ? 1 : 0]
                                       [tt.cluster_stages + tt.cluster_recv];
            const int want = tt.ctas_per_sm > 0 ? tt.ctas_per_sm : tt.cluster_ctas;
            if (want > 0 && want < per_sm) per_sm = want;
            int64_t cap = sms * (per_sm < 1 ? 1 : per_sm) / 2;
            if (cap < 1) cap = 1;
            l.grid = 2 * cap_grid(p.tiles, cap, max_ctas > 0 ? (max_ctas + 1) / 2 : 0);
        }
        break;
    case TL_PATH_PANEL:
        if (p.panel_skew) {
            const int stages = skew_stages(tt);
            l.block = 32 * p.panel_skew_warps;
            l.smem = stages * p.panel_stage;
            if (sms) {
                int per_sm = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                        &per_sm, panel_skew_kernel((int)((16 - (p.ds_a & 15)) & 15), stages),
                        l.block, l.smem) != cudaSuccess ||
                    per_sm < 1) {
                    cudaGetLastError();
                    per_sm = 1;
                }
                l.grid = cap_grid(p.tiles, sms * per_sm, max_ctas);
            }
            break;
        }
        l.block = kPanelThreads;
        l.smem = kPanelStages * p.panel_stage;   // <= kPanelMaxSmem for tiles of <= 32 KiB
        if (p.panel_tma) l.smem += 128;           // the stages start on a 128-byte boundary
        if (sms) {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm,
                                                              p.panel_tma ? panel_tma_kernel(p.eb)
                                                                          : panel_kernel(p.eb, p.panel_vec, p.panel_a1 > 0),
                                                              kPanelThreads, l.smem) !=
                    cudaSuccess ||
                per_sm < 1) {
                cudaGetLastError();
                per_sm = 1;
            }
            l.grid = cap_grid(p.tiles, sms * per_sm, max_ctas);
        }
        break;
    case TL_PATH_BLOCK: {
        const BlockArgs a = block_args(p, tt);
        l.smem = block_smem_bytes(a);
        l.block = 32 * (a.cw + 1) * a.groups;
        if (sms) l.grid = cap_grid(p.tiles, sms * block_ctas_per_sm(p, tt), max_ctas);
        break;
    }
    case TL_PATH_ROWS:
        l.block = p.ext_b >= 16 ? 128 : 256;   // must match rows_threads<R>() in k_rows.cu
        if (sms) l.grid = cap_grid((p.tiles + 511) / 512, sms * 8, max_ctas);
        break;
    case TL_PATH_COLS:
        l.block = kColsThreads;
        if (sms) l.grid = cap_grid((p.tiles + kColsThreads - 1) / kColsThreads, sms * 8, max_ctas);
        break;
    case TL_PATH_WARP:
        l.block = 128;
        if (sms) l.grid = cap_grid((p.tiles + 3) / 4, sms * 16, max_ctas);
        break;
    }
    return l;
}

// The panel tile size and height are tuning options: re-plan the panel layout for them.
void apply_panel_tile(Plan& p, const tl_permute_opts* o) {
    if (p.path == TL_PATH_BLOCK && o && o->panel_tile_kib >= 4 && o->panel_tile_kib <= 48) {
        Plan q = p;                      // the block tile of the asked size, if one fits
        if (plan_block(&q, o->panel_tile_kib * 1024) > 0) p = q;
        return;
    }
    if (p.path != TL_PATH_PANEL || !o) return;
    const bool kib = o->panel_tile_kib >= 4 && o->panel_tile_kib <= 48;
    const bool rows = o->tile_rows >= 16 && o->tile_rows <= 1024;
    if (!kib && !rows) return;
    plan_panel(&p, kib ? o->panel_tile_kib * 1024 : 0, rows ? o->tile_rows : 0);
    if (kPanelStages * p.panel_stage > kPanelMaxSmem) plan_panel(&p, 0);
}

// The tile path's tile height is a launch choice: re-count the tiles for it.
void apply_tile_rows(Plan& p, const TileTuning& tt) {
    // (the converting tile kernels take 128-row tiles only)
    if (p.path != TL_PATH_TILE || tt.rows == p.tile_rows || p.cast != TL_CAST_NONE) return;
    p.tile_rows = tt.rows;
    const int64_t ta = (p.ext_a + p.tile_cols - 1) / p.tile_cols;
    const int64_t tb = (p.ext_b + p.tile_rows - 1) / p.tile_rows;
    p.tiles = ta * tb * p.batch_total;
}

// 16 bytes per step for the generic kernel when dst's innermost axis is contiguous
// and src is a strided view (a gather): the innermost axis is counted in groups of
// 16/eb elements, every group 16-byte aligned in dst.
void generic_vector_mode(GenericArgs& a, int eb, uintptr_t dst) {
    a.vmode = 0;
    if (eb >= 16 || a.n < 1) return;
    const int64_t V = 16 / eb;
    const int in = a.n - 1;
    if (a.ext[in] % V != 0) return;
    auto aligned_side = [&](uintptr_t base, const int64_t* str) {
        if (base % 16 != 0) return false;
        for (int i = 0; i < in; ++i)
            if ((str[i] * eb) % 16 != 0) return false;
        return true;
    };
    // Only gathers (dst contiguous): a scatter from 16-byte loads would spread each
    // warp store over 32 sectors (measured 2.5 -> 1.7 TB/s), where per-element steps
    // keep consecutive lanes on consecutive strided addresses.
    if (a.ds[in] == 1 && aligned_side(dst, a.ds)) {
        a.vmode = 1;
        a.vstep = a.ss[in];
    } else {
        return;
    }
    a.ext[in] /= V;
    a.ss[in] *= V;
    a.ds[in] *= V;
    a.total /= V;
}

void fill_divs(int n, const int64_t* ext, dev::DivU32* div) {
    for (int i = 0; i < n; ++i) div[i] = dev::make_divu32((uint32_t)ext[i]);
}

// ---------------------------------------------------------------- plan cache
// What a launch needs besides the pointers themselves: the plan, the tile tuning and
// the launch shape.  They depend on the layout, the element width, the flags and
// tuning options, the device, and the two base addresses only through their offsets
// within 16 bytes (vector widths, the panel's row misalignment) and through whether
// the two byte ranges meet (in-place and alias cases, never cached).  A repeated
// call with the same key skips the planner; the checks that depend on the pointer
// values themselves (null pointers, caller-given bounds, overlap of the two ranges)
// still run on every call.
struct Prepared {
    Plan p;
    TileTuning tt;
    Launch l;
};

struct PlanKey {
    int32_t dev, ndim, eb, smis, dmis;
    uint32_t flags;
    int32_t o[10];                 // the tuning options and the cast of tl_permute_opts
    int64_t shape[kMaxDims], ss[kMaxDims], ds[kMaxDims];
};

constexpr int kPlanCacheSlots = 256;
struct PlanSlot {
    bool used = false;
    PlanKey key;
    Prepared val;
};
std::mutex g_cache_mu;
PlanSlot g_cache[kPlanCacheSlots];
std::atomic<uint64_t> g_cache_hits{0};
std::atomic<int> g_have_device{-1};   // -1 unknown, 0 no CUDA device in this process, 1 yes

// The current device, or -1 when the process has no CUDA device (remembered after
// the first failed query: a device does not appear in a running process).
int current_device() {
    if (g_have_device.load(std::memory_order_relaxed) == 0) return -1;
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        if (g_have_device.load(std::memory_order_relaxed) < 0) {
            const bool any = cudaGetDeviceCount(&n) == cudaSuccess && n > 0;
            if (!any) cudaGetLastError();
            g_have_device.store(any ? 1 : 0, std::memory_order_relaxed);
            if (!any) return -1;
        }
        return dev;
    }
    cudaGetLastError();
    g_have_device.store(0, std::memory_order_relaxed);
    return -1;
}

// FNV-1a over the key's 64-bit words, then a final mix of the high bits.
uint64_t key_hash(const PlanKey& k) {
    static_assert(sizeof(PlanKey) % 8 == 0, "the key hashes as whole 64-bit words");
    uint64_t w[sizeof(PlanKey) / 8];
    std::memcpy(w, &k, sizeof w);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof(PlanKey) / 8; ++i) h = (h ^ w[i]) * 1099511628211ull;
    return h ^ (h >> 29);
}

// Validates the call and fills `out`: from the cache when the same key was planned
// before, else by planning (and, with a device, sizing the launch) and caching the
// result.  `launch`: a device is required (tl_permute_ex); otherwise the launch
// shape is left at 0 when there is none (tl_plan).
int prepare(const void* src, const void* dst, int ndim, const int64_t* shape,
            const int64_t* ss, const int64_t* ds, int eb, const tl_permute_opts* opts,
            bool launch, Prepared* out) {
    const uint32_t flags = opts ? opts->flags : 0u;
    const int dev = current_device();
    const bool keyable = src && dst && ndim >= 0 && ndim <= kMaxDims &&
                         (ndim == 0 || (shape && ss && ds)) && (dev >= 0 || !launch);
    PlanKey key;
    uint64_t h = 0;
    if (keyable) {
        std::memset(&key, 0, sizeof key);      // padding and unused axes compare equal
        key.dev = dev;
        key.ndim = ndim;
        key.eb = eb;
        key.smis = (int32_t)(reinterpret_cast<uintptr_t>(src) & 15);
        key.dmis = (int32_t)(reinterpret_cast<uintptr_t>(dst) & 15);
        key.flags = flags;
        if (opts) {
            const int32_t o[10] = {opts->max_ctas, opts->tile_group, opts->tile_stages,
                                   opts->tile_ctas_per_sm, opts->tile_l2_promotion,
                                   opts->tile_rows, opts->cluster_recv_stages,
                                   opts->cluster_consumer_warps, opts->panel_tile_kib,
                                   opts->cast};
            std::memcpy(key.o, o, sizeof o);
        }
        for (int i = 0; i < ndim; ++i) {
            key.shape[i] = shape[i];
            key.ss[i] = ss[i];
            key.ds[i] = ds[i];
        }
        h = key_hash(key);
        bool hit = false;
        {
            std::lock_guard<std::mutex> lk(g_cache_mu);
            const PlanSlot& slot = g_cache[h % kPlanCacheSlots];
            if (slot.used && std::memcmp(&slot.key, &key, sizeof key) == 0) {
                *out = slot.val;
                hit = true;
            }
        }
        if (hit) {
            // the checks on the pointer values themselves
            const Plan& p = out->p;
            if (p.total == 0) return TL_OK;
            const int64_t sb = opts ? opts->src_bytes : 0, db = opts ? opts->dst_bytes : 0;
            if (((sb > 0 && p.sbytes > sb) || (db > 0 && p.dbytes > db)) &&
                !(flags & TL_FLAG_TEST_SKIP_HOST_BOUNDS))
                return TL_ERR_BOUNDS;
            const int64_t s0 = (int64_t)(uintptr_t)src, d0 = (int64_t)(uintptr_t)dst;
            if (!(s0 < d0 + p.dbytes && d0 < s0 + p.sbytes)) {
                g_cache_hits.fetch_add(1, std::memory_order_relaxed);
                return TL_OK;
            }
            // the two ranges meet: plan afresh (in-place or alias), as on a miss
        }
    }
    Prepared pr;
    int rc = make_plan(src, dst, ndim, shape, ss, ds, eb, flags, opts ? opts->src_bytes : 0,
                       opts ? opts->dst_bytes : 0, &pr.p, opts ? opts->cast : TL_CAST_NONE);
    if (rc != TL_OK) return rc;
    pr.tt = tile_tuning(opts);
    tile_defaults(pr.p, opts, pr.tt);
    cluster_defaults(pr.p, pr.tt);
    apply_tile_rows(pr.p, pr.tt);
    apply_panel_tile(pr.p, opts);
    DevInfo d;
    const bool have = pr.p.total > 0 && dev >= 0 && get_device_info(&d) == TL_OK;
    if (!have) {
        if (dev >= 0) cudaGetLastError();
        if (launch && pr.p.total > 0) return TL_ERR_CUDA;
    }
    pr.l = launch_shape(pr.p, have ? &d : nullptr, opts ? opts->max_ctas : 0, pr.tt);
    *out = pr;
    // cache plans whose ranges do not meet (and, for launches, whose shape is sized)
    if (keyable && !pr.p.in_place && (have || !launch)) {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        PlanSlot& slot = g_cache[h % kPlanCacheSlots];
        slot.used = true;
        slot.key = key;
        slot.val = pr;
    }
    return TL_OK;
}

int run(const void* src, void* dst, int ndim, const int64_t* shape, const int64_t* ss,
        const int64_t* ds, int eb, cudaStream_t st, const tl_permute_opts* opts) {
    const uint32_t flags = opts ? opts->flags : 0u;
    Prepared pr;
    int rc = prepare(src, dst, ndim, shape, ss, ds, eb, opts, true, &pr);
    if (rc != TL_OK) return rc;
    const Plan& p = pr.p;
    if (p.total == 0) return TL_OK;
    const TileTuning& tt = pr.tt;
    const Launch& l = pr.l;
    // overlap this launch with the drain of the previous kernel in the stream
    const bool pdl = (flags & TL_FLAG_NO_PDL) == 0;
    const uint8_t* s8 = static_cast<const uint8_t*>(src);
    uint8_t* d8 = static_cast<uint8_t*>(dst);
    cudaError_t err = cudaSuccess;

    switch (p.path) {
    case TL_PATH_GENERIC: {
        GenericArgs a{};
        a.src = s8;
        a.dst = d8;
        a.n = p.sorted.n;
        a.total = p.total;
        a.use32 = p.total < (1LL << 32) ? 1 : 0;
        for (int i = 0; i < a.n; ++i) {
            a.ext[i] = p.sorted.ext[i]; a.ss[i] = p.sorted.ss[i]; a.ds[i] = p.sorted.ds[i];
        }
        a.checked = (flags & TL_FLAG_DEBUG_CHECKS) ? 1 : 0;
        if (p.cast != TL_CAST_NONE) {
            a.use32 = a.total < (1LL << 32) ? 1 : 0;
            if (a.use32) fill_divs(a.n, a.ext, a.div);
            err = launch_generic_cast(p.cast, a, l.grid, l.block, st, pdl);
            break;
        }
        if (a.checked) {
            a.src_bytes = opts ? opts->src_bytes : 0;
            a.dst_bytes = opts ? opts->dst_bytes : 0;
            a.status = opts ? opts->dev_status : nullptr;
        } else {
            generic_vector_mode(a, eb, reinterpret_cast<uintptr_t>(dst));
        }
        a.use32 = a.total < (1LL << 32) ? 1 : 0;
        if (a.use32) fill_divs(a.n, a.ext, a.div);
        switch (eb) {
        case 1: err = launch_generic<1>(a, l.grid, l.block, st, pdl); break;
        case 2: err = launch_generic<2>(a, l.grid, l.block, st, pdl); break;
        case 4: err = launch_generic<4>(a, l.grid, l.block, st, pdl); break;
        case 8: err = launch_generic<8>(a, l.grid, l.block, st, pdl); break;
        default: err = launch_generic<16>(a, l.grid, l.block, st, pdl); break;
        }
        break;
    }
    case TL_PATH_CHUNK: {
        ChunkArgs a{};
        a.src = s8;
        a.dst = d8;
        a.rows = p.rows;
        a.vpr = p.row_elems * eb / p.vec_bytes;
        a.log2g = log2i(chunk_group_lanes(a.vpr));
        a.n = p.outer.n;
        a.use32 = p.rows < (1LL << 32) ? 1 : 0;
        for (int i = 0; i < a.n; ++i) {
            a.ext[i] = p.outer.ext[i];
            a.ss[i] = p.outer.ss[i] * eb;
            a.ds[i] = p.outer.ds[i] * p.deb;
        }
        if (a.use32) fill_divs(a.n, a.ext, a.div);
        if (p.cast != TL_CAST_NONE) {
            err = launch_chunk_cast(p.cast, p.vec_bytes, a, l.grid, l.block, st, pdl);
            break;
        }
        switch (p.vec_bytes) {
        case 16: err = launch_chunk<16>(a, l.grid, l.block, st, pdl); break;
        case 8: err = launch_chunk<8>(a, l.grid, l.block, st, pdl); break;
        case 4: err = launch_chunk<4>(a, l.grid, l.block, st, pdl); break;
        case 2: err = launch_chunk<2>(a, l.grid, l.block, st, pdl); break;
        default: err = launch_chunk<1>(a, l.grid, l.block, st, pdl); break;
        }
        break;
    }
    case TL_PATH_TILE:
    case TL_PATH_CLUSTER: {
        alignas(64) CUtensorMap map;
        TileArgs a{};
        rc = encode_tile_map(p, src, tt.promotion, &map, &a.rank);
        if (rc != TL_OK) return rc;
        a.dst = d8;
        a.status = opts ? opts->dev_status : nullptr;
        a.cta_times = opts ? opts->cta_times : nullptr;
        a.ext_a = p.ext_a;
        a.ext_b = p.ext_b;
        a.ds_a = p.ds_a;
        a.tiles_a = (p.ext_a + p.tile_cols - 1) / p.tile_cols;
        a.tiles_b = (p.ext_b + p.tile_rows - 1) / p.tile_rows;
        a.tiles = p.tiles;
        a.group_b = tt.group > 0 && tt.group < a.tiles_b ? tt.group : a.tiles_b;
        a.stages = tt.stages;
        a.nbatch = p.batch.n;
        a.vec_store = p.vec_store ? 1 : 0;
        for (int i = 0; i < 3; ++i) { a.bext[i] = 1; a.bds[i] = 0; }
        int64_t bss[3];
        batch_inner_first(p, a.bext, bss, a.bds);
        a.use32 = p.tiles < (1LL << 32) ? 1 : 0;
        if (a.use32) {
            const int64_t glast = a.tiles_b - ((a.tiles_b - 1) / a.group_b) * a.group_b;
            a.d_item = dev::make_divu32((uint32_t)(a.tiles_a * a.tiles_b));
            a.d_grp = dev::make_divu32((uint32_t)(a.group_b * a.tiles_a));
            a.d_gfull = dev::make_divu32((uint32_t)a.group_b);
            a.d_glast = dev::make_divu32((uint32_t)glast);
            fill_divs(3, a.bext, a.d_bext);
        }
        a.timeout_ns = (flags & TL_FLAG_TEST_DROP_HANDOFF) ? kTestTimeoutNs : kDefaultTimeoutNs;
        a.drop_handoff = (flags & TL_FLAG_TEST_DROP_HANDOFF) ? 1 : 0;
        if (p.path == TL_PATH_CLUSTER) {
            a.stages = tt.cluster_stages;
            a.recv_stages = tt.cluster_recv;
            err = launch_cluster(eb, tt.cluster_warps, map, a, l.grid, st, pdl);
            break;
        }
        if (p.cast != TL_CAST_NONE) {
            err = launch_tile_cast(p.cast, map, a, l.grid, st, pdl);
            break;
        }
        if (p.tile_rows == 256) {
            switch (eb) {
            case 1: err = launch_tile<1, 256>(map, a, l.grid, st, pdl); break;
            case 2: err = launch_tile<2, 256>(map, a, l.grid, st, pdl); break;
            case 4: err = launch_tile<4, 256>(map, a, l.grid, st, pdl); break;
            case 8: err = launch_tile<8, 256>(map, a, l.grid, st, pdl); break;
            default: err = launch_tile<16, 256>(map, a, l.grid, st, pdl); break;
            }
        } else {
            switch (eb) {
            case 1: err = launch_tile<1, 128>(map, a, l.grid, st, pdl); break;
            case 2: err = launch_tile<2, 128>(map, a, l.grid, st, pdl); break;
            case 4: err = launch_tile<4, 128>(map, a, l.grid, st, pdl); break;
            case 8: err = launch_tile<8, 128>(map, a, l.grid, st, pdl); break;
            default: err = launch_tile<16, 128>(map, a, l.grid, st, pdl); break;
            }
        }
        break;
    }
    case TL_PATH_PANEL: {
        PanelArgs a{};
        a.src = s8;
        a.dst = d8;
        a.ext_a = p.ext_a;
        a.ext_b = p.ext_b;
        a.ss_b = p.ss_b;
        a.ds_a = p.ds_a;
        a.ta = p.tile_cols;
        a.tb = p.tile_rows;
        a.pitch = p.pitch;
        a.mode = p.panel_mode;
        a.nblk = p.panel_nblk;
        a.merged = p.panel_b1 > 0 ? 1 : 0;
        a.b1 = a.merged ? p.panel_b1 : p.ext_b;
        a.ss_b2 = p.panel_ss_b2;
        a.d_b1 = dev::make_divu32((uint32_t)a.b1);
        a.stage_bytes = p.panel_stage;
        a.d_nblk = dev::make_divu32((uint32_t)(p.panel_nblk > 0 ? p.panel_nblk : 1));
        a.aligned = p.panel_aligned ? 1 : 0;
        a.vec = p.panel_vec ? 1 : 0;
        a.vpitch = p.panel_mode == kPanelRows ? p.pitch : p.tile_cols * eb;
        a.vdelta = p.panel_mode == kPanelRows && !a.merged ? (int32_t)((p.ss_b * eb) & 15) : 0;
        a.vskew = a.vec && p.panel_mode == kPanelRows ? 1 : 0;
        a.qb8 = (int32_t)std::max<int64_t>(1, ((int64_t)p.tile_rows * eb + 127) / 128);
        a.wrot_s = p.panel_wrot_s;
        a.wrot_m = p.panel_wrot_m;
        a.amerged = p.panel_a1 > 0 ? 1 : 0;
        a.ds_a2 = p.panel_ds_a2;
        a.d_a1 = dev::make_divu32((uint32_t)(p.panel_a1 > 0 ? p.panel_a1 : 1));
        a.run = p.panel_run ? 1 : 0;
        a.words = p.panel_words ? 1 : 0;
        a.tiles_a = (p.ext_a + a.ta - 1) / a.ta;
        a.tiles_b = (p.ext_b + a.tb - 1) / a.tb;
        a.tiles = p.tiles;
        a.nb = p.batch.n;
        for (int i = 0; i < TL_MAX_DIMS; ++i) { a.bext[i] = 1; a.bss[i] = 0; a.bds[i] = 0; }
        for (int i = 0; i < a.nb; ++i) {               // innermost (smallest dst stride) first
            const int j = a.nb - 1 - i;
            a.bext[i] = p.batch.ext[j]; a.bss[i] = p.batch.ss[j]; a.bds[i] = p.batch.ds[j];
        }
        a.d_tb = dev::make_divu32((uint32_t)a.tb);
        a.use32 = p.tiles < (1LL << 32) ? 1 : 0;
        // whole b extent by default (dst written front to back; measured best)
        a.group_b = opts && opts->tile_group > 0 && opts->tile_group < a.tiles_b
                        ? opts->tile_group
                        : a.tiles_b;
        if (a.use32) {
            const int64_t glast = a.tiles_b - ((a.tiles_b - 1) / a.group_b) * a.group_b;
            a.d_item = dev::make_divu32((uint32_t)(a.tiles_a * a.tiles_b));
            a.d_grp = dev::make_divu32((uint32_t)(a.group_b * a.tiles_a));
            a.d_gfull = dev::make_divu32((uint32_t)a.group_b);
            a.d_glast = dev::make_divu32((uint32_t)glast);
            fill_divs(a.nb, a.bext, a.d_bext);
        }
        const bool drop = (flags & TL_FLAG_TEST_DROP_HANDOFF) != 0;
        a.timeout_ns = drop ? kTestTimeoutNs : kDefaultTimeoutNs;
        a.status = opts ? opts->dev_status : nullptr;
        a.cta_times = opts ? opts->cta_times : nullptr;
        a.drop_load = drop && p.panel_tma ? 1 : 0;
        if (p.panel_phase) {
            a.phase = 1;
            a.phi_lg = p.panel_phi_lg;
            a.phase_bytes = p.panel_phase_bytes;
            a.nblk = p.panel_nblk;                 // the cp.async copy of the same tile
            a.d_nblk = dev::make_divu32((uint32_t)p.panel_nblk);
            a.aligned = 0;
        }
        if (p.panel_skew) {
            a.skew = 1;
            a.nblk = p.panel_nblk;
            a.d_nblk = dev::make_divu32((uint32_t)p.panel_nblk);
            err = launch_panel_skew(a, skew_stages(tt), l.grid, l.block, l.smem, st, pdl);
            break;
        }
        if (p.panel_tma) {
            PanelMaps maps;
            // 64-byte L2 fills unless the caller asked for another (measured best for
            // the phase maps' rows of 0.5-1 KiB at odd offsets)
            const int promo = opts && opts->tile_l2_promotion != 0 ? tt.promotion : 64;
            if (encode_panel_maps(p, s8, promo, &maps, &a.tma_rank) == TL_OK) {
                a.tma = 1;
                err = launch_panel_tma(eb, a, maps, l.grid, l.smem, st, pdl);
                break;
            }
            // no maps for this layout: cp.async fills the same phase-major stage (its
            // row pitch, ta * eb + 16, holds the blocks of a misaligned row)
        }
        err = launch_panel(eb, a, l.grid, l.smem, st, pdl);
        break;
    }
    case TL_PATH_BLOCK: {
        BlockArgs a = block_args(p, tt);
        a.src = s8;
        a.dst = d8;
        a.cta_times = opts ? opts->cta_times : nullptr;
        a.status = opts ? opts->dev_status : nullptr;
        const bool drop = (flags & TL_FLAG_TEST_DROP_HANDOFF) != 0;
        a.timeout_ns = drop ? kTestTimeoutNs : kDefaultTimeoutNs;
        a.drop_load = drop ? 1 : 0;
        err = launch_block(eb, a, l.grid, st, pdl);
        break;
    }
    case TL_PATH_COLS: {
        ColsArgs a{};
        a.src = s8;
        a.dst = d8;
        a.units = p.tiles;
        a.n_px = p.tile_rows;
        a.A = (int32_t)p.ext_a;
        a.upp = p.ext_b / a.n_px;
        a.ds_a = p.ds_a;
        a.n = p.batch.n;
        a.use32 = p.tiles < (1LL << 32) && a.upp < (1LL << 32) ? 1 : 0;
        for (int i = 0; i < a.n; ++i) {
            a.ext[i] = p.batch.ext[i]; a.ss[i] = p.batch.ss[i]; a.ds[i] = p.batch.ds[i];
        }
        if (a.use32) {
            a.div_upp = dev::make_divu32((uint32_t)a.upp);
            fill_divs(a.n, a.ext, a.div);
        }
        err = launch_cols(eb, a, l.grid, st, pdl);
        break;
    }
    case TL_PATH_ROWS: {
        RowsArgs a{};
        a.src = s8;
        a.dst = d8;
        a.cta_times = opts ? opts->cta_times : nullptr;
        a.units = p.tiles;
        a.upr = p.ext_a * eb / 16;
        a.ss_b = p.ss_b;
        a.n = p.batch.n;
        a.use32 = p.tiles < (1LL << 32) ? 1 : 0;
        for (int i = 0; i < a.n; ++i) {
            a.ext[i] = p.batch.ext[i]; a.ss[i] = p.batch.ss[i]; a.ds[i] = p.batch.ds[i];
        }
        if (a.use32) {
            a.div_upr = dev::make_divu32((uint32_t)a.upr);
            fill_divs(a.n, a.ext, a.div);
        }
        err = launch_rows(eb, (int)p.ext_b, a, l.grid, l.block, st, pdl);
        break;
    }
    case TL_PATH_WARP: {
        WarpArgs a{};
        a.src = s8;
        a.dst = d8;
        a.tn = p.wtile.n;
        a.bn = p.wbatch.n;
        a.shift = p.shift;
        a.mask = p.mask;
        a.items = p.tiles;
        for (int i = 0; i < a.tn; ++i) {
            a.text[i] = p.wtile.ext[i]; a.tss[i] = p.wtile.ss[i]; a.tds[i] = p.wtile.ds[i];
        }
        for (int i = 0; i < a.bn; ++i) {
            a.bext[i] = p.wbatch.ext[i]; a.bss[i] = p.wbatch.ss[i]; a.bds[i] = p.wbatch.ds[i];
        }
        err = launch_warp(eb, p.P, a, l.grid, l.block, st, pdl);
        break;
    }
    default:
        return TL_ERR_PATH;
    }
    if (err != cudaSuccess) return TL_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return TL_OK;
}

}  // namespace
}  // namespace tl

extern "C" {

int tl_permute(const void* src, void* dst, int ndim, const int64_t* shape,
               const int64_t* src_strides, const int64_t* dst_strides, int elem_bytes,
               tl_stream_t stream) {
    return tl::run(src, dst, ndim, shape, src_strides, dst_strides, elem_bytes,
                   reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int tl_permute_ex(const void* src, void* dst, int ndim, const int64_t* shape,
                  const int64_t* src_strides, const int64_t* dst_strides, int elem_bytes,
                  tl_stream_t stream, const tl_permute_opts* opts) {
    return tl::run(src, dst, ndim, shape, src_strides, dst_strides, elem_bytes,
                   reinterpret_cast<cudaStream_t>(stream), opts);
}

int tl_plan(const void* src, const void* dst, int ndim, const int64_t* shape,
            const int64_t* src_strides, const int64_t* dst_strides, int elem_bytes,
            const tl_permute_opts* opts, tl_plan_info* out) {
    using namespace tl;
    if (!out) return TL_ERR_ARG;
    Prepared pr;
    int rc = prepare(src, dst, ndim, shape, src_strides, dst_strides, elem_bytes, opts, false,
                     &pr);
    if (rc != TL_OK) return rc;
    const Plan& p = pr.p;
    tl_plan_info info{};
    info.path = p.path;
    info.ndim = p.sorted.n;
    for (int i = 0; i < p.sorted.n; ++i) {
        info.extent[i] = p.sorted.ext[i];
        info.src_str[i] = p.sorted.ss[i];
        info.dst_str[i] = p.sorted.ds[i];
    }
    info.vec_bytes = p.vec_bytes;
    info.in_place = p.in_place ? 1 : 0;
    if (p.path == TL_PATH_WARP) {
        info.k = p.k;
        info.shift = p.shift;
        info.mask = p.mask;
    }
    info.tile_rows = p.tile_rows;
    info.tile_cols = p.tile_cols;
    info.pitch = p.pitch;
    if (p.path == TL_PATH_BLOCK) {            // block tile: run lengths and the run pitch
        info.tile_rows = (int32_t)p.blk.Ld;
        info.tile_cols = (int32_t)p.blk.Ls;
        info.pitch = p.blk.pitch;
    }
    info.panel_mode = p.panel_tma ? 2 : p.panel_phase ? 3 : p.panel_mode;
    info.panel_b1 = (int32_t)p.panel_b1;
    info.panel_vec = p.panel_vec ? 1 : p.panel_run ? 2 : p.panel_words ? 3 : p.panel_skew ? 4 : 0;
    info.panel_wrot = p.panel_wrot_s | (p.panel_wrot_m << 8);
    info.panel_a1 = (int32_t)p.panel_a1;
    info.block_runs = p.path == TL_PATH_BLOCK ? 1 << p.blk.r_lg : 0;
    info.tiles = p.tiles;
    const Launch& l = pr.l;
    info.grid = l.grid;
    info.block = l.block;
    info.smem_bytes = l.smem;
    *out = info;
    return TL_OK;
}

uint64_t tl_launch_count(void) { return tl::g_launches.load(std::memory_order_relaxed); }

uint64_t tl_plan_cache_hits(void) { return tl::g_cache_hits.load(std::memory_order_relaxed); }

}  // extern "C"
