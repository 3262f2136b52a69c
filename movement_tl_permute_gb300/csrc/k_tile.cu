// k_tile.cu -- batched 2-D transpose through TMA-staged, 128B-swizzled shared memory.
//
// Plane: axis a is contiguous in src (stride 1), axis b is contiguous in dst
// (stride 1); every other axis is a batch axis.  A tile is TB rows of b by 128
// BYTES of a (128/EB elements).  One producer warp streams tiles HBM -> shared
// memory with `cp.async.bulk.tensor` (TMA, SWIZZLE_128B) into a ring of stages
// guarded by mbarriers; eight consumer warps read each tile column-wise, assemble
// 16-byte runs along b in registers and store them with 16-byte coalesced stores
// (each warp store fills whole 128-byte lines of dst).  CTAs are persistent.
// TB is 128 or 256 (a template parameter; the ring holds at most
// 192 KiB of tiles either way).
//
// Shared-memory column reads are made bank-conflict-free the way the TVM
// "permute_layout" page makes its warp permute conflict-free ("Algorithm", step
// 2): lanes that would hit the same bank visit their registers in an order
// XOR-rotated by a field of their lane index.  With the TMA 128-byte swizzle a
// 16-byte chunk c of row r sits at chunk c ^ (r & 7), so the 8 lane groups of a
// warp must read rows with 8 distinct (r & 7); group g reads its k-th row as
// (k ^ x_g), and the registers are put back in order with a conditional-swap
// network before the stores.  The host bank simulator (tl_bank_conflicts)
// reproduces these access patterns in the unit tests.
#include "tile_common.cuh"

namespace tl {
namespace {

using namespace dev;
using namespace tile;

// TB = tile height in rows of b (128 or 256); the consumers take a tile in 128-row
// blocks.  Taller tiles halve the TMA requests and barrier round trips per byte.
// CAST (TL_CAST_*): each element converted before its store (EB 4 -> 2 bytes, or
// 2 -> 4); DEB is the destination's element width.
template <int EB, int TB, int CAST = TL_CAST_NONE>
__global__ void __launch_bounds__(kTileThreads)
k_tile(const __grid_constant__ CUtensorMap tmap, const TileArgs a) {
    constexpr int DEB = CAST == TL_CAST_NONE ? EB
                        : (CAST == TL_CAST_F32_TO_BF16 || CAST == TL_CAST_F32_TO_F16) ? 2 : 4;
    constexpr uint32_t kBytes = (uint32_t)TB * kRowBytes;   // one stage
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kMaxTileStages];
    __shared__ __align__(8) uint64_t empty[kMaxTileStages];
    // destination of the tile in each stage, packed into one 16-byte word
    __shared__ __align__(16) uint4 info[kMaxTileStages];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t S = (uint32_t)a.stages;    // ring depth, 2 .. kMaxTileStages

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // everything above touched shared memory only
    grid_dependency_wait();
    allow_dependent_launch();
    cta_start(a.cta_times);

    if (warp == kConsumerWarps) {
        // ---------------- producer: one elected lane issues all TMA loads -------------
        if (lane == 0) {
            uint32_t issued = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < a.tiles; t += gridDim.x, ++issued) {
                const uint32_t use = issued / S;
                const uint32_t s = issued - use * S;
                if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                const TileCoord tc = tile_coord(t, a);
                // one 16-byte store, published by the release below
                sts128(smem_addr(&info[s]), pack_out<EB, TB, DEB>(tc, a));
                mbar_arrive_expect_tx(&full[s], kBytes);
                tma_load(smem + s * kBytes, &tmap, &full[s], a.rank,
                         (int)(tc.ta * kRowBytes), (int)(tc.tb * TB), (int)tc.bc[0],
                         (int)tc.bc[1], (int)tc.bc[2]);
            }
            if (!ok) report(a.status, TL_ERR_TIMEOUT);
            // Do not leave while a load may still write this CTA's shared memory (a
            // longer bound than the wait that expired; past it the CTA leaves anyway).
            for (uint32_t i = issued > S ? issued - S : 0; i < issued; ++i)
                mbar_wait(&full[i % S], (i / S) & 1, kDrainFactor * a.timeout_ns);
        }
        cta_finish(a.cta_times);
        return;
    }

    // ---------------- consumers -----------------------------------------------------
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < a.tiles; t += gridDim.x, ++it) {
        const uint32_t use = it / S;
        const uint32_t s = it - use * S;
        if (!mbar_wait(&full[s], use & 1, a.timeout_ns)) {
            if (lane == 0) report(a.status, TL_ERR_TIMEOUT);
            break;
        }
        const TileOut o = unpack_out<DEB>(lds128(smem_addr(&info[s])), a);
        const uint32_t base = smem_addr(smem + s * kBytes);
#pragma unroll
        for (int rb0 = 0; rb0 < TB; rb0 += kRows) {
            if (rb0 != 0 && rb0 >= o.rows) continue;
            if constexpr (CAST == TL_CAST_NONE) consume<EB>(base, o, warp, lane, rb0);
            else if constexpr (DEB == 2) consume_narrow<CAST>(base, o, warp, lane, rb0);
            else consume_widen<CAST>(base, o, warp, lane, rb0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    cta_finish(a.cta_times);
}

}  // namespace

int tile_smem_bytes(int stages, int rows) { return stages * rows * kRowBytes + 1024; }

template <int EB, int TB>
const void* tile_kernel() {
    return reinterpret_cast<const void*>(&k_tile<EB, TB>);
}

template <int EB, int TB>
cudaError_t launch_tile(const CUtensorMap& map, const TileArgs& a, int grid, cudaStream_t st,
                        bool pdl) {
    return launch_kernel(k_tile<EB, TB>, dim3(grid), dim3(kTileThreads),
                         tile_smem_bytes(a.stages, TB), st, pdl, map, a);
}

// the converting tile kernels (128-row tiles)
cudaError_t launch_tile_cast(int cast, const CUtensorMap& map, const TileArgs& a, int grid,
                             cudaStream_t st, bool pdl) {
    switch (cast) {
    case TL_CAST_F32_TO_BF16:
        return launch_kernel(k_tile<4, 128, TL_CAST_F32_TO_BF16>, dim3(grid), dim3(kTileThreads),
                             tile_smem_bytes(a.stages, 128), st, pdl, map, a);
    case TL_CAST_F32_TO_F16:
        return launch_kernel(k_tile<4, 128, TL_CAST_F32_TO_F16>, dim3(grid), dim3(kTileThreads),
                             tile_smem_bytes(a.stages, 128), st, pdl, map, a);
    case TL_CAST_BF16_TO_F32:
        return launch_kernel(k_tile<2, 128, TL_CAST_BF16_TO_F32>, dim3(grid), dim3(kTileThreads),
                             tile_smem_bytes(a.stages, 128), st, pdl, map, a);
    case TL_CAST_F16_TO_F32:
        return launch_kernel(k_tile<2, 128, TL_CAST_F16_TO_F32>, dim3(grid), dim3(kTileThreads),
                             tile_smem_bytes(a.stages, 128), st, pdl, map, a);
    }
    return cudaErrorInvalidValue;
}

const void* tile_cast_kernel(int cast) {
    switch (cast) {
    case TL_CAST_F32_TO_BF16: return reinterpret_cast<const void*>(&k_tile<4, 128, TL_CAST_F32_TO_BF16>);
    case TL_CAST_F32_TO_F16: return reinterpret_cast<const void*>(&k_tile<4, 128, TL_CAST_F32_TO_F16>);
    case TL_CAST_BF16_TO_F32: return reinterpret_cast<const void*>(&k_tile<2, 128, TL_CAST_BF16_TO_F32>);
    case TL_CAST_F16_TO_F32: return reinterpret_cast<const void*>(&k_tile<2, 128, TL_CAST_F16_TO_F32>);
    }
    return nullptr;
}

#define TL_INST(EB, TB)                                                                     \
    template const void* tile_kernel<EB, TB>();                                             \
    template cudaError_t launch_tile<EB, TB>(const CUtensorMap&, const TileArgs&, int,      \
                                             cudaStream_t, bool);
TL_INST(1, 128)
TL_INST(2, 128)
TL_INST(4, 128)
TL_INST(8, 128)
TL_INST(16, 128)
TL_INST(1, 256)
TL_INST(2, 256)
TL_INST(4, 256)
TL_INST(8, 256)
TL_INST(16, 256)
#undef TL_INST

}  // namespace tl
