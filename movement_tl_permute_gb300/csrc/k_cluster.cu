// k_cluster.cu -- the tile transpose split across a 2-CTA cluster, with every
// tile handed from one CTA's shared memory to the other's through distributed
// shared memory (the "copy_async -> dsmem" page of the TVM docs: the source CTA
// maps the destination's shared address and mbarrier into its own window with
// mapa and issues cp.async.bulk.shared::cluster; the bytes landing complete the
// destination CTA's mbarrier, which the destination armed with expect_tx).
//
// The pair is symmetric.  Each CTA runs three roles on its own tiles of the
// cluster's sequence (CTA r loads the tiles whose sequence index is r mod 2):
//   * a loader lane streams its tiles from HBM into a ring of staging slots (TMA);
//   * a pusher lane forwards each landed tile (16384 bytes, one contiguous
//     chunk) into the matching receive slot of the peer CTA;
//   * eight consumer warps transpose the tiles the PEER pushed into this CTA's
//     receive ring, store them to dst, and release each receive slot by arriving
//     on the peer's barrier through DSMEM.  As soon as a tile has landed they also
//     hand the peer's staging slot back: a DSMEM push completes only on the
//     receiving CTA's barrier (bulk async-groups do not track it), so the peer
//     learns that its source was read from this arrive.
// So every SM both reads and writes HBM, and every tile crosses the SM-to-SM
// network once.  The hand-off is a point-to-point bulk copy, not a multicast.
// Every wait is bounded; an expired wait records TL_ERR_TIMEOUT in the status
// word and the CTA drains its own in-flight copies before leaving.
#include "tile_common.cuh"
#include "../../include/tl_permute_device.cuh"

namespace tl {
namespace {

using namespace dev;
using namespace tile;

constexpr int kLoaderWarp = kConsumerWarps;        // warp 8
constexpr int kPusherWarp = kConsumerWarps + 1;    // warp 9

template <int EB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kClusterThreads)
k_cluster(const __grid_constant__ CUtensorMap tmap, const TileArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t loaded[kMaxClusterStages];  // TMA landed in staging slot
    __shared__ __align__(8) uint64_t staged[kMaxClusterStages];  // staging slot free: the PEER
                                                                 // received its push
    __shared__ __align__(8) uint64_t freed[kMaxClusterStages];   // the PEER's receive slot free
    __shared__ __align__(8) uint64_t recv[kMaxClusterStages];    // own receive slot, peer-filled
    const int kStages = a.stages;                                // ring depth (runtime)
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem;                            // kStages tiles
    uint8_t* receive = smem + kStages * kTileBytes;     // kStages tiles
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int64_t cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const bool drop = a.drop_handoff != 0;   // test hook: the hand-off is skipped
    // tiles of this cluster: t_k = cluster + k * nclusters; CTA r loads k = 2j + r
    // and consumes k = 2j + peer.
    const int64_t step2 = 2 * nclusters;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&loaded[s], 1);
            mbar_init(&staged[s], 1);
            mbar_init(&freed[s], kConsumerWarps);
            mbar_init(&recv[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers exist before any remote access
    grid_dependency_wait();
    allow_dependent_launch();

    if (warp == kLoaderWarp && lane == 0) {
        // ---------------------------------- loader ----------------------------------
        uint32_t issued = 0;
        bool ok = true;
        for (int64_t t = cluster + rank * nclusters; t < a.tiles; t += step2, ++issued) {
            const int s = issued % kStages;
            const uint32_t use = issued / kStages;
            if (use > 0 && !mbar_wait_cluster(&staged[s], (use - 1) & 1, a.timeout_ns)) {
                ok = false;
                break;
            }
            const TileCoord tc = tile_coord(t, a);
            mbar_arrive_expect_tx(&loaded[s], kTileBytes);
            tma_load(staging + s * kTileBytes, &tmap, &loaded[s], a.rank,
                     (int)(tc.ta * kRowBytes), (int)(tc.tb * kRows), (int)tc.bc[0],
                     (int)tc.bc[1], (int)tc.bc[2]);
        }
        if (!ok) report(a.status, TL_ERR_TIMEOUT);
        for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
            mbar_wait(&loaded[i % kStages], (i / kStages) & 1, a.timeout_ns);
    } else if (warp == kPusherWarp && lane == 0) {
        // ---------------------------------- pusher ----------------------------------
        uint32_t n = 0;
        bool ok = true;
        for (int64_t t = cluster + rank * nclusters; t < a.tiles; t += step2, ++n) {
            const int s = n % kStages;
            const uint32_t use = n / kStages;
            if (!mbar_wait(&loaded[s], use & 1, a.timeout_ns)) { ok = false; break; }
            if (use > 0 && !mbar_wait_cluster(&freed[s], (use - 1) & 1, a.timeout_ns)) {
                ok = false;
                break;
            }
            if (!drop) {
                // the whole 16 KiB tile is one contiguous chunk
                tl_dev::ChunkLoop one{};
                one.chunk_bytes = kTileBytes;
                tl_dev::dsmem_copy_region(receive + s * kTileBytes, staging + s * kTileBytes,
                                          one, peer, &recv[s]);
            }
            // A DSMEM push completes only on the peer's barrier, so the staging slot
            // is released by the peer once the bytes have landed there.
        }
        if (!ok) report(a.status, TL_ERR_TIMEOUT);
    } else if (warp < kConsumerWarps) {
        // --------------------------------- consumers --------------------------------
        uint32_t it = 0;
        for (int64_t t = cluster + peer * nclusters; t < a.tiles; t += step2, ++it) {
            const int s = it % kStages;
            if (threadIdx.x == 0) mbar_arrive_expect_tx(&recv[s], kTileBytes);
            if (!mbar_wait_cluster(&recv[s], (it / kStages) & 1, a.timeout_ns)) {
                if (lane == 0) report(a.status, TL_ERR_TIMEOUT);
                break;
            }
            // the bytes have landed, so the peer's push has finished reading its
            // staging slot: hand that slot back to the peer's loader
            if (threadIdx.x == 0) mbar_arrive_remote(map_to_rank(smem_addr(&staged[s]), peer));
            const TileOut o = make_out<EB>(tile_coord(t, a), a);
            consume<EB>(smem_addr(receive + s * kTileBytes), o, warp, lane, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(map_to_rank(smem_addr(&freed[s]), peer));
        }
    }
    __syncwarp();
    // Neither CTA leaves while its peer may still touch its shared memory.
    cluster_sync_all();
}

template <int EB>
cudaError_t go(const CUtensorMap& map, const TileArgs& a, int grid, cudaStream_t st, bool pdl) {
    return launch_kernel(k_cluster<EB>, dim3(grid), dim3(kClusterThreads),
                         cluster_smem_bytes(a.stages), st, pdl, map, a);
}

}  // namespace

int cluster_smem_bytes(int stages) { return 2 * stages * kTileBytes + 1024; }

const void* cluster_kernel(int eb) {
    switch (eb) {
    case 1: return reinterpret_cast<const void*>(&k_cluster<1>);
    case 2: return reinterpret_cast<const void*>(&k_cluster<2>);
    case 4: return reinterpret_cast<const void*>(&k_cluster<4>);
    case 8: return reinterpret_cast<const void*>(&k_cluster<8>);
    default: return reinterpret_cast<const void*>(&k_cluster<16>);
    }
}

cudaError_t launch_cluster(int eb, const CUtensorMap& map, const TileArgs& a, int grid,
                           cudaStream_t st, bool pdl) {
    switch (eb) {
    case 1: return go<1>(map, a, grid, st, pdl);
    case 2: return go<2>(map, a, grid, st, pdl);
    case 4: return go<4>(map, a, grid, st, pdl);
    case 8: return go<8>(map, a, grid, st, pdl);
    default: return go<16>(map, a, grid, st, pdl);
    }
}

}  // namespace tl
