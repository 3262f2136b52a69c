// k_cluster.cu -- the tile transpose split across a 2-CTA cluster, with every
// tile handed from one CTA's shared memory to the other's through distributed
// shared memory (the "copy_async -> dsmem" page of the TVM docs: the source CTA
// maps the destination's shared address and mbarrier into its own window with
// mapa and issues cp.async.bulk.shared::cluster; the bytes landing complete the
// destination CTA's mbarrier, which the destination armed with expect_tx).
//
// The pair is symmetric.  Each CTA runs four roles on its own tiles of the
// cluster's sequence (CTA r loads the tiles whose sequence index is r mod 2):
//   * a loader lane streams its tiles from HBM into a ring of staging slots (TMA);
//   * a pusher lane forwards each landed tile (16384 bytes, one contiguous
//     chunk) into the next receive slot of the peer CTA;
//   * a watcher lane arms this CTA's receive slots and, as soon as a push from the
//     peer has landed, hands the peer's staging slot back by arriving on the peer's
//     barrier through DSMEM: a DSMEM push completes only on the receiving CTA's
//     barrier (bulk async-groups do not track it), so the peer learns from this
//     arrive that its source was read;
//   * eight consumer warps transpose the tiles the PEER pushed into this CTA's
//     receive ring, store them to dst, and release each receive slot by arriving
//     on the peer's barrier.
// The staging and receive rings have their own depths: a staging slot is held for
// the HBM load and the push, a receive slot only from the push to the consumers.
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

// NCW consumer warps (8 or 4; four warps take two shares of the tile each, so
// twice as many CTAs fit on an SM), then the loader, pusher and watcher warps.
template <int EB, int NCW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(cluster_threads(NCW), NCW == 4 ? 4 : 2)
k_cluster(const __grid_constant__ CUtensorMap tmap, const TileArgs a) {
    constexpr int kLoaderWarp = NCW, kPusherWarp = NCW + 1, kWatchWarp = NCW + 2;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t loaded[kMaxClusterStages];  // TMA landed in staging slot
    __shared__ __align__(8) uint64_t staged[kMaxClusterStages];  // staging slot free: the PEER
                                                                 // received its push
    __shared__ __align__(8) uint64_t freed[kMaxClusterStages];   // the PEER's receive slot free
    __shared__ __align__(8) uint64_t recv[kMaxClusterStages];    // own receive slot, peer-filled
    const uint32_t SS = (uint32_t)a.stages;        // staging ring depth (runtime)
    const uint32_t SR = (uint32_t)a.recv_stages;   // receive ring depth (runtime)
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* staging = smem;                       // SS tiles
    uint8_t* receive = smem + SS * kTileBytes;     // SR tiles
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    const int64_t cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const bool drop = a.drop_handoff != 0;   // test hook: the hand-off is skipped
    // tiles of this cluster: t_k = cluster + k * nclusters; CTA r loads k = 2j + r
    // and consumes k = 2j + peer.  The n-th tile a CTA loads is the n-th tile its
    // peer receives: staging slot n % SS on one side, receive slot n % SR on the other.
    const int64_t step2 = 2 * nclusters;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < SS; ++s) {
            mbar_init(&loaded[s], 1);
            mbar_init(&staged[s], 1);
        }
        for (uint32_t s = 0; s < SR; ++s) {
            mbar_init(&freed[s], NCW);
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
            const uint32_t use = issued / SS;
            const uint32_t s = issued - use * SS;
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
        for (uint32_t i = issued > SS ? issued - SS : 0; i < issued; ++i)
            mbar_wait(&loaded[i % SS], (i / SS) & 1, kDrainFactor * a.timeout_ns);
    } else if (warp == kPusherWarp && lane == 0) {
        // ---------------------------------- pusher ----------------------------------
        uint32_t n = 0;
        bool ok = true;
        for (int64_t t = cluster + rank * nclusters; t < a.tiles; t += step2, ++n) {
            const uint32_t s = n % SS, r = n % SR;
            if (!mbar_wait(&loaded[s], (n / SS) & 1, a.timeout_ns)) { ok = false; break; }
            if (n >= SR && !mbar_wait_cluster(&freed[r], ((n / SR) - 1) & 1, a.timeout_ns)) {
                ok = false;
                break;
            }
            if (!drop) {
                // the whole 16 KiB tile is one contiguous chunk
                tl_dev::ChunkLoop one{};
                one.chunk_bytes = kTileBytes;
                tl_dev::dsmem_copy_region(receive + r * kTileBytes, staging + s * kTileBytes,
                                          one, peer, &recv[r]);
            }
            // A DSMEM push completes only on the peer's barrier, so the staging slot
            // is released by the peer once the bytes have landed there.
        }
        if (!ok) report(a.status, TL_ERR_TIMEOUT);
    } else if (warp == kWatchWarp && lane == 0) {
        // ---------------------------------- watcher ---------------------------------
        // Arms each receive slot and, the moment the peer's push has landed, hands
        // the peer's staging slot back, so the peer's next load never waits for this
        // CTA's consumers.
        uint32_t it = 0;
        for (int64_t t = cluster + peer * nclusters; t < a.tiles; t += step2, ++it) {
            const uint32_t r = it % SR;
            mbar_arrive_expect_tx(&recv[r], kTileBytes);
            if (!mbar_wait_cluster(&recv[r], (it / SR) & 1, a.timeout_ns)) {
                report(a.status, TL_ERR_TIMEOUT);
                break;
            }
            // CTA-scope release: the push's reads of the peer's slot are complete
            // (they completed this barrier, which the acquire above observed), and a
            // cluster-scope release here cost ~2 us per tile before the peer's loader
            // saw the arrive (per-tile timestamp trace on GB300)
            mbar_arrive_remote_slot(map_to_rank(smem_addr(&staged[it % SS]), peer));
        }
    } else if (warp < NCW) {
        // --------------------------------- consumers --------------------------------
        uint32_t it = 0;
        for (int64_t t = cluster + peer * nclusters; t < a.tiles; t += step2, ++it) {
            const uint32_t r = it % SR;
            const TileOut o = make_out<EB>(tile_coord(t, a), a);   // while the tile flies
            if (!mbar_wait_cluster(&recv[r], (it / SR) & 1, a.timeout_ns)) {
                if (lane == 0) report(a.status, TL_ERR_TIMEOUT);
                break;
            }
#pragma unroll
            for (int v = warp; v < kConsumerWarps; v += NCW)
                consume<EB>(smem_addr(receive + r * kTileBytes), o, v, lane, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive_remote_slot(map_to_rank(smem_addr(&freed[r]), peer));
        }
    }
    __syncwarp();
    // Neither CTA leaves while its peer may still touch its shared memory.
    cluster_sync_all();
}

template <int EB>
cudaError_t go(const CUtensorMap& map, const TileArgs& a, int ncw, int grid, cudaStream_t st,
               bool pdl) {
    const int smem = cluster_smem_bytes(a.stages + a.recv_stages);
    if (ncw == 4)
        return launch_kernel(k_cluster<EB, 4>, dim3(grid), dim3(cluster_threads(4)), smem, st,
                             pdl, map, a);
    return launch_kernel(k_cluster<EB, 8>, dim3(grid), dim3(cluster_threads(8)), smem, st, pdl,
                         map, a);
}

template <int NCW>
const void* kernel_of(int eb) {
    switch (eb) {
    case 1: return reinterpret_cast<const void*>(&k_cluster<1, NCW>);
    case 2: return reinterpret_cast<const void*>(&k_cluster<2, NCW>);
    case 4: return reinterpret_cast<const void*>(&k_cluster<4, NCW>);
    case 8: return reinterpret_cast<const void*>(&k_cluster<8, NCW>);
    default: return reinterpret_cast<const void*>(&k_cluster<16, NCW>);
    }
}

}  // namespace

int cluster_smem_bytes(int slots) { return slots * kTileBytes + 1024; }

const void* cluster_kernel(int eb, int ncw) {
    return ncw == 4 ? kernel_of<4>(eb) : kernel_of<8>(eb);
}

cudaError_t launch_cluster(int eb, int ncw, const CUtensorMap& map, const TileArgs& a, int grid,
                           cudaStream_t st, bool pdl) {
    switch (eb) {
    case 1: return go<1>(map, a, ncw, grid, st, pdl);
    case 2: return go<2>(map, a, ncw, grid, st, pdl);
    case 4: return go<4>(map, a, ncw, grid, st, pdl);
    case 8: return go<8>(map, a, ncw, grid, st, pdl);
    default: return go<16>(map, a, ncw, grid, st, pdl);
    }
}

}  // namespace tl
