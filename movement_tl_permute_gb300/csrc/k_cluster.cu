// k_cluster.cu -- the tile transpose split across a 2-CTA cluster, with the tile
// handed from one CTA's shared memory to the other's through distributed shared
// memory (the "copy_async -> dsmem" page of the TVM docs: the source CTA maps
// the destination's shared address and mbarrier into its own window with mapa
// and issues cp.async.bulk.shared::cluster; the bytes landing complete the
// destination CTA's mbarrier, which the destination armed with expect_tx).
//
// Rank 0 of each cluster is the producer: a loader lane streams tiles from HBM
// into a ring of staging slots with TMA, and a pusher lane forwards each landed
// tile (16384 bytes, one contiguous chunk) into the matching receive slot of rank
// 1.  Rank 1 is the consumer: its eight warps transpose the received tile and
// store it to dst exactly as the single-CTA tile kernel does, then release the
// receive slot by arriving on rank 0's barrier through DSMEM.  The hand-off is a
// plain point-to-point bulk copy, not a multicast.  Every wait is bounded; an
// expired wait records TL_ERR_TIMEOUT in the status word and the CTA drains its
// own in-flight copies before leaving.
#include "tile_common.cuh"

namespace tl {
namespace {

using namespace dev;
using namespace tile;

constexpr int kStages = kTileStages;

template <int EB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTileThreads)
k_cluster(const __grid_constant__ CUtensorMap tmap, const TileArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t loaded[kStages];   // rank 0: TMA landed in staging slot
    __shared__ __align__(8) uint64_t staged[kStages];   // rank 0: staging slot free again
    __shared__ __align__(8) uint64_t freed[kStages];    // rank 0: rank 1's receive slot free
    __shared__ __align__(8) uint64_t recv[kStages];     // rank 1: tile landed in receive slot
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int64_t cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const bool drop = a.pad != 0;   // test hook: the hand-off is skipped

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

    if (rank == 0) {
        if (warp == kConsumerWarps && lane == 0) {
            // ------------------------------ loader ------------------------------
            uint32_t issued = 0;
            bool ok = true;
            for (int64_t t = cluster; t < a.tiles; t += nclusters, ++issued) {
                const int s = issued % kStages;
                const uint32_t use = issued / kStages;
                if (use > 0 && !mbar_wait(&staged[s], (use - 1) & 1, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                const TileCoord tc = tile_coord(t, a);
                mbar_arrive_expect_tx(&loaded[s], kTileBytes);
                tma_load(smem + s * kTileBytes, &tmap, &loaded[s], a.rank,
                         (int)(tc.ta * kRowBytes), (int)(tc.tb * kRows), (int)tc.bc[0],
                         (int)tc.bc[1], (int)tc.bc[2]);
            }
            if (!ok) report(a.status, TL_ERR_TIMEOUT);
            for (uint32_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait(&loaded[i % kStages], (i / kStages) & 1, a.timeout_ns);
        } else if (warp == kConsumerWarps - 1 && lane == 0) {
            // ------------------------------ pusher ------------------------------
            uint32_t n = 0;
            bool ok = true;
            for (int64_t t = cluster; t < a.tiles; t += nclusters, ++n) {
                const int s = n % kStages;
                const uint32_t use = n / kStages;
                if (!mbar_wait(&loaded[s], use & 1, a.timeout_ns)) { ok = false; break; }
                if (use > 0 && !mbar_wait_cluster(&freed[s], (use - 1) & 1, a.timeout_ns)) {
                    ok = false;
                    break;
                }
                if (!drop) {
                    const uint32_t dst = map_to_rank(smem_addr(smem + s * kTileBytes), 1);
                    const uint32_t bar = map_to_rank(smem_addr(&recv[s]), 1);
                    bulk_copy_to_peer(dst, smem_addr(smem + s * kTileBytes), kTileBytes, bar);
                }
                bulk_commit();
                // the previous push has finished reading its staging slot
                bulk_wait_read<1>();
                if (n > 0) mbar_arrive(&staged[(n - 1) % kStages]);
            }
            bulk_wait_read<0>();
            if (n > 0) mbar_arrive(&staged[(n - 1) % kStages]);
            if (!ok) report(a.status, TL_ERR_TIMEOUT);
        }
    } else if (warp < kConsumerWarps) {
        // ------------------------------ consumer ------------------------------
        uint32_t it = 0;
        for (int64_t t = cluster; t < a.tiles; t += nclusters, ++it) {
            const int s = it % kStages;
            if (threadIdx.x == 0) mbar_arrive_expect_tx(&recv[s], kTileBytes);
            if (!mbar_wait_cluster(&recv[s], (it / kStages) & 1, a.timeout_ns)) {
                if (lane == 0) report(a.status, TL_ERR_TIMEOUT);
                break;
            }
            const TileOut o = make_out<EB>(tile_coord(t, a), a);
            consume<EB>(smem_addr(smem + s * kTileBytes), o, warp, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(map_to_rank(smem_addr(&freed[s]), 0));
        }
    }
    __syncwarp();
    // Neither CTA leaves while its peer may still touch its shared memory.
    cluster_sync_all();
}

template <int EB>
cudaError_t go(const CUtensorMap& map, const TileArgs& a, int grid, cudaStream_t st) {
    k_cluster<EB><<<grid, kTileThreads, cluster_smem_bytes(), st>>>(map, a);
    return cudaGetLastError();
}

}  // namespace

int cluster_smem_bytes() { return kStages * kTileBytes + 1024; }

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
                           cudaStream_t st) {
    switch (eb) {
    case 1: return go<1>(map, a, grid, st);
    case 2: return go<2>(map, a, grid, st);
    case 4: return go<4>(map, a, grid, st);
    case 8: return go<8>(map, a, grid, st);
    default: return go<16>(map, a, grid, st);
    }
}

}  // namespace tl
