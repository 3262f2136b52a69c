// device_primitives.cu -- test kernels for include/tl_permute_device.cuh.
//
// TEST INFRASTRUCTURE: built by tests/test_gpu_device_primitives.py into its own
// shared library; the product never loads it.  Each extern "C" launcher takes
// device pointers and plain sizes and returns a cudaError_t (0 = launched).
#include <cuda_runtime.h>

#include <cstdint>

#include "tl_permute_device.cuh"

// Argument blocks shared with the Python side (ctypes structures of the same layout).
namespace tdp {
struct TileArgs {
    int32_t n;
    int32_t ext[4];
    int64_t src_str[4];
    int64_t dst_str[4];
    int32_t shift, mask;
    int32_t in_place;
    int32_t items;
};

struct RegionArgs {
    tl_dev::ChunkLoop loop;
    int32_t src_bytes;   // bytes of the source image CTA 0 stages in shared memory
    int32_t dst_bytes;   // bytes of the destination image CTA 1 holds (and writes back)
    int32_t src_off;     // byte offset of the region in the source image
    int32_t dst_off;     // byte offset of the region in the destination image
    uint64_t timeout_ns;
};
}  // namespace tdp
using tdp::RegionArgs;
using tdp::TileArgs;

namespace {

template <int EB> struct Raw;
template <> struct Raw<1> { using T = uint8_t; };
template <> struct Raw<2> { using T = uint16_t; };
template <> struct Raw<4> { using T = uint32_t; };
template <> struct Raw<8> { using T = uint2; };
template <> struct Raw<16> { using T = uint4; };


tl_dev::WarpTile make_tile(const TileArgs& a, const int64_t* str) {
    tl_dev::WarpTile t;
    t.n = a.n;
    for (int i = 0; i < 4; ++i) {
        t.ext[i] = i < a.n ? a.ext[i] : 1;
        t.str[i] = i < a.n ? str[i] : 0;
    }
    return t;
}

// One warp per item: the item's 32*P elements go global -> shared, are permuted
// in shared memory (in place or into a second buffer), and go back to global.
template <int EB, int P>
__global__ void k_warp_smem(const uint8_t* src, uint8_t* dst, TileArgs a, tl_dev::WarpTile ts,
                            tl_dev::WarpTile td) {
    using T = typename Raw<EB>::T;
    constexpr int N = 32 * P;
    __shared__ T bufA[N];
    __shared__ T bufB[N];
    const int lane = threadIdx.x;
    const T* s = reinterpret_cast<const T*>(src) + (int64_t)blockIdx.x * N;
    T* d = reinterpret_cast<T*>(dst) + (int64_t)blockIdx.x * N;
    for (int i = lane; i < N; i += 32) bufA[i] = s[i];
    __syncwarp();
    T* out = a.in_place ? bufA : bufB;
    tl_dev::warp_permute_layout<P>(out, bufA, ts, td, a.shift, a.mask);
    for (int i = lane; i < N; i += 32) d[i] = out[i];
}

// Fragment round trip: rotated load from global, unrotate, lane-major store:
// dst[lane + 32*j] = tile element j of this lane.
template <int EB, int P>
__global__ void k_fragment(const uint8_t* src, uint8_t* dst, TileArgs a, tl_dev::WarpTile ts) {
    using T = typename Raw<EB>::T;
    T regs[P];
    tl_dev::warp_load_fragment<P>(regs, reinterpret_cast<const T*>(src), ts, a.shift, a.mask);
    tl_dev::warp_fragment_unrotate<P>(regs, a.shift, a.mask);
    T* d = reinterpret_cast<T*>(dst);
    const int lane = tl_dev::lane_id();
#pragma unroll
    for (int j = 0; j < P; ++j) d[lane + 32 * j] = regs[j];
}

template <int EB, int P>
cudaError_t go_warp(const void* src, void* dst, const TileArgs& a) {
    const tl_dev::WarpTile ts = make_tile(a, a.src_str), td = make_tile(a, a.dst_str);
    k_warp_smem<EB, P><<<a.items, 32>>>(static_cast<const uint8_t*>(src),
                                        static_cast<uint8_t*>(dst), a, ts, td);
    return cudaGetLastError();
}

template <int EB, int P>
cudaError_t go_frag(const void* src, void* dst, const TileArgs& a) {
    k_fragment<EB, P><<<1, 32>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), a,
                                 make_tile(a, a.src_str));
    return cudaGetLastError();
}

#define TDP_DISPATCH(FN)                                                       \
    switch (eb * 100 + P) {                                                    \
    case 101: return FN<1, 1>(src, dst, a);                                    \
    case 104: return FN<1, 4>(src, dst, a);                                    \
    case 108: return FN<1, 8>(src, dst, a);                                    \
    case 202: return FN<2, 2>(src, dst, a);                                    \
    case 204: return FN<2, 4>(src, dst, a);                                    \
    case 208: return FN<2, 8>(src, dst, a);                                    \
    case 401: return FN<4, 1>(src, dst, a);                                    \
    case 402: return FN<4, 2>(src, dst, a);                                    \
    case 404: return FN<4, 4>(src, dst, a);                                    \
    case 408: return FN<4, 8>(src, dst, a);                                    \
    case 416: return FN<4, 16>(src, dst, a);                                   \
    case 116: return FN<1, 16>(src, dst, a);                                   \
    case 216: return FN<2, 16>(src, dst, a);                                   \
    case 802: return FN<8, 2>(src, dst, a);                                    \
    case 804: return FN<8, 4>(src, dst, a);                                    \
    case 808: return FN<8, 8>(src, dst, a);                                    \
    case 1608: return FN<16, 8>(src, dst, a);                                  \
    case 1602: return FN<16, 2>(src, dst, a);                                  \
    case 1604: return FN<16, 4>(src, dst, a);                                  \
    }                                                                          \
    return cudaErrorInvalidValue;

}  // namespace

extern "C" int tdp_warp_smem(const void* src, void* dst, int eb, int P, const TileArgs* args) {
    const TileArgs a = *args;
    TDP_DISPATCH(go_warp)
}

extern "C" int tdp_fragment(const void* src, void* dst, int eb, int P, const TileArgs* args) {
    const TileArgs a = *args;
    TDP_DISPATCH(go_frag)
}

// ---------------------------------------------------------------------------
// Thread-axis layouts: one warp loads its registers through layout L from `src`
// and writes them out lane-major (regs[j] of lane l to frag[l * P + j]); a second
// launch reads them back from `frag` and stores them through L into `dst`.
namespace {
template <int EB, int P>
__global__ void k_lanes_load(const uint8_t* src, uint8_t* frag, tl_dev::ThreadAxisLayout t) {
    using T = typename Raw<EB>::T;
    T regs[P];
    tl_dev::warp_load_lanes<P>(regs, reinterpret_cast<const T*>(src), t);
    T* f = reinterpret_cast<T*>(frag) + tl_dev::lane_id() * P;
#pragma unroll
    for (int j = 0; j < P; ++j) f[j] = regs[j];
}

template <int EB, int P>
__global__ void k_lanes_store(const uint8_t* frag, uint8_t* dst, tl_dev::ThreadAxisLayout t) {
    using T = typename Raw<EB>::T;
    T regs[P];
    const T* f = reinterpret_cast<const T*>(frag) + tl_dev::lane_id() * P;
#pragma unroll
    for (int j = 0; j < P; ++j) regs[j] = f[j];
    tl_dev::warp_store_lanes<P>(regs, reinterpret_cast<T*>(dst), t);
}

template <int EB, int P>
cudaError_t go_lanes(const void* src, void* frag, void* dst, const tl_dev::ThreadAxisLayout& t) {
    k_lanes_load<EB, P><<<1, 32>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(frag), t);
    k_lanes_store<EB, P><<<1, 32>>>(static_cast<const uint8_t*>(frag), static_cast<uint8_t*>(dst), t);
    return cudaGetLastError();
}
}  // namespace

extern "C" int tdp_lanes(const void* src, void* frag, void* dst, int eb, int P,
                         const tl_dev::ThreadAxisLayout* layout) {
    const tl_dev::ThreadAxisLayout t = *layout;
    switch (eb * 100 + P) {
    case 101: return go_lanes<1, 1>(src, frag, dst, t);
    case 102: return go_lanes<1, 2>(src, frag, dst, t);
    case 108: return go_lanes<1, 8>(src, frag, dst, t);
    case 202: return go_lanes<2, 2>(src, frag, dst, t);
    case 208: return go_lanes<2, 8>(src, frag, dst, t);
    case 401: return go_lanes<4, 1>(src, frag, dst, t);
    case 402: return go_lanes<4, 2>(src, frag, dst, t);
    case 404: return go_lanes<4, 4>(src, frag, dst, t);
    case 408: return go_lanes<4, 8>(src, frag, dst, t);
    case 416: return go_lanes<4, 16>(src, frag, dst, t);
    case 804: return go_lanes<8, 4>(src, frag, dst, t);
    case 808: return go_lanes<8, 8>(src, frag, dst, t);
    case 1602: return go_lanes<16, 2>(src, frag, dst, t);
    }
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// DSMEM region copy between the two CTAs of a cluster
// ---------------------------------------------------------------------------
namespace {


__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = tl_dev::smem_u32(bar);
    const uint64_t t0 = tl_dev::global_timer_ns();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if (tl_dev::global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// CTA 0 stages the source image, copies the region into CTA 1's destination
// image through DSMEM; CTA 1 waits on its mbarrier and writes its image back.
// status[0]: 1 copied, 2 declined by the chunk rule; status[1]: 1 CTA 1 saw the
// bytes land, 0 its bounded wait expired.
__global__ void __cluster_dims__(2, 1, 1) k_dsmem(const uint8_t* src, uint8_t* dst,
                                                   int32_t* status, RegionArgs a) {
    extern __shared__ __align__(128) uint8_t image[];
    __shared__ __align__(8) uint64_t bar;
    const uint32_t rank = cluster_rank();
    const uint32_t total = tl_dev::chunk_loop_bytes(a.loop);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tl_dev::smem_u32(&bar))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const uint8_t* from = rank == 0 ? src : dst;          // CTA 1 starts from dst's canaries
    const int nbytes = rank == 0 ? a.src_bytes : a.dst_bytes;
    for (int i = threadIdx.x; i < nbytes; i += blockDim.x) image[i] = from[i];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    cluster_sync();
    if (rank == 1 && threadIdx.x == 0)
        asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                         tl_dev::smem_u32(&bar)),
                     "r"(total)
                     : "memory");
    if (rank == 0 && threadIdx.x == 0) {
        const bool ok = tl_dev::dsmem_copy_region(image + a.dst_off, image + a.src_off, a.loop, 1,
                                                  &bar);
        status[0] = ok ? 1 : 2;
    }
    if (rank == 1) {
        const bool landed = wait_bar(&bar, 0, a.timeout_ns);
        if (threadIdx.x == 0) status[1] = landed ? 1 : 0;
        __syncthreads();
        for (int i = threadIdx.x; i < a.dst_bytes; i += blockDim.x) dst[i] = image[i];
    }
    cluster_sync();   // CTA 0 stays until CTA 1 is done with the copy it issued
}

// ---------------------------------------------------------------------------
// wait_until_global between two co-resident blocks (cooperative launch)
// ---------------------------------------------------------------------------
__global__ void k_wait(uint32_t* flag, uint32_t* data, uint32_t* out, int32_t* status, int n,
                       int publish, uint64_t timeout_ns) {
    if (blockIdx.x == 0) {
        if (!publish) return;
        for (int i = threadIdx.x; i < n; i += blockDim.x) data[i] = 2654435761u * i + 12345u;
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint64_t t0 = tl_dev::global_timer_ns();
            while (tl_dev::global_timer_ns() - t0 < 200000) {}   // let the waiter spin ~0.2 ms
            tl_dev::st_release_gpu(flag, 7u);
        }
        return;
    }
    __shared__ int ok;
    if (threadIdx.x == 0) {
        uint32_t v = 0;
        ok = tl_dev::wait_until_global(flag, [](uint32_t x) { return x >= 1u; }, timeout_ns, &v)
                 ? 1 : 0;
        status[0] = ok;
        status[1] = (int32_t)v;
    }
    __syncthreads();
    if (ok)
        for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = data[i];
}

// The same protocol on a 64-bit word: relaxed polls at system scope with a 100 ns
// backoff between them, the publisher releasing 2^40 + 7 (so that only a 64-bit
// read sees the value its predicate wants).
__global__ void k_wait64(uint64_t* flag, uint32_t* data, uint32_t* out, int32_t* status, int n,
                         int publish, uint64_t timeout_ns) {
    if (blockIdx.x == 0) {
        if (!publish) return;
        for (int i = threadIdx.x; i < n; i += blockDim.x) data[i] = 2246822519u * i + 7u;
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint64_t t0 = tl_dev::global_timer_ns();
            while (tl_dev::global_timer_ns() - t0 < 200000) {}
            tl_dev::st_release_gpu(flag, (1ull << 40) + 7ull);
        }
        return;
    }
    __shared__ int ok;
    if (threadIdx.x == 0) {
        uint64_t v = 0;
        ok = tl_dev::wait_until_global<tl_dev::WaitScope::sys>(
                 flag, [](uint64_t x) { return x > (1ull << 32); }, timeout_ns, &v, 100u)
                 ? 1 : 0;
        status[0] = ok;
        status[1] = (int32_t)(v >> 32);
        status[2] = (int32_t)(v & 0xffffffffu);
    }
    __syncthreads();
    if (ok)
        for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = data[i];
}

}  // namespace

extern "C" int tdp_wait64(uint64_t* flag, uint32_t* data, uint32_t* out, int32_t* status, int n,
                          int publish, uint64_t timeout_ns) {
    void* args[] = {&flag, &data, &out, &status, &n, &publish, &timeout_ns};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&k_wait64), dim3(2),
                                       dim3(128), args, 0, 0);
}

extern "C" int tdp_dsmem(const void* src, void* dst, int32_t* status, const RegionArgs* args) {
    const RegionArgs a = *args;
    const int smem = a.src_bytes > a.dst_bytes ? a.src_bytes : a.dst_bytes;
    if (smem > 48 * 1024) return cudaErrorInvalidValue;
    k_dsmem<<<2, 128, smem>>>(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                              status, a);
    return cudaGetLastError();
}

extern "C" int tdp_wait(uint32_t* flag, uint32_t* data, uint32_t* out, int32_t* status, int n,
                        int publish, uint64_t timeout_ns) {
    void* args[] = {&flag, &data, &out, &status, &n, &publish, &timeout_ns};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&k_wait), dim3(2), dim3(128),
                                       args, 0, 0);
}

// ---------------------------------------------------------------------------
// DSMEM ceiling: the cluster hand-off pattern with no HBM traffic
// ---------------------------------------------------------------------------
namespace {

// Each CTA of a pair pushes `iters` 16 KiB tiles into the peer's 2-slot receive
// ring (one bulk copy each, completing on the peer's barrier); the peer releases
// each slot back with a remote arrive.  status[blockIdx.x] = 1 done, 0 a bounded
// wait expired.
__global__ void __cluster_dims__(2, 1, 1) k_dsmem_stream(int iters, uint64_t timeout_ns,
                                                          int32_t* status) {
    constexpr int S = 2;
    constexpr uint32_t kTile = 16384;
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ __align__(8) uint64_t recv[S], freed[S];
    uint8_t* staging = sm;
    uint8_t* receive = sm + S * kTile;
    const uint32_t rank = cluster_rank(), peer = rank ^ 1u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tl_dev::smem_u32(&recv[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tl_dev::smem_u32(&freed[s])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_sync();
    bool ok = true;
    if (threadIdx.x == 0) {                          // pusher
        tl_dev::ChunkLoop one{};
        one.chunk_bytes = kTile;
        for (int i = 0; i < iters && ok; ++i) {
            const int s = i % S;
            if (i >= S) ok = wait_bar(&freed[s], ((i / S) - 1) & 1, timeout_ns);
            if (ok) tl_dev::dsmem_copy_region(receive + s * kTile, staging + s * kTile, one, peer,
                                              &recv[s]);
        }
    } else if (threadIdx.x == 32) {                  // receiver
        for (int i = 0; i < iters && ok; ++i) {
            const int s = i % S;
            asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                             tl_dev::smem_u32(&recv[s])),
                         "r"(kTile)
                         : "memory");
            ok = wait_bar(&recv[s], (i / S) & 1, timeout_ns);
            if (ok) {
                uint32_t remote;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                             : "=r"(remote)
                             : "r"(tl_dev::smem_u32(&freed[s])), "r"(peer));
                asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                                 remote)
                             : "memory");
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 || threadIdx.x == 32) atomicAnd(&status[blockIdx.x], ok ? 1 : 0);
    cluster_sync();
}

}  // namespace

extern "C" int tdp_dsmem_stream(int grid, int iters, uint64_t timeout_ns, int32_t* status) {
    const int smem = 4 * 16384;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_dsmem_stream),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_dsmem_stream<<<grid, 64, smem>>>(iters, timeout_ns, status);
    return cudaGetLastError();
}
