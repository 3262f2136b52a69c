// tl_device.cuh -- device helpers shared by the permute kernels: raw-bit element
// types, 32-bit division by invariant integers, and inline PTX for mbarriers, TMA
// and the global timer.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "../../include/tl_permute.h"

namespace tl {
namespace dev {

// ---------------------------------------------------------------------------
// Raw-bit element of EB bytes (moved, never converted).
// ---------------------------------------------------------------------------
template <int EB> struct Bits;
template <> struct Bits<1> { using T = uint8_t; };
template <> struct Bits<2> { using T = uint16_t; };
template <> struct Bits<4> { using T = uint32_t; };
template <> struct Bits<8> { using T = uint2; };
template <> struct Bits<16> { using T = uint4; };

template <int EB>
__device__ __forceinline__ void copy_elem(uint8_t* d, const uint8_t* s) {
    using T = typename Bits<EB>::T;
    *reinterpret_cast<T*>(d) = *reinterpret_cast<const T*>(s);
}

// ---------------------------------------------------------------------------
// Element conversions of the fused permute + cast (IEEE 754, ties to even).  NaNs
// keep their sign and upper payload bits (the lowest payload bit set if those are
// all zero) when narrowed, and their payload when widened.
// ---------------------------------------------------------------------------
// binary32 -> bfloat16: the upper half rounded to nearest even by adding 0x7FFF
// plus the kept half's lowest bit before truncating (finite and infinite values;
// a carry out of the largest finite value gives infinity, as it should).
__device__ __forceinline__ uint32_t f32_to_bf16(uint32_t b) {
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) {
        const uint32_t pay = (b >> 16) & 0x7Fu;
        return ((b >> 16) & 0x8000u) | 0x7F80u | (pay ? pay : 1u);
    }
    return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;
}
// binary32 -> binary16 (CUDA's round-to-nearest-even conversion for numbers)
__device__ __forceinline__ uint32_t f32_to_f16(uint32_t b) {
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) {
        const uint32_t pay = (b & 0x7FFFFFu) >> 13;
        return ((b >> 16) & 0x8000u) | 0x7C00u | (pay ? pay : 1u);
    }
    return __half_as_ushort(__float2half_rn(__uint_as_float(b)));
}
// bfloat16 -> binary32: exact
__device__ __forceinline__ uint32_t bf16_to_f32(uint32_t h) { return (h & 0xFFFFu) << 16; }
// binary16 -> binary32: exact (CUDA's conversion for numbers)
__device__ __forceinline__ uint32_t f16_to_f32(uint32_t h) {
    h &= 0xFFFFu;
    if ((h & 0x7C00u) == 0x7C00u && (h & 0x3FFu))
        return ((h & 0x8000u) << 16) | 0x7F800000u | ((h & 0x3FFu) << 13);
    return __float_as_uint(__half2float(__ushort_as_half((unsigned short)h)));
}

// Cast c: source / destination element bytes and the conversion of one element.
template <int CAST> struct Cast;
template <> struct Cast<TL_CAST_NONE> {};
template <> struct Cast<TL_CAST_F32_TO_BF16> {
    static constexpr int kSrc = 4, kDst = 2;
    __device__ static uint32_t cvt(uint32_t x) { return f32_to_bf16(x); }
};
template <> struct Cast<TL_CAST_F32_TO_F16> {
    static constexpr int kSrc = 4, kDst = 2;
    __device__ static uint32_t cvt(uint32_t x) { return f32_to_f16(x); }
};
template <> struct Cast<TL_CAST_BF16_TO_F32> {
    static constexpr int kSrc = 2, kDst = 4;
    __device__ static uint32_t cvt(uint32_t x) { return bf16_to_f32(x); }
};
template <> struct Cast<TL_CAST_F16_TO_F32> {
    static constexpr int kSrc = 2, kDst = 4;
    __device__ static uint32_t cvt(uint32_t x) { return f16_to_f32(x); }
};

// ---------------------------------------------------------------------------
// Division of unsigned 32-bit numerators by a divisor fixed at launch time
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994: a magic multiplier with a post-shift).
// ---------------------------------------------------------------------------
struct DivU32 {
    uint32_t d = 1, m = 0, s = 0;
};

inline DivU32 make_divu32(uint32_t d) {
    DivU32 r;
    r.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;           // l = ceil(log2 d)
    r.s = l;
    // m = floor(2^32 * (2^l - d) / d) + 1   (fits in 32 bits for d >= 1)
    r.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return r;
}

__device__ __forceinline__ uint32_t div_u32(uint32_t n, const DivU32& v) {
    uint32_t t = __umulhi(n, v.m);
    return (uint32_t)(((uint64_t)t + n) >> v.s);
}

// ---------------------------------------------------------------------------
// PTX: shared-memory addresses, mbarriers, TMA, timer
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA) and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// After a bounded wait has expired, a CTA waits this many times as long for its own
// loads in flight before it leaves (a load that never lands leaves it anyway).
constexpr uint64_t kDrainFactor = 4;

// Waits for the phase of parity `parity` to complete.  Bounded: returns false once
// `timeout_ns` of wall time has passed without completion.  Each try_wait already
// suspends the thread for a while, so the loop does not spin hot.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(a, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// 2-D .. 5-D TMA tile load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                         int rank, int c0, int c1, int c2, int c3, int c4) {
    const uint32_t d = smem_addr(smem_dst), b = smem_addr(bar);
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    switch (rank) {
    case 2:
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(d),
            "l"(m), "r"(b), "r"(c0), "r"(c1)
            : "memory");
        break;
    case 3:
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(d),
            "l"(m), "r"(b), "r"(c0), "r"(c1), "r"(c2)
            : "memory");
        break;
    case 4:
        asm volatile(
            "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(d),
            "l"(m), "r"(b), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
            : "memory");
        break;
    default:
        asm volatile(
            "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(d),
            "l"(m), "r"(b), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
            : "memory");
        break;
    }
}

// Shared-memory loads of 4, 8 and 16 bytes.
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

// 16-byte shared-memory store (one aligned vector store).
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// 16-byte global store / load.
__device__ __forceinline__ void stg128(void* p, uint4 v) {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ uint4 ldg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel of the stream drains; it
// must wait for that kernel's completion (and memory visibility) before any
// global access.  Without the launch attribute both instructions are no-ops.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-CTA timing (measurement): thread 0 records the CTA's start, and every warp
// that calls cta_finish raises its finish to the time it got there (%globaltimer).
__device__ __forceinline__ void cta_start(uint64_t* times) {
    if (times && threadIdx.x == 0) times[2 * blockIdx.x] = global_timer_ns();
}
__device__ __forceinline__ void cta_finish(uint64_t* times) {
    if (times && (threadIdx.x & 31) == 0)
        atomicMax(reinterpret_cast<unsigned long long*>(&times[2 * blockIdx.x + 1]),
                  (unsigned long long)global_timer_ns());
}

// Records the first error of a launch in the caller's status word (if any).
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace dev
}  // namespace tl

namespace tl {
namespace dev {

// ---------------------------------------------------------------------------
// Cluster / distributed shared memory (sm_90+ PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Maps a shared::cta address of this CTA to the same variable in CTA `rank` of
// the cluster (PTX mapa).
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait on a local barrier whose arrivals / transactions come from the
// peer CTA (cluster-scope acquire).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_cluster(a, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// Arrive on a barrier of another CTA of the cluster (address from map_to_rank),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}

// The same arrive with a CTA-scope release, for a consumer handing a shared-memory
// slot back after reading it: the reads are complete (their values already fed
// the thread's stores), and a cluster-scope release would also wait until the
// thread's global stores reach L2 (1-2 us per tile measured on GB300 inside the
// cluster transpose).
__device__ __forceinline__ void mbar_arrive_remote_slot(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

}  // namespace dev
}  // namespace tl
