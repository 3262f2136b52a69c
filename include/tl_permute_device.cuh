/*
 * tl_permute_device.cuh -- device-side building blocks of the layout permute for
 * use inside your own CUDA kernels (header-only, sm_90 or newer; written for
 * sm_103a).  The library's own kernels use them too; nothing here touches library
 * state, allocates, or needs libtl_permute.so at run time.
 *
 *   warp_load_fragment / warp_store_fragment / warp_permute_layout
 *       The register-staged warp permute of the TVM "permute_layout" page
 *       ("Algorithm", step 3) on any memory space (shared, global): each of the 32
 *       lanes stages P elements, visiting its registers in the XOR-rotated order
 *       j = r ^ ((lane >> shift) & mask) that tl_choose_xor_k picks on the host so
 *       that both phases are shared-memory bank-conflict-free.
 *   warp_fragment_unrotate
 *       Turns the rotated registers into the plain lane-major fragment (register j
 *       of lane l = element l + 32*j of the tile), the thread-axis layout a
 *       consumer such as an MMA operand expects.
 *   dsmem_copy_region
 *       The "copy_async -> dsmem" page ("Algorithm", steps 1-3): one thread maps
 *       the destination buffer and mbarrier into another CTA of the cluster (mapa)
 *       and issues one cp.async.bulk.shared::cluster per contiguous chunk; the
 *       destination CTA arms its mbarrier with the total bytes and waits.
 *   wait_until_global
 *       The spin wait of the TVM wait_until pull request: relaxed polls of one
 *       global word until a predicate holds, then one acquire load closing the
 *       edge (its value discarded), with a wall-clock bound added.
 *
 * Element types are raw bits: use uint8_t, uint16_t, uint32_t, uint2 or uint4 for
 * 1, 2, 4, 8 and 16-byte elements.
 */
#pragma once

#include <cstdint>

namespace tl_dev {

// ---------------------------------------------------------------------------
// Warp tile layouts
// ---------------------------------------------------------------------------

/* A warp tile: up to 4 axes iterated row-major over `ext`; the element at
 * coordinates c sits at offset sum c[i] * str[i] (elements) from the base pointer
 * ("Buffers and memory", "Declaring buffers").  prod(ext) must be 32 * P. */
struct WarpTile {
    int32_t n;
    int32_t ext[4];
    int64_t str[4];
};

__device__ __forceinline__ int lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
    return (int)l;
}

/* Offset of the tile element with row-major index f. */
__device__ __forceinline__ int64_t tile_offset(const WarpTile& t, int64_t f) {
    int64_t off = 0;
#pragma unroll
    for (int i = 3; i >= 0; --i) {
        if (i < t.n) {
            const int64_t c = f % t.ext[i];
            f /= t.ext[i];
            off += c * t.str[i];
        }
    }
    return off;
}

/* Tile iteration index held in register r of `lane`. */
__device__ __forceinline__ int warp_iteration(int r, int lane, int shift, int mask) {
    return r ^ ((lane >> shift) & mask);
}

/* Phase 1: lane l reads into regs[r] the element with row-major index
 * l + 32 * (r ^ ((l >> shift) & mask)) of tile `t` over `src`. */
template <int P, typename T>
__device__ __forceinline__ void warp_load_fragment(T (&regs)[P], const T* src, const WarpTile& t,
                                                   int shift, int mask) {
    const int lane = lane_id();
#pragma unroll
    for (int r = 0; r < P; ++r)
        regs[r] = src[tile_offset(t, lane + 32LL * warp_iteration(r, lane, shift, mask))];
}

/* Phase 2: the same visiting order, writing through tile `t` over `dst`. */
template <int P, typename T>
__device__ __forceinline__ void warp_store_fragment(const T (&regs)[P], T* dst, const WarpTile& t,
                                                    int shift, int mask) {
    const int lane = lane_id();
#pragma unroll
    for (int r = 0; r < P; ++r)
        dst[tile_offset(t, lane + 32LL * warp_iteration(r, lane, shift, mask))] = regs[r];
}

/* Both phases with a warp barrier after each, so dst may alias src as long as
 * the warp's tile reads exactly the elements it writes (all 32 lanes must call). */
template <int P, typename T>
__device__ __forceinline__ void warp_permute_layout(T* dst, const T* src, const WarpTile& src_tile,
                                                    const WarpTile& dst_tile, int shift, int mask) {
    T regs[P];
    warp_load_fragment<P>(regs, src, src_tile, shift, mask);
    __syncwarp();
    warp_store_fragment<P>(regs, dst, dst_tile, shift, mask);
    __syncwarp();
}

/* Reorders registers loaded in the rotated order so that regs[j] holds tile
 * element lane + 32 * j.  XOR by x = (lane >> shift) & mask is applied one bit at
 * a time with conditional swaps (no dynamic register indexing). */
template <int P, typename T>
__device__ __forceinline__ void warp_fragment_unrotate(T (&regs)[P], int shift, int mask) {
    const int x = (lane_id() >> shift) & mask;
#pragma unroll
    for (int bit = 1; bit < P; bit <<= 1) {
        const bool flip = (x & bit) != 0;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            if (r & bit) continue;
            const T a = regs[r], b = regs[r | bit];
            regs[r] = flip ? b : a;
            regs[r | bit] = flip ? a : b;
        }
    }
}

/* Inverse of warp_fragment_unrotate (an XOR permutation is its own inverse). */
template <int P, typename T>
__device__ __forceinline__ void warp_fragment_rotate(T (&regs)[P], int shift, int mask) {
    warp_fragment_unrotate<P>(regs, shift, mask);
}

// ---------------------------------------------------------------------------
// DSMEM region copy ("copy_async -> dsmem")
// ---------------------------------------------------------------------------

/* The region as contiguous chunks: `chunk_bytes` contiguous bytes on both sides
 * at every coordinate of up to 4 outer axes (outer_n = 0: one chunk).  Strides are
 * in BYTES.  tl_layout_canon gives the split: the chunk is the common stride-1
 * chain (its last axis), the outer axes are the rest. */
struct ChunkLoop {
    uint32_t chunk_bytes;
    int32_t outer_n;
    int32_t outer_ext[4];
    int64_t src_stride[4];
    int64_t dst_stride[4];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

/* Total bytes the copy delivers (what the destination arms its mbarrier with). */
__device__ __forceinline__ uint32_t chunk_loop_bytes(const ChunkLoop& c) {
    uint32_t n = c.chunk_bytes;
    for (int i = 0; i < c.outer_n; ++i) n *= (uint32_t)c.outer_ext[i];
    return n;
}

/* Issue the copy from this CTA's shared memory (`src`) into the same-named
 * shared buffer `dst` of cluster CTA `peer`; each chunk completes its bytes on the
 * peer's mbarrier `peer_bar` (also named by this CTA's address of the variable).
 * Call from ONE thread after src is written and fenced (fence.proxy.async when it
 * was written by ordinary stores).  Returns false, issuing nothing, when a chunk
 * is under 16 bytes or not a multiple of 16 (the bulk-copy rule the page states),
 * or when an address or outer stride is not 16-byte aligned.
 * The copy is point to point, never a multicast; nothing here waits.  Its only
 * completion is the peer's barrier: the issuing CTA must not overwrite `src`
 * until the peer has seen the bytes land (have the peer signal back, e.g. with a
 * remote mbarrier arrive) -- cp.async.bulk.wait_group does not track this form. */
__device__ __forceinline__ bool dsmem_copy_region(void* dst, const void* src, const ChunkLoop& c,
                                                  uint32_t peer, uint64_t* peer_bar) {
    if (c.chunk_bytes < 16 || (c.chunk_bytes & 15u) != 0) return false;
    if (((smem_u32(dst) | smem_u32(src)) & 15u) != 0) return false;
    for (int i = 0; i < c.outer_n; ++i)
        if (((c.src_stride[i] | c.dst_stride[i]) & 15) != 0) return false;
    uint32_t rdst, rbar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rdst) : "r"(smem_u32(dst)), "r"(peer));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(rbar)
                 : "r"(smem_u32(peer_bar)), "r"(peer));
    const uint32_t s0 = smem_u32(src);
    int32_t idx[4] = {0, 0, 0, 0};
    const uint32_t total = chunk_loop_bytes(c) / c.chunk_bytes;
    for (uint32_t k = 0; k < total; ++k) {
        int64_t so = 0, d = 0;
        for (int i = 0; i < c.outer_n; ++i) {
            so += idx[i] * c.src_stride[i];
            d += idx[i] * c.dst_stride[i];
        }
        asm volatile(
            "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
            " [%0], [%1], %2, [%3];" ::"r"(rdst + (uint32_t)d),
            "r"(s0 + (uint32_t)so), "r"(c.chunk_bytes), "r"(rbar)
            : "memory");
        for (int i = c.outer_n - 1; i >= 0; --i) {      // odometer over the outer axes
            if (++idx[i] < c.outer_ext[i]) break;
            idx[i] = 0;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// Bounded spin wait on a global word (the wait_until pull request)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

/* Spin on *word with relaxed loads (the first one peeled) until pred(value)
 * holds, then issue one acquire load of the word whose value is discarded (it
 * may be later than the accepted one).  The accepted value goes to *value.
 * Returns false, without the acquire, once timeout_ns of wall time has passed.
 * Publishers release the word (st.release, atom, red).  Waits inside a CTA or a
 * cluster belong on an mbarrier instead. */
template <typename Pred>
__device__ __forceinline__ bool wait_until_global(const uint32_t* word, Pred pred,
                                                  uint64_t timeout_ns, uint32_t* value) {
    uint32_t v = ld_relaxed_gpu(word);
    if (!pred(v)) {
        const uint64_t t0 = global_timer_ns();
#pragma unroll 1
        do {
            if (global_timer_ns() - t0 > timeout_ns) return false;
            v = ld_relaxed_gpu(word);
        } while (!pred(v));
    }
    (void)ld_acquire_gpu(word);
    *value = v;
    return true;
}

/* The publishing side: a release store of a word. */
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

}  // namespace tl_dev
