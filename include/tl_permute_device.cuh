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
 *   ThreadAxisLayout / warp_load_lanes / warp_store_lanes
 *       Thread-axis ("1 @ laneid") layouts of the "Buffers and memory" page
 *       ("Buffer APIs", "Registers -- local"): every axis is bound either to the
 *       lane index with a lane stride or to the lane's registers with a register
 *       stride, so coordinate c sits in register sum(c * reg_str) of lane
 *       sum(c * lane_str); the load / store move a lane's registers (its `local`
 *       slice) from / to memory holding the same tensor under memory strides.
 *       tl_thread_axis_check (host C ABI) validates a layout and counts its
 *       registers.
 *   dsmem_copy_region
 *       The "copy_async -> dsmem" page ("Algorithm", steps 1-3): one thread maps
 *       the destination buffer and mbarrier into another CTA of the cluster (mapa)
 *       and issues one cp.async.bulk.shared::cluster per contiguous chunk; the
 *       destination CTA arms its mbarrier with the total bytes and waits.
 *   wait_until_global
 *       The spin wait of the TVM wait_until pull request: relaxed polls of one
 *       global word (32 or 64 bits, at a chosen scope, with an opt-in backoff)
 *       until a predicate holds, then one acquire load closing the edge (its value
 *       discarded), with a wall-clock bound added.
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
// Thread-axis layouts ("Buffers and memory", "Buffer APIs", "Registers -- local")
// ---------------------------------------------------------------------------

/* A warp's thread-axis layout over up to 4 axes: axis k is bound to the lane index
 * (lane_str[k] > 0, reg_str[k] == 0) or to the lane's registers (reg_str[k] > 0,
 * lane_str[k] == 0); the coordinate c lives in register sum(c * reg_str) of lane
 * sum(c * lane_str).  The page's S[(32, 8) : (1 @ laneid, 1)] is n = 2, ext = (32, 8),
 * lane_str = (1, 0), reg_str = (0, 1): element (l, j) in register j of lane l.
 * mem_str are the element strides of the same tensor in memory.  Lane and register
 * strides must place the prod(ext) coordinates on 32 lanes x P registers once each
 * (tl_thread_axis_check verifies a layout on the host and returns P). */
struct ThreadAxisLayout {
    int32_t n;
    int32_t ext[4];
    int32_t lane_str[4];
    int32_t reg_str[4];
    int64_t mem_str[4];
};

/* Memory offset (elements) of the part of a coordinate that the lane index fixes. */
__device__ __forceinline__ int64_t lane_offset(const ThreadAxisLayout& t, int lane) {
    int64_t off = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < t.n && t.lane_str[k] > 0)
            off += (int64_t)((lane / t.lane_str[k]) % t.ext[k]) * t.mem_str[k];
    return off;
}

/* Memory offset (elements) of the part of a coordinate that register j fixes. */
__device__ __forceinline__ int64_t register_offset(const ThreadAxisLayout& t, int j) {
    int64_t off = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (k < t.n && t.reg_str[k] > 0)
            off += (int64_t)((j / t.reg_str[k]) % t.ext[k]) * t.mem_str[k];
    return off;
}

/* The calling lane's P registers of layout `t` from memory at `src` (every lane of
 * the warp calls it; no synchronisation is needed, each lane reads its own). */
template <int P, typename T>
__device__ __forceinline__ void warp_load_lanes(T (&regs)[P], const T* src,
                                                const ThreadAxisLayout& t) {
    const T* base = src + lane_offset(t, lane_id());
#pragma unroll
    for (int j = 0; j < P; ++j) regs[j] = base[register_offset(t, j)];
}

/* The calling lane's P registers of layout `t` to memory at `dst`. */
template <int P, typename T>
__device__ __forceinline__ void warp_store_lanes(const T (&regs)[P], T* dst,
                                                 const ThreadAxisLayout& t) {
    T* base = dst + lane_offset(t, lane_id());
#pragma unroll
    for (int j = 0; j < P; ++j) base[register_offset(t, j)] = regs[j];
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

/* Memory scope of the polls and of the closing acquire (the pull request's
 * `scope`): .cta, .cluster, .gpu or .sys. */
enum class WaitScope { cta, cluster, gpu, sys };

/* Relaxed and acquire loads of a 32- or 64-bit global word at scope S (the pull
 * request's ptx_type: any 4- or 8-byte type is read as its raw bits; 128 bits is
 * refused at compile time, its value is not a scalar a predicate can test). */
template <WaitScope S, typename W>
__device__ __forceinline__ W ld_wait_word(const W* p, bool acquire) {
    static_assert(sizeof(W) == 4 || sizeof(W) == 8, "wait words are 32 or 64 bits");
    if constexpr (sizeof(W) == 4) {
        uint32_t v;
#define TL_LD32(SEM, SC)                                                                   \
    asm volatile("ld." SEM "." SC ".global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory")
        if (acquire) {
            if constexpr (S == WaitScope::cta) TL_LD32("acquire", "cta");
            else if constexpr (S == WaitScope::cluster) TL_LD32("acquire", "cluster");
            else if constexpr (S == WaitScope::gpu) TL_LD32("acquire", "gpu");
            else TL_LD32("acquire", "sys");
        } else {
            if constexpr (S == WaitScope::cta) TL_LD32("relaxed", "cta");
            else if constexpr (S == WaitScope::cluster) TL_LD32("relaxed", "cluster");
            else if constexpr (S == WaitScope::gpu) TL_LD32("relaxed", "gpu");
            else TL_LD32("relaxed", "sys");
        }
#undef TL_LD32
        W w;
        __builtin_memcpy(&w, &v, 4);
        return w;
    } else {
        uint64_t v;
#define TL_LD64(SEM, SC)                                                                   \
    asm volatile("ld." SEM "." SC ".global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory")
        if (acquire) {
            if constexpr (S == WaitScope::cta) TL_LD64("acquire", "cta");
            else if constexpr (S == WaitScope::cluster) TL_LD64("acquire", "cluster");
            else if constexpr (S == WaitScope::gpu) TL_LD64("acquire", "gpu");
            else TL_LD64("acquire", "sys");
        } else {
            if constexpr (S == WaitScope::cta) TL_LD64("relaxed", "cta");
            else if constexpr (S == WaitScope::cluster) TL_LD64("relaxed", "cluster");
            else if constexpr (S == WaitScope::gpu) TL_LD64("relaxed", "gpu");
            else TL_LD64("relaxed", "sys");
        }
#undef TL_LD64
        W w;
        __builtin_memcpy(&w, &v, 8);
        return w;
    }
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    return ld_wait_word<WaitScope::gpu>(p, false);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    return ld_wait_word<WaitScope::gpu>(p, true);
}

/* Spin on *word with relaxed loads at scope S (the first one peeled) until
 * pred(value) holds, then issue one acquire load of the word whose value is
 * discarded (it may be later than the accepted one).  The accepted value goes to
 * *value.  backoff_ns > 0 sleeps that long (__nanosleep) between polls, which the
 * pull request measured as never faster (+1.35 % at 20 ns, +30 % at 2 us), so it
 * is opt-in.  Returns false, without the acquire, once timeout_ns of wall time has
 * passed.  W is a 32- or 64-bit word type.  Publishers release the word
 * (st.release, atom, red).  Waits inside a CTA or a cluster belong on an
 * mbarrier instead (shared memory is not a global word). */
template <WaitScope S = WaitScope::gpu, typename W, typename Pred>
__device__ __forceinline__ bool wait_until_global(const W* word, Pred pred, uint64_t timeout_ns,
                                                  W* value, uint32_t backoff_ns = 0) {
    W v = ld_wait_word<S>(word, false);
    if (!pred(v)) {
        const uint64_t t0 = global_timer_ns();
#pragma unroll 1
        do {
            if (global_timer_ns() - t0 > timeout_ns) return false;
            if (backoff_ns) __nanosleep(backoff_ns);
            v = ld_wait_word<S>(word, false);
        } while (!pred(v));
    }
    (void)ld_wait_word<S>(word, true);
    *value = v;
    return true;
}

/* The publishing side: a release store of a word. */
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_gpu(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

}  // namespace tl_dev
