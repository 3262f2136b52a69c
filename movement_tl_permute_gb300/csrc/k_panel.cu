// k_panel.cu -- transpose of the plane through shared memory for the layouts the
// TMA tile path cannot take: rows whose byte pitch is not a multiple of 16, more
// than three batch axes, or a plane with a tiny extent (an interleaved-channel axis
// of 3).
//
// Plane: axis a is contiguous in src, axis b is contiguous in dst; the rest are
// batch axes.  A tile is ta elements of a by tb elements of b.  Each CTA runs a
// ring of kPanelStages shared-memory stages: while it stores one tile, the
// asynchronous copies (cp.async, 16 bytes each, no registers involved) of the next
// tiles are in flight.  Each src row of a tile is copied as the aligned 16-byte
// blocks that cover it, whatever the element alignment (a block that holds a byte
// of the row never crosses a page the row does not touch), and lands at the same
// offset inside its first block; when the tile's src rows are packed back to back
// the whole tile is one run of blocks.
//
// The copy walks the tile in src order, so consecutive threads read consecutive
// src addresses; the stores walk it in dst order, so consecutive threads write
// consecutive dst addresses: element by element (f -> a = f / tb, b = f % tb), as
// 4-byte words (packed 1- and 2-byte rows, and 1-byte rows per dst row), as 16-byte
// runs along the tile rows when the dst rows are 16-byte aligned (drain_vec), or as
// 16-byte pieces of the tile's single dst run (drain_run).  Rows whose pitch is off
// the 16-byte grid are staged phase-major (rows b = j mod phi together), filled by
// cp.async or, in k_panel_tma, by TMA loads through one tensor map per phase.  The
// row pitch and the lanes' read rotations are chosen on the host by simulating the
// walks' warp accesses against the banks (the bank model of the TVM
// "permute_layout" page, "Algorithm", step 2).  Element offsets follow the strided
// addressing of "Buffers and memory", "Declaring buffers".
#include "tl_kernels.h"

namespace tl {
namespace {

// 16-byte asynchronous copy global -> shared, cached in L2 only
__device__ __forceinline__ void cp_async16(uint32_t saddr, uintptr_t gaddr) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gaddr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct PanelTile {
    int64_t so, dof;      // element offsets of the tile's (a0, b0) in src and dst
    int64_t dob;          // dst offset of (b0, batch item) alone
    int64_t b0;           // first b of the tile
    uint32_t va, vb;      // valid elements of a and b
    int64_t a0;           // first a of the tile
    int32_t c[3];         // coordinates on the three innermost batch axes
};

// dst element offset of the tile's row a0 + e at b0: e * ds_a past the tile's origin,
// or, when a is two merged axes (AM, its own kernels), from the split of the absolute a
template <bool AM>
__device__ __forceinline__ int64_t drow_off(const PanelArgs& a, const PanelTile& ti, uint32_t e) {
    if constexpr (!AM) {
        return ti.dof + (int64_t)e * a.ds_a;
    } else {
        const uint32_t x = (uint32_t)ti.a0 + e;
        const uint32_t hi = dev::div_u32(x, a.d_a1);
        return ti.dob + (int64_t)(x - hi * a.d_a1.d) * a.ds_a + (int64_t)hi * a.ds_a2;
    }
}

// Byte offset of tile row b in a block-row stage: b * pitch, or, for phase-major
// stages (filled by TMA phase maps or by cp.async in the same arrangement), row
// b / phi of the block of phase b % phi.
// (1-byte elements never take a phase-major stage: their block rows stay b * pitch)
template <int EB>
__device__ __forceinline__ uint32_t stage_row(const PanelArgs& a, uint32_t b) {
    if constexpr (EB != 1) {
        if (a.phase)
            return (b & ((1u << a.phi_lg) - 1u)) * (uint32_t)a.phase_bytes +
                   (b >> a.phi_lg) * (uint32_t)a.pitch;
    }
    return b * (uint32_t)a.pitch;
}

// src offset of b (elements); b is one axis of stride ss_b, or two merged axes
__device__ __forceinline__ int64_t b_offset(int64_t b, const PanelArgs& a) {
    if (!a.merged) return b * a.ss_b;
    const uint32_t hi = dev::div_u32((uint32_t)b, a.d_b1);
    return (int64_t)((uint32_t)b - hi * a.d_b1.d) * a.ss_b + (int64_t)hi * a.ss_b2;
}

// src offset of tile row bb relative to the tile's first row
__device__ __forceinline__ int64_t row_offset(uint32_t bb, const PanelTile& ti,
                                              const PanelArgs& a) {
    if (!a.merged) return (int64_t)bb * a.ss_b;
    return b_offset(ti.b0 + bb, a) - b_offset(ti.b0, a);
}

// tile t -> (column block of a, row block of b, batch item).  Tile rows are
// visited in groups of group_b, b fastest inside a group: concurrently running
// CTAs then write runs of group_b * tb elements of dst rows while the tiles beside
// each other along a, which share the 16-byte blocks at their row ends, are in
// flight together and meet those blocks in L2.
// The batch loop is unrolled over TL_MAX_DIMS (keeping the coordinates) or a plain
// loop: measured per width, 1-byte tiles store a third faster with the plain loop
// (odd-pitch u8 transposes 2.4 -> 3.6 TB/s), the wider ones keep the unrolled one.
template <bool AM, bool UNROLLED>
__device__ __forceinline__ PanelTile panel_tile(int64_t t, const PanelArgs& a) {
    int64_t item, ia, ib;
    if (a.use32) {
        const uint32_t t32 = (uint32_t)t;
        const uint32_t it = dev::div_u32(t32, a.d_item);
        const uint32_t local = t32 - it * a.d_item.d;
        const uint32_t grp = dev::div_u32(local, a.d_grp);
        const uint32_t first = grp * a.d_gfull.d;
        const uint32_t in_grp = local - grp * a.d_grp.d;
        const dev::DivU32& dg = first + a.d_gfull.d > (uint32_t)a.tiles_b ? a.d_glast : a.d_gfull;
        const uint32_t qa = dev::div_u32(in_grp, dg);
        item = it;
        ia = qa;
        ib = first + (in_grp - qa * dg.d);
    } else {
        const int64_t per_item = a.tiles_a * a.tiles_b;
        item = t / per_item;
        const int64_t local = t - item * per_item;
        const int64_t grp = local / (a.group_b * a.tiles_a);
        const int64_t first = grp * a.group_b;
        const int64_t gsize = min(a.group_b, a.tiles_b - first);
        const int64_t in_grp = local - grp * a.group_b * a.tiles_a;
        ia = in_grp / gsize;
        ib = first + in_grp % gsize;
    }
    const int64_t a0 = ia * a.ta, b0 = ib * a.tb;
    PanelTile r;
    r.va = (uint32_t)min((int64_t)a.ta, a.ext_a - a0);
    r.vb = (uint32_t)min((int64_t)a.tb, a.ext_b - b0);
    r.b0 = b0;
    r.a0 = a0;
    r.so = a0 + b_offset(b0, a);
    r.dof = AM ? b0 : a0 * a.ds_a + b0;
    auto axis = [&](int i) {           // batch axis i: its coordinate, offsets added
        int64_t c;
        if (a.use32) {
            const uint32_t q = dev::div_u32((uint32_t)item, a.d_bext[i]);
            c = (uint32_t)item - q * a.d_bext[i].d;
            item = q;
        } else {
            c = item % a.bext[i];
            item /= a.bext[i];
        }
        r.so += c * a.bss[i];
        r.dof += c * a.bds[i];
        return c;
    };
    r.c[0] = r.c[1] = r.c[2] = 0;
    if constexpr (UNROLLED) {          // (the TMA loads take the three innermost coordinates)
#pragma unroll
        for (int i = 0; i < TL_MAX_DIMS; ++i) {
            if (i >= a.nb) break;
            const int64_t c = axis(i);
            if (i < 3) r.c[i] = (int32_t)c;
        }
    } else {
        for (int i = 0; i < a.nb; ++i) axis(i);
    }
    if constexpr (AM) {          // (b0, batch item) alone, then the split of a0
        const uint32_t hi = dev::div_u32((uint32_t)a0, a.d_a1);
        r.dob = r.dof;
        r.dof += (int64_t)((uint32_t)a0 - hi * a.d_a1.d) * a.ds_a + (int64_t)hi * a.ds_a2;
    }
    return r;
}

// Start the copies of one tile into the stage at shared address `sb`: the
// 16-byte blocks covering each src row of the tile (or the tile's single run).
template <int EB>
__device__ __forceinline__ void issue(const PanelArgs& a, const PanelTile& ti, uint32_t sb) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(a.src + ti.so * EB);
    // row b of a block-row stage: b * pitch, plus 16 bytes per V = 16 / EB rows when
    // the stage is skewed for 16-byte dst runs
    constexpr uint32_t V = 16 / EB;
    const uint32_t skew = a.vskew ? 16u : 0u;
    if (a.mode == kPanelRows && a.aligned) {
        // every row starts on a block boundary: nblk blocks per full row, the valid
        // rows only
        const uint32_t nblk = (uint32_t)a.nblk, n = ti.vb * nblk;
        const uint32_t blocks = (ti.va * EB + 15) >> 4, pitch = (uint32_t)a.pitch;
        for (uint32_t g = threadIdx.x; g < n; g += kPanelThreads) {
            const uint32_t b = dev::div_u32(g, a.d_nblk), k = g - b * nblk;
            if (k < blocks)
                cp_async16(sb + b * pitch + (b / V) * skew + 16 * k,
                           base + (uintptr_t)(row_offset(b, ti, a) * EB) + 16 * k);
        }
    } else if (a.mode == kPanelRows) {
        const uint32_t nblk = (uint32_t)a.nblk, n = (uint32_t)a.tb * nblk;
        const uint32_t pitch = (uint32_t)a.pitch;
        for (uint32_t g = threadIdx.x; g < n; g += kPanelThreads) {
            const uint32_t b = dev::div_u32(g, a.d_nblk), k = g - b * nblk;
            if (b >= ti.vb) continue;
            const uintptr_t row = base + (uintptr_t)(row_offset(b, ti, a) * EB);
            const uint32_t blocks = ((uint32_t)(row & 15) + ti.va * EB + 15) >> 4;
            if (k < blocks)
                cp_async16(sb + (skew ? b * pitch + (b / V) * skew : stage_row<EB>(a, b)) + 16 * k,
                           (row & ~uintptr_t(15)) + 16 * k);
        }
    } else {   // kPanelFlat: rows packed back to back (ss_b == ta == va)
        const uint32_t blocks = ((uint32_t)(base & 15) + ti.vb * (uint32_t)a.ta * EB + 15) >> 4;
        for (uint32_t k = threadIdx.x; k < blocks; k += kPanelThreads)
            cp_async16(sb + 16 * k, (base & ~uintptr_t(15)) + 16 * k);
    }
}

// V = 16 / EB elements in b order as one 16-byte vector
__device__ __forceinline__ uint4 pack16(const uint2 (&v)[2]) {
    return make_uint4(v[0].x, v[0].y, v[1].x, v[1].y);
}
__device__ __forceinline__ uint4 pack16(const uint32_t (&v)[4]) {
    return make_uint4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ uint4 pack16(const uint16_t (&v)[8]) {
    auto w = [&](int i) { return (uint32_t)v[2 * i] | ((uint32_t)v[2 * i + 1] << 16); };
    return make_uint4(w(0), w(1), w(2), w(3));
}
__device__ __forceinline__ uint4 pack16(const uint8_t (&v)[16]) {
    auto w = [&](int i) {
        return (uint32_t)v[4 * i] | ((uint32_t)v[4 * i + 1] << 8) |
               ((uint32_t)v[4 * i + 2] << 16) | ((uint32_t)v[4 * i + 3] << 24);
    };
    return make_uint4(w(0), w(1), w(2), w(3));
}

// dst address of the 16-byte run of tile row a0 + e at b0, for a walk whose e steps
// by de: a pointer advanced by de * ds_a, or, for merged a, the split of each e
template <int EB, bool AM>
struct RunPtr {
    uint8_t* p;
    int64_t step;
    __device__ __forceinline__ RunPtr(const PanelArgs& a, const PanelTile& ti, uint32_t e,
                                      uint32_t b0, uint32_t de)
        : p(a.dst + (ti.dof + (int64_t)e * a.ds_a + b0) * EB), step((int64_t)de * a.ds_a * EB) {}
    __device__ __forceinline__ uint8_t* at(const PanelArgs&, const PanelTile&, uint32_t) const {
        return p;
    }
    __device__ __forceinline__ void next() { p += step; }
};
template <int EB>
struct RunPtr<EB, true> {
    uint32_t b0;
    __device__ __forceinline__ RunPtr(const PanelArgs&, const PanelTile&, uint32_t, uint32_t b,
                                      uint32_t)
        : b0(b) {}
    __device__ __forceinline__ uint8_t* at(const PanelArgs& a, const PanelTile& ti,
                                           uint32_t e) const {
        return a.dst + (drow_off<true>(a, ti, e) + b0) * EB;
    }
    __device__ __forceinline__ void next() {}
};

// Store one landed tile as 16-byte dst runs (used when the dst rows of every tile
// start on 16-byte boundaries and tb * EB is a whole number of 16-byte blocks).
// Unit (e, q) is dst row e of the tile, block q of it (elements b = qV .. qV + V - 1,
// V = 16 / EB).  A warp takes 4 rows x 8 blocks, so each of its stores writes four
// 128-byte pieces (lanes past the last block of a row idle); a thread keeps its block
// q for the whole tile and walks e, so the V row addresses
// are computed once.  Block-row stages are skewed: row b starts 16 bytes
// further per V rows (at b * pitch + 16 * (b / V)), so the 8 blocks of a warp read
// 8 distinct 16-byte bank groups at every step whatever the pitch (the host's pitch
// search replays these reads on the bank model of the TVM "permute_layout" page,
// "Algorithm" step 2).
template <int EB, bool AM>
__device__ __forceinline__ void drain_vec(const PanelArgs& a, const PanelTile& ti,
                                          const uint8_t* st) {
    using T = typename dev::Bits<EB>::T;
    constexpr uint32_t V = 16 / EB, kWarps = kPanelThreads / 32;
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t qb8 = (uint32_t)a.qb8;
    // the warp's 8-block groups (qg, stepping kWarps) and 4-row groups (g4)
    uint32_t qg0 = warp, g40 = 0, gstep = 1;
    if (qb8 < kWarps) {
        const uint32_t per = kWarps / qb8;
        if (warp >= per * qb8) return;
        qg0 = warp % qb8;
        g40 = warp / qb8;
        gstep = per;
    }
    const uint32_t mis0 = (uint32_t)(reinterpret_cast<uintptr_t>(a.src + ti.so * EB) & 15);
    const uint32_t P = (uint32_t)a.vpitch, delta = (uint32_t)a.vdelta;
    const uint32_t skew = a.vskew ? 16u : 0u;
    // row addresses as offsets into the dynamic shared memory, so that every read is
    // a shared-window load
    extern __shared__ __align__(16) uint8_t smem_rows[];
    const uint32_t st0 = (uint32_t)(st - smem_rows);
    for (uint32_t qg = qg0; qg < qb8; qg += kWarps) {
        const uint32_t q = 8 * qg + (lane & 7), b0 = q * V;
        if (b0 >= ti.vb) continue;
        uint32_t ro[V];
#pragma unroll
        for (uint32_t k = 0; k < V; ++k) {
            const uint32_t b = b0 + k;
            ro[k] = st0 + b * P + q * skew + ((mis0 + b * delta) & 15u);
        }
        uint32_t e = 4 * g40 + (lane >> 3);
        RunPtr<EB, AM> rp(a, ti, e, b0, 4 * gstep);
        if (b0 + V <= ti.vb) {
#pragma unroll 2
            for (; e < ti.va; e += 4 * gstep, rp.next()) {
                T v[V];
#pragma unroll
                for (uint32_t k = 0; k < V; ++k)
                    v[k] = *reinterpret_cast<const T*>(&smem_rows[ro[k] + e * EB]);
                dev::stg128(rp.at(a, ti, e), pack16(v));
            }
        } else {           // the block holds the last valid rows of a ragged tile
            for (; e < ti.va; e += 4 * gstep, rp.next()) {
                uint8_t* dp = rp.at(a, ti, e);
#pragma unroll
                for (uint32_t k = 0; k < V; ++k)
                    if (b0 + k < ti.vb)
                        *reinterpret_cast<T*>(dp + k * EB) =
                            *reinterpret_cast<const T*>(&smem_rows[ro[k] + e * EB]);
            }
        }
    }
}

// Store one landed tile whose dst is a single run (a short b axis packed in dst, as
// planes -> interleaved channels: tb == ext_b <= 16, ds_a == tb) as 16-byte pieces
// of that run, V = 16 / EB elements each: element f of the run is stage row
// b = f % tb, column a = f / tb; one division per piece, then b steps and wraps.
// Stage row b starts at b * vpitch + ((mis0 + b * vdelta) & 15) (block rows, or
// packed rows with vpitch = ta * EB).  The elements before the run's first 16-byte
// boundary and after its last one are stored singly.
template <int EB>
__device__ __forceinline__ void drain_run(const PanelArgs& a, const PanelTile& ti,
                                          const uint8_t* st) {
    using T = typename dev::Bits<EB>::T;
    constexpr uint32_t V = 16 / EB;
    extern __shared__ __align__(16) uint8_t smem_run[];
    const uint32_t tb = (uint32_t)a.tb, P = (uint32_t)a.vpitch, delta = (uint32_t)a.vdelta;
    const uint32_t st0 = (uint32_t)(st - smem_run);
    const uint32_t mis0 = (uint32_t)(reinterpret_cast<uintptr_t>(a.src + ti.so * EB) & 15);
    auto at = [&](uint32_t b, uint32_t e) {
        return *reinterpret_cast<const T*>(
            &smem_run[st0 + b * P + ((mis0 + b * delta) & 15u) + e * EB]);
    };
    uint8_t* d = a.dst + ti.dof * EB;
    const uint32_t n = ti.va * tb;
    const uint32_t lead = (uint32_t)((16 - (reinterpret_cast<uintptr_t>(d) & 15)) & 15) / EB;
    const uint32_t head = min(n, lead);
    const uint32_t nu = (n - head) / V, tail = head + nu * V;
    if (threadIdx.x < head) {
        const uint32_t e = dev::div_u32(threadIdx.x, a.d_tb);
        reinterpret_cast<T*>(d)[threadIdx.x] = at(threadIdx.x - e * tb, e);
    }
    if (tail + threadIdx.x < n) {
        const uint32_t f = tail + threadIdx.x, e = dev::div_u32(f, a.d_tb);
        reinterpret_cast<T*>(d)[f] = at(f - e * tb, e);
    }
    for (uint32_t u = threadIdx.x; u < nu; u += kPanelThreads) {
        const uint32_t f0 = head + u * V;
        uint32_t e = dev::div_u32(f0, a.d_tb), b = f0 - e * tb;
        T v[V];
#pragma unroll
        for (uint32_t k = 0; k < V; ++k) {
            v[k] = at(b, e);
            const bool wrap = ++b == tb;
            b = wrap ? 0 : b;
            e += wrap ? 1 : 0;
        }
        dev::stg128(d + (size_t)f0 * EB, pack16(v));
    }
}

// Store one landed tile of 1-byte elements in block rows whose dst rows are not on the
// 16-byte grid, as 4-byte words (written for 4 / EB elements a word; 2-byte elements
// measured faster with element stores, so only 1-byte tiles take it): warp i takes the tile's dst rows a = i, i + 8,
// ..., lane w packing word w (4 / EB consecutive b) of each from 4 / EB stage rows.  The
// dst rows of one warp are 8 pitches apart, a multiple of 4 bytes, so they share their
// head (the elements before the first 4-byte boundary) and the lanes' stage rows:
// those addresses and the packing shifts are computed once per tile.  Lane w reads its
// k-th element as (k + wrot_m * (w >> wrot_s)) mod (4 / EB) of its word, the rotation
// chosen on the host together with the row pitch by simulating these reads on the
// banks.  Head and tail elements are stored singly.
template <int EB>
__device__ __forceinline__ void drain_words(const PanelArgs& a, const PanelTile& ti,
                                            const uint8_t* st) {
    using T = typename dev::Bits<EB>::T;
    constexpr uint32_t V = 4 / EB, kWarps = kPanelThreads / 32;
    extern __shared__ __align__(16) uint8_t smem_w[];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp >= ti.va) return;
    const uint32_t st0 = (uint32_t)(st - smem_w);
    const uint32_t delta = (uint32_t)a.vdelta;
    const uint32_t mis0 = (uint32_t)(reinterpret_cast<uintptr_t>(a.src + ti.so * EB) & 15);
    auto row = [&](uint32_t b) { return st0 + stage_row<EB>(a, b) + ((mis0 + b * delta) & 15u); };
    uint8_t* d0 = a.dst + (ti.dof + (int64_t)warp * a.ds_a) * EB;   // first dst row of the warp
    const int64_t dstep = (int64_t)kWarps * a.ds_a * EB;
    const uint32_t lead = (uint32_t)((4 - (reinterpret_cast<uintptr_t>(d0) & 3)) & 3) / EB;
    const uint32_t head = min(ti.vb, lead);
    const uint32_t nw = (ti.vb - head) / V, tail = head + nw * V;
    for (uint32_t w = lane; w < nw; w += 32) {
        const uint32_t rot = (uint32_t)a.wrot_m * (w >> a.wrot_s);
        uint32_t ro[V], sh[V];
#pragma unroll
        for (uint32_t k = 0; k < V; ++k) {
            const uint32_t kk = (k + rot) & (V - 1);
            ro[k] = row(head + w * V + kk);
            sh[k] = 8 * EB * kk;
        }
        uint8_t* dp = d0 + (size_t)(head + w * V) * EB;
        for (uint32_t e = warp; e < ti.va; e += kWarps, dp += dstep) {
            uint32_t word = 0;
#pragma unroll
            for (uint32_t k = 0; k < V; ++k)
                word |= (uint32_t)(*reinterpret_cast<const T*>(&smem_w[ro[k] + e * EB])) << sh[k];
            *reinterpret_cast<uint32_t*>(dp) = word;
        }
    }
    // head and tail elements: lane j < head stores element j, lane j < vb - tail
    // element tail + j, of every dst row of the warp
    const uint32_t nh = ti.vb - tail;
    if (lane < head || lane < nh) {
        const uint32_t rh = row(lane), rt = row(tail + lane);
        uint8_t* dp = d0;
        for (uint32_t e = warp; e < ti.va; e += kWarps, dp += dstep) {
            if (lane < head)
                reinterpret_cast<T*>(dp)[lane] = *reinterpret_cast<const T*>(&smem_w[rh + e * EB]);
            if (lane < nh)
                reinterpret_cast<T*>(dp)[tail + lane] =
                    *reinterpret_cast<const T*>(&smem_w[rt + e * EB]);
        }
    }
}

// Store one landed tile from the stage at `st` to dst, in dst order: 16-byte runs
// (VEC), or element by element (4-byte words for packed rows of 1- and 2-byte
// elements).
template <int EB, bool VEC, bool AM>
__device__ __forceinline__ void drain(const PanelArgs& a, const PanelTile& ti, const uint8_t* st) {
    if constexpr (VEC) {
        drain_vec<EB, AM>(a, ti, st);
        return;
    }
    // (the run and word walks need one dst offset step per row of a: not merged)
    if constexpr (EB <= 8 && !AM) {
        if (a.run) {
            drain_run<EB>(a, ti, st);
            return;
        }
    }
    if constexpr (EB == 1 && !AM) {
        if (a.words) {
            drain_words<EB>(a, ti, st);
            return;
        }
    }
    using T = typename dev::Bits<EB>::T;
    T* d = reinterpret_cast<T*>(a.dst) + ti.dof;
    const uint32_t ta = (uint32_t)a.ta, tb = (uint32_t)a.tb, pitch = (uint32_t)a.pitch;
    const uint32_t mis0 = (uint32_t)(reinterpret_cast<uintptr_t>(a.src + ti.so * EB) & 15);
    const bool rows = a.mode == kPanelRows;
    // byte offset of tile row b inside its first 16-byte block
    auto mis = [&](uint32_t b) { return (mis0 + (uint32_t)(row_offset(b, ti, a) * EB)) & 15u; };
    if constexpr (EB < 4) {
        if (!rows) {
            // Packed src rows (a short a axis, such as interleaved channels): each dst
            // row a gets its run of b in 4-byte words, a lane packing 4 / EB elements
            // that sit ta elements apart in the stage (lanes 4 * ta bytes apart).  An
            // even ta puts lanes on the same banks, so lane l reads its k-th element
            // as element (k + wrot_m * (l >> wrot_s)) mod (4 / EB) of its word, the
            // rotation picked on the host by simulating the banks (the XOR rotation
            // of the TVM "permute_layout" page, "Algorithm" step 2, as a modular
            // one).  The elements before the first 4-byte boundary of the row and
            // after the last one are stored singly.
            constexpr uint32_t V = 4 / EB;
            const uint32_t rot = (uint32_t)a.wrot_m * ((threadIdx.x & 31) >> a.wrot_s);
            auto elem = [&](uint32_t b, uint32_t e) {
                return *reinterpret_cast<const T*>(st + mis0 + (b * ta + e) * EB);
            };
            for (uint32_t e = 0; e < ti.va; ++e) {
                T* drow = AM ? reinterpret_cast<T*>(a.dst) + drow_off<AM>(a, ti, e)
                             : d + (int64_t)e * a.ds_a;
                const uint32_t lead = (uint32_t)((4 - (reinterpret_cast<uintptr_t>(drow) & 3)) & 3);
                const uint32_t head = min(ti.vb, lead / EB);
                const uint32_t nw = (ti.vb - head) / V, tail = head + nw * V;
                if (threadIdx.x < head) drow[threadIdx.x] = elem(threadIdx.x, e);
                if (tail + threadIdx.x < ti.vb) drow[tail + threadIdx.x] = elem(tail + threadIdx.x, e);
                uint32_t* wrow = reinterpret_cast<uint32_t*>(drow + head);
                if (a.wrot_m == 0) {         // no rotation: constant element positions
                    for (uint32_t w = threadIdx.x; w < nw; w += kPanelThreads) {
                        uint32_t word = 0;
#pragma unroll
                        for (uint32_t k = 0; k < V; ++k)
                            word |= (uint32_t)elem(head + w * V + k, e) << (8 * EB * k);
                        wrow[w] = word;
                    }
                } else {
                    for (uint32_t w = threadIdx.x; w < nw; w += kPanelThreads) {
                        uint32_t word = 0;
#pragma unroll
                        for (uint32_t k = 0; k < V; ++k) {
                            const uint32_t kk = (k + rot) & (V - 1);
                            word |= (uint32_t)elem(head + w * V + kk, e) << (8 * EB * kk);
                        }
                        wrow[w] = word;
                    }
                }
            }
            return;
        }
        if (tb <= 16 && a.ds_a == (int64_t)tb && tb == a.ext_b && !a.merged && !AM) {
            // A short b axis packed in dst (planes -> interleaved channels): the tile's
            // dst is one run of va * tb elements, stored as 4-byte words; element f of
            // the run is (a, b) = (f / tb, f % tb).
            constexpr uint32_t V = 4 / EB;
            const uint32_t ssb16 = (uint32_t)((a.ss_b * EB) & 15);
            auto elem = [&](uint32_t f) {
                const uint32_t e = dev::div_u32(f, a.d_tb), b = f - e * tb;
                return *reinterpret_cast<const T*>(st + b * pitch + ((mis0 + b * ssb16) & 15) +
                                                   e * EB);
            };
            const uint32_t n = ti.va * tb;
            const uint32_t lead = (uint32_t)((4 - (reinterpret_cast<uintptr_t>(d) & 3)) & 3);
            const uint32_t head = min(n, lead / EB);
            const uint32_t nw = (n - head) / V, tail = head + nw * V;
            if (threadIdx.x < head) d[threadIdx.x] = elem(threadIdx.x);
            if (tail + threadIdx.x < n) d[tail + threadIdx.x] = elem(tail + threadIdx.x);
            uint32_t* wrun = reinterpret_cast<uint32_t*>(d + head);
            for (uint32_t w = threadIdx.x; w < nw; w += kPanelThreads) {
                uint32_t word = 0;
#pragma unroll
                for (uint32_t k = 0; k < V; ++k)
                    word |= (uint32_t)elem(head + w * V + k) << (8 * EB * k);
                wrun[w] = word;
            }
            return;
        }
    }
    if (kPanelThreads % tb == 0) {
        // each thread keeps one b and steps a by kPanelThreads / tb
        const uint32_t b = threadIdx.x % tb, de = kPanelThreads / tb;
        if (b >= ti.vb) return;
        const uint8_t* sp = rows ? st + stage_row<EB>(a, b) + mis(b) : st + mis0 + b * ta * EB;
        uint32_t e = threadIdx.x / tb;
        if constexpr (AM) {          // two-level dst offsets of a: one split per row
            T* dst = reinterpret_cast<T*>(a.dst) + b;
#pragma unroll 4
            for (; e < ti.va; e += de)
                dst[drow_off<AM>(a, ti, e)] = *reinterpret_cast<const T*>(sp + e * EB);
            return;
        }
        T* dp = d + b;
        const int64_t dstep = (int64_t)de * a.ds_a;
        dp += (int64_t)e * a.ds_a;
#pragma unroll 4
        for (; e < ti.va; e += de, dp += dstep) *dp = *reinterpret_cast<const T*>(sp + e * EB);
        return;
    }
    const uint32_t n = ta * tb;
#pragma unroll 4
    for (uint32_t f = threadIdx.x; f < n; f += kPanelThreads) {
        const uint32_t e = dev::div_u32(f, a.d_tb), b = f - e * tb;   // a, b in the tile
        if (e >= ti.va || b >= ti.vb) continue;
        const uint32_t off = rows ? stage_row<EB>(a, b) + mis(b) + e * EB : mis0 + (b * ta + e) * EB;
        T* drow = AM ? reinterpret_cast<T*>(a.dst) + drow_off<AM>(a, ti, e) : d + (int64_t)e * a.ds_a;
        drow[b] = *reinterpret_cast<const T*>(st + off);
    }
}

// The two store modes are separate kernels so that each keeps its own register
// budget (the element-store kernel fits four CTAs per SM).  The 1-byte run-store
// kernel with merged a (16 row addresses plus the row split per step) gets two CTAs
// per SM: at three it spilled (80 registers), and without the spill it measured
// 1.08-1.17x faster on GB300 (16^7 reversed u8 4.02 -> 4.68 TB/s, 24^6 reversed
// 3.10 -> 3.62).
template <int EB, bool VEC, bool AM>
__global__ void __launch_bounds__(kPanelThreads, (VEC && AM && EB == 1) ? 2 : VEC ? 3 : 4)
k_panel(const PanelArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t sbase = dev::smem_addr(smem);
    const uint32_t stage = (uint32_t)a.stage_bytes;
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < a.tiles ? (a.tiles - first + step - 1) / step : 0;

    // Every thread commits one group per tile slot (empty groups included), so
    // wait_group counts the same groups in every thread.
    for (int s = 0; s < kPanelStages - 1; ++s) {
        if (s < mine) issue<EB>(a, panel_tile<AM, EB != 1>(first + s * step, a), sbase + s * stage);
        cp_async_commit();
    }
    uint32_t slot = 0, ahead = kPanelStages - 1;    // stage of tile i and of tile i + S - 1
    for (int64_t i = 0; i < mine; ++i) {
        const int64_t nxt = i + kPanelStages - 1;
        if (nxt < mine) issue<EB>(a, panel_tile<AM, EB != 1>(first + nxt * step, a), sbase + ahead * stage);
        cp_async_commit();
        cp_async_wait<kPanelStages - 1>();           // tile i has landed (this thread's part)
        __syncthreads();                             // ... and every other thread's part
        drain<EB, VEC, AM>(a, panel_tile<AM, EB != 1>(first + i * step, a), smem + slot * stage);
        __syncthreads();                             // stage `slot` may be refilled
        slot = slot + 1 == kPanelStages ? 0 : slot + 1;
        ahead = ahead + 1 == kPanelStages ? 0 : ahead + 1;
    }
    cp_async_wait<0>();
    dev::cta_finish(a.cta_times);
}

// The panel transpose for block rows whose pitch TMA cannot take directly (a row
// pitch P that is not a multiple of 16 bytes, or an unaligned base): the rows
// b = j mod phi (phi = 16 / gcd(P, 16)) form a tensor of pitch phi * P, a multiple
// of 16, whose base is aligned down to 16 bytes; phase map j describes it.  One
// thread fills each stage with phi TMA tile loads, box (ta + 16 / EB) x (tb / phi)
// elements at x = a0 (a0 * EB is a multiple of 16 bytes), y = b0 / phi, landing as
// phi blocks of tb / phi rows of pitch ta * EB + 16 bytes; each row holds its
// elements at the row's own offset inside its first 16 bytes, exactly where the
// cp.async copy puts them, so the same drains read the stage (stage_row maps b to
// its phase block).  Completion is one mbarrier per stage; every thread waits on it
// with a bounded wait, and on expiry all of them stop, the status word records
// TL_ERR_TIMEOUT, and the loading thread waits (bounded) for its loads in flight
// before the CTA leaves.
template <int EB>
__global__ void __launch_bounds__(kPanelThreads, 4)
k_panel_tma(const __grid_constant__ PanelMaps maps, const PanelArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[kPanelStages];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const uint32_t stage = (uint32_t)a.stage_bytes;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPanelStages; ++s) dev::mbar_init(&full[s], 1);
        dev::fence_barrier_init();
    }
    __syncthreads();
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);
    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < a.tiles ? (a.tiles - first + step - 1) / step : 0;
    const uint32_t phi = 1u << a.phi_lg;
    const uint32_t box_bytes = ((uint32_t)a.ta * EB + 16) * ((uint32_t)a.tb >> a.phi_lg);
    auto load = [&](int64_t i, uint32_t s) {          // one thread: tile i into stage s
        const PanelTile ti = panel_tile<false, true>(first + i * step, a);
        dev::mbar_arrive_expect_tx(&full[s], phi * box_bytes);
        for (uint32_t j = 0; j < phi; ++j) {
            if (a.drop_load && i == 0 && j == 0) continue;   // test hook: the wait expires
            dev::tma_load(smem + s * stage + j * (uint32_t)a.phase_bytes, &maps.m[j], &full[s],
                          a.tma_rank, (int)ti.a0, (int)(ti.b0 >> a.phi_lg), ti.c[0], ti.c[1],
                          ti.c[2]);
        }
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
        for (; issued < kPanelStages - 1 && issued < mine; ++issued) load(issued, (uint32_t)issued);
    uint32_t slot = 0, ahead = kPanelStages - 1;
    int64_t i = 0;
    for (; i < mine; ++i) {
        const int64_t nxt = i + kPanelStages - 1;
        if (threadIdx.x == 0 && nxt < mine) {
            dev::fence_proxy_async_smem();          // the stage's last reads came before
            load(nxt, ahead);
            issued = nxt + 1;
        }
        const bool ok = dev::mbar_wait(&full[slot], (uint32_t)(i / kPanelStages) & 1u,
                                       (uint64_t)a.timeout_ns);
        if (__syncthreads_or(!ok)) break;           // every thread leaves together
        drain<EB, false, false>(a, panel_tile<false, true>(first + i * step, a), smem + slot * stage);
        __syncthreads();                            // stage `slot` may be refilled
        slot = slot + 1 == kPanelStages ? 0 : slot + 1;
        ahead = ahead + 1 == kPanelStages ? 0 : ahead + 1;
    }
    if (threadIdx.x == 0 && i < mine) {
        dev::report(a.status, TL_ERR_TIMEOUT);
        // do not leave while a load may still write this CTA's shared memory (a
        // longer bound than the wait that expired; past it the CTA leaves anyway)
        for (int64_t k = i; k < issued; ++k)
            dev::mbar_wait(&full[k % kPanelStages], (uint32_t)(k / kPanelStages) & 1u,
                           dev::kDrainFactor * (uint64_t)a.timeout_ns);
    }
    dev::cta_finish(a.cta_times);
}

// ---------------------------------------------------------------- the skew walk
// 1-byte elements whose dst rows (the columns a of the plane) sit at an odd pitch Pd:
// the dst rows start at offsets that differ modulo 16, so no walk of the tile rows
// gives 16-byte stores.  Instead each lane stores whole 16-byte-aligned pieces of dst
// rows: the piece of dst row x starting at tile row r is aligned when
// r = phase(x) (mod 16), and phase(x + 1) = phase(x) + delta with delta = -Pd mod 16,
// odd, so the 16 columns of a strip take each phase once.  A lane owns a strip of 16
// columns and a block of 16 tile rows; taking the columns in phase order, the
// piece of step k starts at row 16 * block + k: the rows the lane reads slide by one
// per step, a window of 16 stage rows of the strip kept in registers (31 rows read for
// 16 pieces).  The strips start e columns into the tile, e chosen so that the strip's
// first column has phase 0; both e and the phases stay the same from tile to tile (the
// tile sides are multiples of 16), so each tile owns the pieces starting in its rows,
// and the first tile of a plane row or column also stores the few elements before its
// first pieces.
//
// Stage: tile row r (0 .. kSkewRows + 14) holds the 16-byte blocks around its src
// bytes (columns 0 .. ta + 14) at r * pitch + 16 * (r / 16), each element at its src
// offset modulo 16, as the cp.async copy puts it; the lanes of a warp read rows 16
// apart, which the 16 bytes added per 16 rows put in distinct bank groups.  A row's 16
// columns of a strip are read as the two aligned 16-byte words around them and
// shifted into place in registers.

__host__ __device__ constexpr uint32_t inv16(uint32_t d) {           // the inverse of an odd d modulo 16
    uint32_t x = 1;
    while (((d * x) & 15u) != 1u) x += 2;
    return x;
}

__device__ __forceinline__ const PanelTile skew_tile(int64_t t, const PanelArgs& a) {
    return panel_tile<false, false>(t, a);
}

// Start the copies of one tile and its 15 extra rows and columns into the stage `sb`:
// thread t copies block k = t mod nblk of rows t / nblk, + rstep, + 2 rstep, ...
// (rstep = threads / nblk), so consecutive threads read consecutive blocks of a row.
__device__ __forceinline__ void issue_skew(const PanelArgs& a, const PanelTile& ti, uint32_t sb,
                                           uint32_t k, uint32_t r0, uint32_t rstep) {
    const uint32_t ncols = (uint32_t)min(a.ext_a - ti.a0, (int64_t)a.ta + 15);
    const uint32_t nrows = (uint32_t)min(a.ext_b - ti.b0, (int64_t)kSkewRows + 15);
    const uint32_t pitch = (uint32_t)a.pitch;
    const int64_t rowstep = (int64_t)rstep * a.ss_b;
    uintptr_t row = reinterpret_cast<uintptr_t>(a.src + ti.so + (int64_t)r0 * a.ss_b);
    for (uint32_t r = r0; r < nrows; r += rstep, row += rowstep)
        if (16 * k < (uint32_t)(row & 15) + ncols)       // block k holds a byte of the row
            cp_async16(sb + r * pitch + 16 * (r >> 4) + 16 * k, (row & ~uintptr_t(15)) + 16 * k);
}

// The tile's column phase: its strips start at column e (the first column of phase 0);
// mis0 is the offset modulo 16 of its first src element.
struct SkewPhase {
    uint32_t e, mis0;
};
template <uint32_t DELTA>
__device__ __forceinline__ SkewPhase skew_phase(const PanelArgs& a, const PanelTile& ti) {
    constexpr uint32_t DINV = inv16(DELTA);
    const uint32_t rho0 = (16u - ((uint32_t)reinterpret_cast<uintptr_t>(a.dst + ti.dof) & 15u)) & 15u;
    SkewPhase ph;
    ph.e = ((16u - rho0) * DINV) & 15u;
    ph.mis0 = (uint32_t)reinterpret_cast<uintptr_t>(a.src + ti.so) & 15u;
    return ph;
}

// Row c (0..30) of a lane's window, relative to the lane's first row: the byte offset
// of the aligned 16-byte word holding the row's strip column 0 (bits 0..23) and that
// column's offset inside it (bits 24..27); the same for every lane of the tile.
__device__ __forceinline__ uint32_t skew_row_entry(const PanelArgs& a, const SkewPhase& ph,
                                                   uint32_t c) {
    const uint32_t u = ((ph.mis0 + c * (uint32_t)a.vdelta) & 15u) + ph.e;       // 0 .. 30
    return (c * (uint32_t)a.pitch + 16 * (c >> 4) + (u & 16u)) | ((u & 15u) << 24);
}

// The first n < 16 bytes of a 16-byte piece (rows past the plane's end are not stored).
__device__ __noinline__ void skew_store_part(uint8_t* dp, uint32_t w0, uint32_t w1, uint32_t w2,
                                             uint32_t w3, uint32_t n) {
    for (uint32_t i = 0; i < n; ++i) {
        const uint32_t w = i < 4 ? w0 : i < 8 ? w1 : i < 12 ? w2 : w3;
        dp[i] = (uint8_t)(w >> (8 * (i & 3u)));
    }
}

// Store one landed tile (stage at shared-window offset st0) as 16-byte dst pieces;
// rowtab holds the tile's skew_row_entry values.
template <uint32_t DELTA>
__device__ __forceinline__ void drain_skew(const PanelArgs& a, const PanelTile& ti,
                                           const SkewPhase& ph, const uint32_t* rowtab,
                                           uint32_t st0) {
    constexpr uint32_t DINV = inv16(DELTA);
    extern __shared__ __align__(16) uint8_t smem_sk[];
    const uint32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t blk = lane & 15, strip = 2 * warp + (lane >> 4);
    const uint32_t ta = (uint32_t)a.ta, pitch = (uint32_t)a.pitch;
    uint8_t* const d = a.dst + ti.dof;
    const int64_t Pd = a.ds_a;
    const uint32_t e = ph.e;
    const uint32_t xlim = (uint32_t)min(a.ext_a - ti.a0, (int64_t)ta + 16);
    const uint32_t ylim = (uint32_t)min(a.ext_b - ti.b0, (int64_t)kSkewRows + 16);
    // the lane's 16 columns of stage row 16 * blk + c, in column order
    const uint32_t lbase = st0 + blk * (16 * pitch + 16) + 16 * strip;
    auto load_row = [&](uint32_t c, uint32_t (&w)[4]) {
        const uint32_t t = rowtab[c];
        const uint32_t off = lbase + (t & 0xFFFFFFu);
        const uint4 A = *reinterpret_cast<const uint4*>(&smem_sk[off]);
        const uint4 B = *reinterpret_cast<const uint4*>(&smem_sk[off + 16]);
        const uint32_t lo = t >> 24;
        const bool h2 = (lo & 8u) != 0, h1 = (lo & 4u) != 0;
        const uint32_t v[6] = {h2 ? A.z : A.x, h2 ? A.w : A.y, h2 ? B.x : A.z,
                               h2 ? B.y : A.w, h2 ? B.z : B.x, h2 ? B.w : B.y};
        uint32_t y[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) y[i] = h1 ? v[i + 1] : v[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __funnelshift_r(y[i], y[i + 1], 8 * (lo & 3u));
    };
    uint32_t W[16][4];
#pragma unroll
    for (uint32_t c = 0; c < 16; ++c) load_row(c, W[c]);
    const uint32_t x0 = e + 16 * strip;
    // the piece of step k is at dst + (x0 + j) * Pd + 16 * blk + k; from one step to the
    // next j grows by DINV, less 16 where it wraps
    const int64_t up = (int64_t)DINV * Pd + 1, wrap = ((int64_t)DINV - 16) * Pd + 1;
    uint8_t* dp = d + (int64_t)x0 * Pd + 16 * blk;
#pragma unroll
    for (uint32_t k = 0; k < 16; ++k) {
        // step k: column x0 + j of phase k, rows 16 * blk + k .. + 15 (window slots)
        const uint32_t j = (k * DINV) & 15u, wi = j >> 2, sel = (j & 3u) | (((j & 3u) + 4u) << 4);
        uint32_t o[4];
#pragma unroll
        for (uint32_t q = 0; q < 4; ++q) {
            const uint32_t t0 = __byte_perm(W[(k + 4 * q) & 15][wi], W[(k + 4 * q + 1) & 15][wi], sel);
            const uint32_t t1 = __byte_perm(W[(k + 4 * q + 2) & 15][wi], W[(k + 4 * q + 3) & 15][wi], sel);
            o[q] = __byte_perm(t0, t1, 0x5410);
        }
        const uint32_t r0 = 16 * blk + k;
        if (x0 + j < xlim && r0 < ylim) {
            if (r0 + 16 <= ylim)
                dev::stg128(dp, make_uint4(o[0], o[1], o[2], o[3]));
            else           // the last rows of the plane
                skew_store_part(dp, o[0], o[1], o[2], o[3], ylim - r0);
        }
        if (k < 15) {
            load_row(16 + k, W[k]);
            dp += ((((k + 1) * DINV) & 15u) > j) ? up : wrap;
        }
    }
}

// Elements no tile's pieces reach: the rows before each column's first piece (the
// plane's first row block), and the columns before the first strip (its first column
// block), element by element.  Tile t's coordinates are derived again here, so that the
// walk above holds none of them (the walk fits 128 registers a thread without spilling).
template <uint32_t DELTA>
__device__ __forceinline__ void drain_skew_edges(const PanelArgs& a, int64_t t, uint32_t st0) {
    extern __shared__ __align__(16) uint8_t smem_ed[];
    const PanelTile ti = skew_tile(t, a);
    const SkewPhase ph = skew_phase<DELTA>(a, ti);
    const uint32_t ta = (uint32_t)a.ta, pitch = (uint32_t)a.pitch, e = ph.e;
    const uint32_t ds16 = (uint32_t)a.vdelta;
    uint8_t* const d = a.dst + ti.dof;
    const int64_t Pd = a.ds_a;
    const uint32_t xlim = (uint32_t)min(a.ext_a - ti.a0, (int64_t)ta + 16);
    const uint32_t ylim = (uint32_t)min(a.ext_b - ti.b0, (int64_t)kSkewRows + 16);
    auto at = [&](uint32_t r, uint32_t x) -> uint8_t {
        return smem_ed[st0 + r * pitch + 16 * (r >> 4) + ((ph.mis0 + r * ds16) & 15u) + x];
    };
    if (ti.b0 == 0) {
        const uint32_t xs = ti.a0 == 0 ? 0u : e, xe = min(ta + e, xlim);
        const uint32_t nr = min(15u, ylim);
        if (xe > xs) {
            const uint32_t n = (xe - xs) * 16;
            for (uint32_t f = threadIdx.x; f < n; f += blockDim.x) {
                const uint32_t r = f & 15u, x = xs + (f >> 4);
                if (r < nr) d[(int64_t)x * Pd + r] = at(r, x);
            }
        }
    }
    if (ti.a0 == 0) {
        const uint32_t xe = min(e, xlim), nr = min((uint32_t)kSkewRows, ylim);
        const uint32_t n = xe * kSkewRows;
        for (uint32_t f = threadIdx.x; f < n; f += blockDim.x) {
            const uint32_t r = f % kSkewRows, x = f / kSkewRows;
            if (r < nr) d[(int64_t)x * Pd + r] = at(r, x);
        }
    }
}

// Persistent CTAs of 32 * warps threads, a ring of STAGES stages filled by cp.async
// (every thread copies part of each tile, then all wait and drain it).  One stage per
// CTA runs two CTAs per SM (at most 128 registers a thread), each loading while the
// other drains; two stages run one CTA per SM that loads the next tile while it drains.
template <uint32_t DELTA, int STAGES>
__global__ void __launch_bounds__(kPanelThreads, STAGES == 1 ? 2 : 1) k_panel_skew(const PanelArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ uint32_t rowtab[32];
    const uint32_t sbase = dev::smem_addr(smem);
    const uint32_t stage = (uint32_t)a.stage_bytes;
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);
    // (a CTA's tile count fits 32 bits: the grid is at most a few CTAs per SM)
    const uint32_t mine = blockIdx.x < a.tiles
        ? (uint32_t)((a.tiles - blockIdx.x + gridDim.x - 1) / gridDim.x) : 0u;
    auto tile_of = [&](uint32_t i) { return (int64_t)blockIdx.x + (int64_t)i * gridDim.x; };
    // this thread's copy block and first row (threads past rstep * nblk copy nothing),
    // derived again for each copy so that the walk holds none of it
    auto issue = [&](uint32_t i, uint32_t sb) {
        const uint32_t nblk = (uint32_t)a.nblk;
        const uint32_t r0 = dev::div_u32(threadIdx.x, a.d_nblk), k = threadIdx.x - r0 * nblk;
        const uint32_t rstep = dev::div_u32(blockDim.x, a.d_nblk);
        const uint32_t cr0 = r0 < rstep ? r0 : (uint32_t)kSkewRows + 16;
        issue_skew(a, skew_tile(tile_of(i), a), sb, k, cr0, rstep);
    };
    for (uint32_t s = 0; s < STAGES - 1; ++s) {
        if (s < mine) issue(s, sbase + s * stage);
        cp_async_commit();
    }
    uint32_t slot = 0, ahead = STAGES - 1;
    for (uint32_t i = 0; i < mine; ++i) {
        const uint32_t nxt = i + STAGES - 1;
        if (nxt < mine) issue(nxt, sbase + ahead * stage);
        cp_async_commit();
        const int64_t t = tile_of(i);
        const PanelTile ti = skew_tile(t, a);
        const SkewPhase ph = skew_phase<DELTA>(a, ti);
        const bool edge = ti.b0 == 0 || ti.a0 == 0;
        if (threadIdx.x < 31) rowtab[threadIdx.x] = skew_row_entry(a, ph, threadIdx.x);
        cp_async_wait<STAGES - 1>();
        __syncthreads();
        drain_skew<DELTA>(a, ti, ph, rowtab, slot * stage);
        if (edge) drain_skew_edges<DELTA>(a, t, slot * stage);
        __syncthreads();
        slot = slot + 1 == STAGES ? 0 : slot + 1;
        ahead = ahead + 1 == STAGES ? 0 : ahead + 1;
    }
    cp_async_wait<0>();
    dev::cta_finish(a.cta_times);
}

}  // namespace

// The planner takes TMA phase maps for 2-byte elements only (measured; the other
// widths fill the phase-major stage by cp.async).
const void* panel_tma_kernel(int eb) {
    return eb == 2 ? reinterpret_cast<const void*>(&k_panel_tma<2>) : nullptr;
}

cudaError_t launch_panel_tma(int eb, const PanelArgs& a, const PanelMaps& maps, int grid,
                             int smem, cudaStream_t st, bool pdl) {
    if (eb != 2) return cudaErrorInvalidValue;
    return launch_kernel(k_panel_tma<2>, dim3(grid), dim3(kPanelThreads), smem, st, pdl, maps, a);
}

namespace {
template <int EB, bool VEC>
const void* pick(bool am) {
    return am ? reinterpret_cast<const void*>(&k_panel<EB, VEC, true>)
              : reinterpret_cast<const void*>(&k_panel<EB, VEC, false>);
}
}  // namespace

const void* panel_kernel(int eb, bool vec, bool am) {
    switch (eb) {
    case 1: return vec ? pick<1, true>(am) : pick<1, false>(am);
    case 2: return vec ? pick<2, true>(am) : pick<2, false>(am);
    case 4: return vec ? pick<4, true>(am) : pick<4, false>(am);
    case 8: return vec ? pick<8, true>(am) : pick<8, false>(am);
    default: return pick<16, false>(am);
    }
}

namespace {
template <int STAGES>
const void* skew_pick(int delta) {
    switch (delta) {
    case 1: return reinterpret_cast<const void*>(&k_panel_skew<1, STAGES>);
    case 3: return reinterpret_cast<const void*>(&k_panel_skew<3, STAGES>);
    case 5: return reinterpret_cast<const void*>(&k_panel_skew<5, STAGES>);
    case 7: return reinterpret_cast<const void*>(&k_panel_skew<7, STAGES>);
    case 9: return reinterpret_cast<const void*>(&k_panel_skew<9, STAGES>);
    case 11: return reinterpret_cast<const void*>(&k_panel_skew<11, STAGES>);
    case 13: return reinterpret_cast<const void*>(&k_panel_skew<13, STAGES>);
    case 15: return reinterpret_cast<const void*>(&k_panel_skew<15, STAGES>);
    default: return nullptr;
    }
}
}  // namespace

const void* panel_skew_kernel(int delta, int stages) {
    return stages == 1 ? skew_pick<1>(delta) : stages == 2 ? skew_pick<2>(delta) : nullptr;
}

cudaError_t launch_panel_skew(const PanelArgs& a, int stages, int grid, int block, int smem,
                              cudaStream_t st, bool pdl) {
    using Kernel = void (*)(const PanelArgs);
    const Kernel k =
        reinterpret_cast<Kernel>(panel_skew_kernel((int)((16 - (a.ds_a & 15)) & 15), stages));
    if (!k || block <= 0 || block > kPanelThreads || block % 32 != 0) return cudaErrorInvalidValue;
    return launch_kernel(k, dim3(grid), dim3(block), smem, st, pdl, a);
}

cudaError_t launch_panel(int eb, const PanelArgs& a, int grid, int smem, cudaStream_t st,
                         bool pdl) {
    using Kernel = void (*)(const PanelArgs);
    const Kernel k = reinterpret_cast<Kernel>(panel_kernel(eb, a.vec != 0, a.amerged != 0));
    return launch_kernel(k, dim3(grid), dim3(kPanelThreads), smem, st, pdl, a);
}

}  // namespace tl
