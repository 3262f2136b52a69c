// tile_common.cuh -- pieces shared by the TMA tile transpose (k_tile.cu) and its
// 2-CTA cluster variant (k_cluster.cu): the 128-byte swizzle address, the
// bank-conflict-free column reads of a 128 x 128-byte tile, the 16-byte run
// stores with ragged-edge masking, and the tile-order decode.
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
#pragma once

#include "tl_device.cuh"
#include "tl_kernels.h"

namespace tl {
namespace tile {

using namespace dev;

constexpr int kRows = 128;            // tile rows (b)
constexpr int kRowBytes = 128;        // tile row bytes (a)
constexpr int kTileBytes = kRows * kRowBytes;
constexpr int kConsumerWarps = 8;

// Byte address (relative to the tile) of byte `col` of row `row` under the
// 128-byte TMA swizzle: 16-byte chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t col) {
    return row * kRowBytes + ((((col >> 4) ^ row) & 7u) << 4) + (col & 15u);
}

template <typename T>
__device__ __forceinline__ void cswap(bool p, T& a, T& b) {
    T x = p ? b : a;
    T y = p ? a : b;
    a = x;
    b = y;
}

// Element e (EB bytes) of a 16-byte vector.
template <int EB>
__device__ __forceinline__ void store_elem(uint8_t* p, const uint4& v, int e) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (EB == 16) {
        *reinterpret_cast<uint4*>(p) = v;
    } else if constexpr (EB == 8) {
        *reinterpret_cast<uint2*>(p) = make_uint2(w[2 * e], w[2 * e + 1]);
    } else if constexpr (EB == 4) {
        *reinterpret_cast<uint32_t*>(p) = w[e];
    } else if constexpr (EB == 2) {
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
    } else {
        *p = (uint8_t)(w[e >> 2] >> (8 * (e & 3)));
    }
}

// Where one tile's columns land in dst, computed once per tile (by the producer
// of the single-CTA kernel, which publishes it through the stage's full barrier).
struct TileOut {
    uint8_t* base;       // dst byte address of the tile's element (a0, b0)
    int64_t cstride;     // bytes between consecutive columns a in dst
    int32_t cols, rows;  // valid columns (a) and rows (b) of this tile
    int32_t full;        // every column and row valid and 16-byte runs aligned
    int32_t vec;         // 16-byte runs aligned (else element-wise stores)
};

// Stores the 16-byte run of (16/EB) consecutive rows starting at tile row `row`
// of tile column `col`.
template <int EB>
__device__ __forceinline__ void put(const TileOut& o, int col, int row, const uint4& v) {
    constexpr int V = 16 / EB;
    uint8_t* p = o.base + (int64_t)col * o.cstride + row * EB;
    if (o.full) {                       // warp-uniform fast path: interior tile
        stg128(p, v);
        return;
    }
    if (col >= o.cols || row >= o.rows) return;
    if (o.vec && row + V <= o.rows) {
        stg128(p, v);
    } else {
#pragma unroll
        for (int e = 0; e < V; ++e)
            if (row + e < o.rows) store_elem<EB>(p + e * EB, v, e);
    }
}

// Consumer work for the 128-row block starting at tile row rb0 (a multiple of
// 128): every warp handles its share of the block.
template <int EB>
__device__ __forceinline__ void consume(uint32_t tile, const TileOut& o, int warp, int lane,
                                        int rb0);

template <>
__device__ __forceinline__ void consume<4>(uint32_t tile, const TileOut& o, int warp, int lane,
                                           int rb0) {
    // warp unit: 32 rows x 4 columns (one 16-byte chunk); 32 units per tile
    const int cw = lane & 3, g = lane >> 2, x = (lane >> 3) & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int col = 4 * cb + cw;
        const int row0 = rb0 + rb * 32 + 4 * g;
        uint32_t r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = lds32(tile + swz(row0 + (k ^ x), 4 * col));
        cswap(x & 1, r[0], r[1]);
        cswap(x & 1, r[2], r[3]);
        cswap(x & 2, r[0], r[2]);
        cswap(x & 2, r[1], r[3]);
        put<4>(o, col, row0, make_uint4(r[0], r[1], r[2], r[3]));
    }
}

template <>
__device__ __forceinline__ void consume<8>(uint32_t tile, const TileOut& o, int warp, int lane,
                                           int rb0) {
    // warp unit: 32 rows x 2 columns; half-warp wavefronts of 16 lanes
    const int cw = lane & 1, g = lane >> 1, x = (lane >> 3) & 1;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int col = 2 * cb + cw;
        const int row0 = rb0 + rb * 32 + 2 * g;
        uint2 r0 = lds64(tile + swz(row0 + x, 8 * col));
        uint2 r1 = lds64(tile + swz(row0 + (1 ^ x), 8 * col));
        cswap(x != 0, r0, r1);
        put<8>(o, col, row0, make_uint4(r0.x, r0.y, r1.x, r1.y));
    }
}

template <>
__device__ __forceinline__ void consume<16>(uint32_t tile, const TileOut& o, int warp, int lane,
                                           int rb0) {
    // warp unit: 32 rows x 1 column; quarter-warp wavefronts read 8 distinct chunks
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int row = rb0 + rb * 32 + lane;
        uint4 v = lds128(tile + swz(row, 16 * cb));
        put<16>(o, cb, row, v);
    }
}

template <>
__device__ __forceinline__ void consume<2>(uint32_t tile, const TileOut& o, int warp, int lane,
                                           int rb0) {
    // warp unit: 64 rows x 4 words (8 columns); 16 units per tile
    const int cw = lane & 3, g = lane >> 2, x = g;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int word = 4 * cb + cw;
        const int row0 = rb0 + rb * 64 + 8 * g;
        uint32_t r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) r[k] = lds32(tile + swz(row0 + (k ^ x), 4 * word));
#pragma unroll
        for (int k = 0; k < 8; k += 2) cswap(x & 1, r[k], r[k + 1]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (!(k & 2)) cswap(x & 2, r[k], r[k + 2]);
#pragma unroll
        for (int k = 0; k < 4; ++k) cswap(x & 4, r[k], r[k + 4]);
        uint4 lo, hi;
        lo.x = __byte_perm(r[0], r[1], 0x5410); hi.x = __byte_perm(r[0], r[1], 0x7632);
        lo.y = __byte_perm(r[2], r[3], 0x5410); hi.y = __byte_perm(r[2], r[3], 0x7632);
        lo.z = __byte_perm(r[4], r[5], 0x5410); hi.z = __byte_perm(r[4], r[5], 0x7632);
        lo.w = __byte_perm(r[6], r[7], 0x5410); hi.w = __byte_perm(r[6], r[7], 0x7632);
        put<2>(o, 2 * word, row0, lo);
        put<2>(o, 2 * word + 1, row0, hi);
    }
}

template <>
__device__ __forceinline__ void consume<1>(uint32_t tile, const TileOut& o, int warp, int lane,
                                           int rb0) {
    // warp unit: 128 rows x 4 words (16 columns); 8 units per tile, one per warp
    const int cw = lane & 3, g = lane >> 2, x = g;
    const int cb = warp;
    const int word = 4 * cb + cw;
    const int row0 = rb0 + 16 * g;
    uint32_t r[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) r[k] = lds32(tile + swz(row0 + (k ^ x), 4 * word));
#pragma unroll
    for (int k = 0; k < 16; k += 2) cswap(x & 1, r[k], r[k + 1]);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (!(k & 2)) cswap(x & 2, r[k], r[k + 2]);
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (!(k & 4)) cswap(x & 4, r[k], r[k + 4]);
    // 4x4 byte transposes: out[cc] word q = byte cc of rows 4q .. 4q+3
    uint32_t w[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t lo01 = __byte_perm(r[4 * q], r[4 * q + 1], 0x5140);
        const uint32_t lo23 = __byte_perm(r[4 * q + 2], r[4 * q + 3], 0x5140);
        const uint32_t hi01 = __byte_perm(r[4 * q], r[4 * q + 1], 0x7362);
        const uint32_t hi23 = __byte_perm(r[4 * q + 2], r[4 * q + 3], 0x7362);
        w[0][q] = __byte_perm(lo01, lo23, 0x5410);
        w[1][q] = __byte_perm(lo01, lo23, 0x7632);
        w[2][q] = __byte_perm(hi01, hi23, 0x5410);
        w[3][q] = __byte_perm(hi01, hi23, 0x7632);
    }
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
        put<1>(o, 4 * word + cc, row0, make_uint4(w[cc][0], w[cc][1], w[cc][2], w[cc][3]));
}

// ---------------------------------------------------------------------------
// Fused permute + cast: the same column reads, each element converted before the
// store.  N converted elements of DEB bytes go to tile column `col` from row `row`
// (words: the N elements packed little-endian).
template <int DEB, int N>
__device__ __forceinline__ void put_cast(const TileOut& o, int col, int row,
                                         const uint32_t (&w)[N * DEB / 4]) {
    uint8_t* p = o.base + (int64_t)col * o.cstride + row * DEB;
    if (o.full || (col < o.cols && o.vec && row + N <= o.rows)) {
        if constexpr (N * DEB == 8) {
            *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
        } else {
            stg128(p, make_uint4(w[0], w[1], w[2], w[3]));
            stg128(p + 16, make_uint4(w[4], w[5], w[6], w[7]));
        }
        return;
    }
    if (col >= o.cols) return;
#pragma unroll
    for (int e = 0; e < N; ++e) {
        if (row + e >= o.rows) break;
        if constexpr (DEB == 2)
            *reinterpret_cast<uint16_t*>(p + 2 * e) = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
        else
            *reinterpret_cast<uint32_t*>(p + 4 * e) = w[e];
    }
}

// Column reads of consume<4> (four rows of one fp32 column per lane), converted to
// four 16-bit elements: 8 bytes per lane and column.
template <int CAST>
__device__ __forceinline__ void consume_narrow(uint32_t tile, const TileOut& o, int warp,
                                               int lane, int rb0) {
    const int cw = lane & 3, g = lane >> 2, x = (lane >> 3) & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int col = 4 * cb + cw;
        const int row0 = rb0 + rb * 32 + 4 * g;
        uint32_t r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) r[k] = lds32(tile + swz(row0 + (k ^ x), 4 * col));
        cswap(x & 1, r[0], r[1]);
        cswap(x & 1, r[2], r[3]);
        cswap(x & 2, r[0], r[2]);
        cswap(x & 2, r[1], r[3]);
        const uint32_t w[2] = {Cast<CAST>::cvt(r[0]) | (Cast<CAST>::cvt(r[1]) << 16),
                               Cast<CAST>::cvt(r[2]) | (Cast<CAST>::cvt(r[3]) << 16)};
        put_cast<2, 4>(o, col, row0, w);
    }
}

// Column reads of consume<2> (eight rows of two 16-bit columns per lane), converted
// to fp32: 32 bytes per lane and column.
template <int CAST>
__device__ __forceinline__ void consume_widen(uint32_t tile, const TileOut& o, int warp,
                                              int lane, int rb0) {
    const int cw = lane & 3, g = lane >> 2, x = g;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = warp + kConsumerWarps * i;
        const int cb = u & 7, rb = u >> 3;
        const int word = 4 * cb + cw;
        const int row0 = rb0 + rb * 64 + 8 * g;
        uint32_t r[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) r[k] = lds32(tile + swz(row0 + (k ^ x), 4 * word));
#pragma unroll
        for (int k = 0; k < 8; k += 2) cswap(x & 1, r[k], r[k + 1]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (!(k & 2)) cswap(x & 2, r[k], r[k + 2]);
#pragma unroll
        for (int k = 0; k < 4; ++k) cswap(x & 4, r[k], r[k + 4]);
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            lo[k] = Cast<CAST>::cvt(r[k] & 0xFFFFu);
            hi[k] = Cast<CAST>::cvt(r[k] >> 16);
        }
        put_cast<4, 8>(o, 2 * word, row0, lo);
        put_cast<4, 8>(o, 2 * word + 1, row0, hi);
    }
}

// Tile t -> (ta, tb, batch coordinates).  Within a batch item tiles are visited in
// groups of `group_b` tile rows, b fastest inside a group, so concurrently
// running CTAs write runs of many 128-byte lines (one group spanning all of b
// makes the writes one front-to-back stream).
// Every coordinate is a TMA box coordinate, so each fits in 32 bits.
struct TileCoord {
    int32_t ta, tb;
    int32_t bc[3];
};

__device__ __forceinline__ TileCoord tile_coord(int64_t t, const TileArgs& a) {
    TileCoord r;
    if (a.use32) {
        // the same decode with 32-bit division by invariant integers
        const uint32_t t32 = (uint32_t)t;
        uint32_t item = div_u32(t32, a.d_item);
        const uint32_t local = t32 - item * a.d_item.d;
        const uint32_t grp = div_u32(local, a.d_grp);
        const uint32_t first_tb = grp * a.d_gfull.d;
        const uint32_t in_grp = local - grp * a.d_grp.d;
        const bool last = first_tb + a.d_gfull.d > (uint32_t)a.tiles_b;
        const DivU32& dg = last ? a.d_glast : a.d_gfull;
        const uint32_t ta = div_u32(in_grp, dg);
        r.ta = ta;
        r.tb = first_tb + (in_grp - ta * dg.d);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const uint32_t q = div_u32(item, a.d_bext[i]);
            r.bc[i] = item - q * a.d_bext[i].d;
            item = q;
        }
        return r;
    }
    const int64_t per_item = a.tiles_a * a.tiles_b;
    int64_t item = t / per_item;
    const int64_t local = t - item * per_item;
    const int64_t grp = local / (a.group_b * a.tiles_a);
    const int64_t first_tb = grp * a.group_b;
    const int64_t gsize = min(a.group_b, a.tiles_b - first_tb);
    const int64_t in_grp = local - grp * a.group_b * a.tiles_a;
    r.tb = (int32_t)(first_tb + in_grp % gsize);
    r.ta = (int32_t)(in_grp / gsize);
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        r.bc[i] = 0;
        if (i < a.nbatch) {
            r.bc[i] = (int32_t)(item % a.bext[i]);
            item /= a.bext[i];
        }
    }
    return r;
}

// Destination record of the tile at coordinates tc (tiles of TB rows; DEB: the
// destination element bytes, EB's unless the permute converts).
template <int EB, int TB = kRows, int DEB = EB>
__device__ __forceinline__ TileOut make_out(const TileCoord& tc, const TileArgs& a) {
    constexpr int TA = kRowBytes / EB;
    const int64_t a0 = tc.ta * TA, b0 = tc.tb * TB;
    int64_t base = a0 * a.ds_a + b0;
#pragma unroll
    for (int i = 0; i < 3; ++i) base += tc.bc[i] * a.bds[i];
    TileOut o;
    o.base = a.dst + base * DEB;
    o.cstride = a.ds_a * DEB;
    o.cols = (int32_t)min((int64_t)TA, a.ext_a - a0);
    o.rows = (int32_t)min((int64_t)TB, a.ext_b - b0);
    o.vec = a.vec_store;
    o.full = (o.vec && o.cols == TA && o.rows == TB) ? 1 : 0;
    return o;
}

// The record of a tile as one 16-byte word (the producer stores it with one aligned
// 16-byte store, each consumer warp reads it with one 16-byte load): the dst
// address, then valid columns (bits 0-8), valid rows (9-17) and "full" (bit 18).
// The column stride and the run alignment are the same for every tile.
template <int EB, int TB = kRows, int DEB = EB>
__device__ __forceinline__ uint4 pack_out(const TileCoord& tc, const TileArgs& a) {
    const TileOut o = make_out<EB, TB, DEB>(tc, a);
    const uint64_t p = reinterpret_cast<uint64_t>(o.base);
    return make_uint4((uint32_t)p, (uint32_t)(p >> 32),
                      (uint32_t)o.cols | ((uint32_t)o.rows << 9) | ((uint32_t)o.full << 18), 0u);
}

template <int DEB>
__device__ __forceinline__ TileOut unpack_out(const uint4 v, const TileArgs& a) {
    TileOut o;
    o.base = reinterpret_cast<uint8_t*>((uint64_t)v.x | ((uint64_t)v.y << 32));
    o.cstride = a.ds_a * DEB;
    o.cols = (int32_t)(v.z & 511u);
    o.rows = (int32_t)((v.z >> 9) & 511u);
    o.full = (int32_t)((v.z >> 18) & 1u);
    o.vec = a.vec_store;
    return o;
}

}  // namespace tile
}  // namespace tl
