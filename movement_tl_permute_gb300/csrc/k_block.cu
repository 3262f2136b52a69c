// k_block.cu -- permutes whose plane (src-contiguous axis a by dst-contiguous axis b)
// is too small for a useful tile: high-rank permutes of short axes (the `B.permute`
// of the TVM "Buffers and memory" page, "Buffer APIs", on tensors such as 12^7 or
// 9^8), where the rows a panel tile moves on one side are a few dozen bytes.
//
// The tile is up to four axes T chosen on the host so that it is a few long
// contiguous runs on both sides: the src run is the chain of T's axes from src
// stride 1, each of src stride the product of the extents before it, and the other
// axes of T index the src runs; the dst run and its index axes likewise from dst
// stride 1.
//
// Stage layout.  Every axis of T has a shared-memory byte stride: a src-run axis its
// src byte stride, a src-run index axis a stride the host picks congruent to its src
// byte stride modulo 16 (with room between runs for the 16-byte blocks around each).
// An element then sits in the stage at the same offset modulo 16 as in src, so each
// src run is one bulk copy of the aligned 16-byte blocks covering it, and the stage
// offset of element (dst run j, position i) is TA[i] + TB[j] from two per-CTA tables
// -- one add, whatever the runs' offsets inside their blocks.  The strides are chosen
// on the host by replaying the store walk's warp reads on the bank model of the TVM
// "permute_layout" page ("Algorithm", step 2).
//
// Pipelines.  A producer warp issues the bulk copies of each tile (its lanes take the
// runs in turn) into a ring of kBlockStages stages, completion counted on the stage's
// mbarrier; its consumer warps store each landed tile along its dst runs, each thread
// V consecutive dst elements per piece (one vector store when the dst runs allow it),
// in one of the walks the host picks (consecutive pieces in dst order, or groups of
// pieces across several dst runs).  A CTA runs one pipeline over its tiles in order, or
// two side by side that take its tiles from a shared counter.  Waits are bounded: a
// wait that expires reports TL_ERR_TIMEOUT, and the CTA leaves once its own copies have
// landed (or a longer bound has passed).  Element offsets follow the strided addressing
// of "Buffers and memory", "Declaring buffers".
#include "tl_kernels.h"

namespace tl {
namespace {

using dev::lds128;
using dev::lds32;
using dev::lds64;

// One bulk copy global -> this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t sdst, uintptr_t gsrc, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(sdst), "l"(gsrc), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint32_t lds8(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

constexpr uint32_t kEndRecord = 0xFFFFFFFFu;   // the vc of the record that ends a pipeline

struct BlockTile {
    int64_t so, dof;   // element offsets of the tile's origin in src and dst
    uint32_t vc;       // valid extent of the chunked axis in this tile
};

// tile t -> (chunk of the chunked axis, batch item): chunk fastest, then the batch
// axes innermost first
__device__ __forceinline__ BlockTile block_tile(int64_t t, const BlockArgs& a) {
    int64_t chunk, item;
    if (a.use32) {
        const uint32_t q = dev::div_u32((uint32_t)t, a.d_nc);
        chunk = (uint32_t)t - q * a.d_nc.d;
        item = q;
    } else {
        item = t / a.nc;
        chunk = t - item * a.nc;
    }
    BlockTile r;
    const int64_t c0 = chunk * a.c_k;
    r.so = c0 * a.c_ss;
    r.dof = c0 * a.c_ds;
    r.vc = (uint32_t)min((int64_t)a.c_k, a.c_ext - c0);
    for (int i = 0; i < a.nb; ++i) {
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
    }
    return r;
}

// A piece: V elements of EB bytes as 4-byte words (one word when V * EB < 4).
template <int EB, int V>
struct Piece {
    static constexpr int kWords = V * EB < 4 ? 1 : V * EB / 4;
    uint32_t w[kWords];
};

// Loads the V stage elements at sj + off[k] into a piece.
template <int EB, int V>
__device__ __forceinline__ void gather(Piece<EB, V>& pc, uint32_t sj, const uint32_t* off) {
    if constexpr (EB >= 4) {
#pragma unroll
        for (int k = 0; k < V; ++k) {
            if constexpr (EB == 16) {
                const uint4 x = lds128(sj + off[k]);
                pc.w[0] = x.x; pc.w[1] = x.y; pc.w[2] = x.z; pc.w[3] = x.w;
            } else if constexpr (EB == 8) {
                const uint2 x = lds64(sj + off[k]);
                pc.w[2 * k] = x.x;
                pc.w[2 * k + 1] = x.y;
            } else {
                pc.w[k] = lds32(sj + off[k]);
            }
        }
    } else {
        constexpr int kPer = 4 / EB;                  // elements per word
#pragma unroll
        for (int q = 0; q < Piece<EB, V>::kWords; ++q) {
            uint32_t x = 0;
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                if (q * kPer + e < V) {
                    const uint32_t y = EB == 2 ? lds16(sj + off[q * kPer + e])
                                               : lds8(sj + off[q * kPer + e]);
                    x |= y << (8 * EB * e);
                }
            }
            pc.w[q] = x;
        }
    }
}

// Stores a piece as one vector at p (aligned to V * EB bytes).
template <int EB, int V>
__device__ __forceinline__ void put(uint8_t* p, const Piece<EB, V>& pc) {
    if constexpr (V * EB == 16) {
        dev::stg128(p, make_uint4(pc.w[0], pc.w[1], pc.w[2], pc.w[3]));
    } else if constexpr (V * EB == 8) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pc.w[0], pc.w[1]);
    } else if constexpr (V * EB == 4) {
        *reinterpret_cast<uint32_t*>(p) = pc.w[0];
    } else if constexpr (V * EB == 2) {
        *reinterpret_cast<uint16_t*>(p) = (uint16_t)pc.w[0];
    } else {
        *p = (uint8_t)pc.w[0];
    }
}

// Bytes of a dst element: the source's, or the cast's target type's.
template <int EB, int CAST>
__host__ __device__ constexpr int dst_bytes() {
    if constexpr (CAST == TL_CAST_NONE) return EB;
    else return dev::Cast<CAST>::kDst;
}

// Loads the V stage elements at sj + off[k] (CAST's source type), converts each, and
// packs them as a piece of the destination type.
template <int CAST, int V>
__device__ __forceinline__ void gather_cast(Piece<dev::Cast<CAST>::kDst, V>& pc, uint32_t sj,
                                            const uint32_t* off) {
    using C = dev::Cast<CAST>;
    if constexpr (C::kDst == 2) {                   // fp32 -> 16-bit: two elements a word
#pragma unroll
        for (int q = 0; q < Piece<2, V>::kWords; ++q) {
            uint32_t x = C::cvt(lds32(sj + off[2 * q]));
            if (2 * q + 1 < V) x |= C::cvt(lds32(sj + off[2 * q + 1])) << 16;
            pc.w[q] = x;
        }
    } else {                                        // 16-bit -> fp32: one element a word
#pragma unroll
        for (int k = 0; k < V; ++k) pc.w[k] = C::cvt(lds16(sj + off[k]));
    }
}

// Where TA keeps dst-run position i: in order, except that for V >= 8 the four
// entries q of every piece sit at (q * W + piece) * 4, so that the lanes of a warp
// (consecutive pieces) read consecutive 16-byte words.
template <int V>
__device__ __forceinline__ uint32_t ta_slot(uint32_t i, uint32_t W) {
    if constexpr (V >= 8) {
        const uint32_t v = i / V, e = i - v * V;
        return ((e >> 2) * W + v) * 4 + (e & 3);
    } else {
        return i;
    }
}

// The V entries of TA of piece v (4-byte stage offsets).
template <int V>
__device__ __forceinline__ void load_offsets(uint32_t ta, uint32_t v, uint32_t W, uint32_t* off) {
    if constexpr (V >= 4) {
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const uint4 x = lds128(ta + 16 * (V >= 8 ? q * W + v : v));
            off[4 * q] = x.x;
            off[4 * q + 1] = x.y;
            off[4 * q + 2] = x.z;
            off[4 * q + 3] = x.w;
        }
    } else if constexpr (V == 2) {
        const uint2 x = lds64(ta + 8 * v);
        off[0] = x.x;
        off[1] = x.y;
    } else {
        off[0] = lds32(ta + 4 * v);
    }
}

template <int EB, int V, int CAST = TL_CAST_NONE>
__global__ void __launch_bounds__(32 * kBlockMaxWarps, 2) k_block(const BlockArgs a) {
    // dst element bytes (the cast's target type) and a piece of V of them
    constexpr int DEB = dst_bytes<EB, CAST>();
    using PieceT = Piece<DEB, V>;
    // loads piece v of a dst run from the stage (converting under a cast)
    auto load_piece = [](PieceT& pc, uint32_t sj, const uint32_t* off) {
        if constexpr (CAST == TL_CAST_NONE) gather<EB, V>(pc, sj, off);
        else gather_cast<CAST, V>(pc, sj, off);
    };
    extern __shared__ __align__(16) uint8_t smem[];
    // per pipeline: its ring's barriers and tile records (dof lo / hi, vc, origin mod 16)
    __shared__ __align__(8) uint64_t full_[kBlockMaxGroups][kBlockStages];
    __shared__ __align__(8) uint64_t empty_[kBlockMaxGroups][kBlockStages];
    __shared__ __align__(16) uint4 info_[kBlockMaxGroups][kBlockStages];
    __shared__ int32_t landed_[kBlockMaxGroups][kBlockStages];
    // bytes the copies of a whole tile move, by the tile origin's offset inside its
    // 16-byte block
    __shared__ uint32_t tot[16];
    __shared__ uint32_t next_tile;        // the CTA's tiles handed out so far
    const uint32_t stage = (uint32_t)a.stage_bytes;
    // this warp's pipeline: cw consumer warps and a producer warp, the pipelines side by
    // side in the CTA
    const int wpg = a.cw + 1;
    const int grp = (int)(threadIdx.x >> 5) / wpg;
    uint64_t* full = full_[grp];
    uint64_t* empty = empty_[grp];
    uint4* info = info_[grp];
    int32_t* landed = landed_[grp];
    const uint32_t sbase = dev::smem_addr(smem) + (uint32_t)grp * (uint32_t)a.ring_bytes;
    uint32_t* TA = reinterpret_cast<uint32_t*>(smem + a.table_off);       // [Ld, padded to 4]
    uint4* TB = reinterpret_cast<uint4*>(TA + ((a.Ld + 3) & ~3));        // [Rd]
    uint4* TR = TB + a.Rd;                                                // [Rs]
    const int warp = (int)(threadIdx.x >> 5) - grp * wpg, lane = threadIdx.x & 31;

    // the tables (from the arguments only: before the dependency wait)
    if (threadIdx.x < 16) tot[threadIdx.x] = 0;
    if (threadIdx.x == 0) next_tile = 0;
    __syncthreads();
    for (int32_t i = threadIdx.x; i < a.Ld; i += blockDim.x) {
        uint32_t x = (uint32_t)i, o = 0;
        for (int k = 0; k < a.nd; ++k) {
            const uint32_t q = x / (uint32_t)a.dext[k];
            o += (x - q * (uint32_t)a.dext[k]) * a.dsq[k];
            x = q;
        }
        TA[ta_slot<V>((uint32_t)i, (uint32_t)a.W)] = o;
    }
    for (int32_t j = threadIdx.x; j < a.Rd; j += blockDim.x) {
        uint32_t x = (uint32_t)j, o = 0, c = 0;
        int64_t dofs = 0;
        for (int k = 0; k < a.nj; ++k) {
            const uint32_t q = x / (uint32_t)a.jext[k];
            const uint32_t dg = x - q * (uint32_t)a.jext[k];
            x = q;
            o += dg * a.jsq[k];
            dofs += (int64_t)dg * a.jds[k];
            if (k == a.jck) c = dg;
        }
        dofs *= DEB;                                         // in bytes
        TB[j] = make_uint4(o, c, (uint32_t)(uint64_t)dofs, (uint32_t)((uint64_t)dofs >> 32));
    }
    for (int32_t r = threadIdx.x; r < a.Rs; r += blockDim.x) {
        uint32_t x = (uint32_t)r, o = 0, c = 0;
        int64_t sb = 0;
        for (int k = 0; k < a.nr; ++k) {
            const uint32_t q = x / (uint32_t)a.rext[k];
            const uint32_t dg = x - q * (uint32_t)a.rext[k];
            x = q;
            o += dg * a.rsq[k];
            sb += (int64_t)dg * a.rsb[k];
            if (k == a.rck) c = dg;
        }
        TR[r] = make_uint4((uint32_t)(uint64_t)sb, (uint32_t)((uint64_t)sb >> 32), o, c);
        for (uint32_t m = 0; m < 16; m += EB)
            atomicAdd(&tot[m], (((m + (uint32_t)sb) & 15) + (uint32_t)a.Ls * EB + 15) & ~15u);
    }
    if (threadIdx.x == 0) {
        for (int g = 0; g < a.groups; ++g)
            for (int s = 0; s < kBlockStages; ++s) {
                dev::mbar_init(&full_[g][s], 1);           // producer lane 0 arrives
                dev::mbar_init(&empty_[g][s], (uint32_t)a.cw);
            }
        dev::fence_barrier_init();
    }
    __syncthreads();
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);

    if (warp == a.cw) {
        // ---------------- producer: one bulk copy per src run ---------------------------
        // The CTA's tiles are blockIdx.x + k * gridDim.x; its pipelines take them in
        // turn from a shared counter (with one pipeline: in order), so that a pipeline
        // running slower takes fewer.  A tile past the end goes to the consumers as an
        // end record.
        uint32_t issued = 0;
        bool ok = true;
        for (;; ++issued) {
            const uint32_t use = issued / kBlockStages, s = issued - use * kBlockStages;
            if (use > 0) {
                const bool got = dev::mbar_wait(&empty[s], (use - 1) & 1, a.timeout_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                dev::fence_proxy_async_smem();   // the consumers' reads of the stage came first
            }
            uint32_t k = issued;                           // one pipeline: in order
            if (a.groups > 1) {
                if (lane == 0) k = atomicAdd(&next_tile, 1u);
                k = __shfl_sync(0xffffffffu, k, 0);
            }
            const int64_t t = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
            if (t >= a.tiles) {
                if (lane == 0) {
                    dev::sts128(dev::smem_addr(&info[s]), make_uint4(0, 0, kEndRecord, 0));
                    dev::mbar_arrive_expect_tx(&full[s], 0);
                }
                __syncwarp();
                ++issued;
                break;
            }
            const BlockTile ti = block_tile(t, a);
            const uintptr_t base = reinterpret_cast<uintptr_t>(a.src) + (uintptr_t)(ti.so * EB);
            const uint32_t tmis = (uint32_t)(base & 15);
            // bytes of a src run in this tile, and the runs inside its chunk
            const uint32_t len = (uint32_t)(a.ls_chunk ? a.ls_inner * ti.vc : a.Ls) * EB;
            const uint32_t rlim = a.rck >= 0 ? ti.vc : 0xffffffffu;
            const uint32_t sdst = sbase + s * stage + 16 + tmis;
            uint32_t bytes;
            if (ti.vc == (uint32_t)a.c_k) {
                bytes = tot[tmis];                         // a whole tile: every run, in full
            } else {
                uint32_t mine = 0;
                for (int32_t r = lane; r < a.Rs; r += 32) {
                    const uint4 tr = lds128(dev::smem_addr(&TR[r]));
                    if (tr.w < rlim) mine += (((tmis + tr.x) & 15) + len + 15) & ~15u;
                }
                bytes = __reduce_add_sync(0xffffffffu, mine);
            }
            if (lane == 0) {
                dev::sts128(dev::smem_addr(&info[s]),
                            make_uint4((uint32_t)(uint64_t)ti.dof,
                                       (uint32_t)((uint64_t)ti.dof >> 32), ti.vc, tmis));
                dev::mbar_arrive_expect_tx(&full[s], bytes);      // before any copy lands
            }
            __syncwarp();
            const uint32_t bar = dev::smem_addr(&full[s]);
            // the next run's table entry is read before this run's copy is issued
            int32_t r = lane;
            uint4 tr = make_uint4(0, 0, 0, 0);
            if (r < a.Rs) tr = lds128(dev::smem_addr(&TR[r]));
            while (r < a.Rs) {
                const int32_t rn = r + 32;
                uint4 trn = make_uint4(0, 0, 0, 0);
                if (rn < a.Rs) trn = lds128(dev::smem_addr(&TR[rn]));
                const bool drop = a.drop_load && issued == 0 && r == 0;   // test hook
                if (tr.w < rlim && !drop) {
                    const uintptr_t g = base + (uintptr_t)((uint64_t)tr.x | ((uint64_t)tr.y << 32));
                    const uint32_t mis = (uint32_t)(g & 15);
                    bulk_load(sdst + tr.z - mis, g - mis, (mis + len + 15) & ~15u, bar);
                }
                r = rn;
                tr = trn;
            }
        }
        if (!ok && lane == 0) dev::report(a.status, TL_ERR_TIMEOUT);
        // Do not leave while a copy may still write this CTA's shared memory (a longer
        // bound than the wait that expired; past it the CTA leaves anyway).
        for (uint32_t i = issued > kBlockStages ? issued - kBlockStages : 0; i < issued; ++i)
            dev::mbar_wait(&full[i % kBlockStages], (i / kBlockStages) & 1,
                           dev::kDrainFactor * a.timeout_ns);
        dev::cta_finish(a.cta_times);
        return;
    }

    // ---------------- consumers: store each tile along its dst runs ------------------
    // Two walks over the pieces (V dst elements each, W per dst run), picked on the host
    // with the bank model.  r_lg == 0: the consumer threads take consecutive pieces in
    // dst order (a warp's pieces run on into the next dst run).  r_lg > 0: a warp-step
    // takes a group of 32 >> r_lg consecutive pieces in each of 1 << r_lg consecutive
    // dst runs, whose stage reads spread over more banks (lane = (pl, rl)).
    const uint32_t W = (uint32_t)a.W, Rd = (uint32_t)a.Rd;
    const uint32_t GW = (uint32_t)a.GW, GR = (uint32_t)a.GR, cw = (uint32_t)a.cw;
    const uint32_t dgw = cw % GW, dgr = cw / GW;            // one step of the consumer warps
    const uint32_t pw_lg = 5 - (uint32_t)a.r_lg;
    const uint32_t pl = (uint32_t)lane & ((1u << pw_lg) - 1), rl = (uint32_t)lane >> pw_lg;
    const uint32_t ct = (uint32_t)warp * 32 + lane;         // 0 .. consumer threads - 1
    const uint32_t ta = dev::smem_addr(TA), tb = dev::smem_addr(TB);
    uint32_t it = 0;
    for (;; ++it) {
        const uint32_t use = it / kBlockStages, s = it - use * kBlockStages;
        // consumer warp 0 waits for the stage; the others sleep on a named barrier and
        // then take the completed phase themselves (one try, for its acquire)
        if (warp == 0) {
            const bool got = dev::mbar_wait(&full[s], use & 1, a.timeout_ns);
            if (lane == 0) landed[s] = got ? 1 : 0;
        }
        if (grp == 0)
            asm volatile("bar.sync 1, %0;" ::"r"(32 * cw) : "memory");
        else
            asm volatile("bar.sync 2, %0;" ::"r"(32 * cw) : "memory");
        if (!landed[s] || !dev::mbar_wait(&full[s], use & 1, a.timeout_ns)) {
            if (lane == 0) dev::report(a.status, TL_ERR_TIMEOUT);
            break;
        }
        const uint4 inf = lds128(dev::smem_addr(&info[s]));
        if (inf.z == kEndRecord) break;
        const int64_t dof = (int64_t)((uint64_t)inf.x | ((uint64_t)inf.y << 32));
        const uint32_t vc = inf.z;
        const uint32_t sb = sbase + s * stage + 16 + inf.w;
        // pieces of a dst run, and dst runs, inside this tile's chunk
        const uint32_t wlim = a.ld_chunk ? (uint32_t)a.ld_inner * vc / V : W;
        const uint32_t jlim = a.jck >= 0 ? vc : 0xffffffffu;
        uint8_t* dt = a.dst + dof * DEB;
        // stores piece v of dst run j (when inside the chunk) from its loaded parts
        auto store = [&](bool in, uint32_t v, const uint4& tj, const PieceT& pc) {
            if (in && v < wlim && tj.y < jlim)
                put<DEB, V>(dt + (int64_t)((uint64_t)tj.z | ((uint64_t)tj.w << 32)) + v * (V * DEB),
                           pc);
        };
        if (a.r_lg == 0) {
            // single elements: two pieces per step (the second repeats the first past
            // the last one, unstored), so that the table and stage reads of both are in
            // flight together (measured on GB300: 9^8 fp32 permutes 4.6 -> 5.7 TB/s;
            // wider pieces ran 0.8-1.0x as fast two at a time)
            const uint32_t step = 32 * cw;
            const uint32_t dv = step % W, dj = step / W;
            uint32_t v = ct % W, j = ct / W;
            while (j < Rd) {
                uint32_t v1 = v + dv, j1 = j + dj;             // the next piece
                if (v1 >= W) {
                    v1 -= W;
                    ++j1;
                }
                const uint4 t0 = lds128(tb + 16 * j);
                uint32_t o0[V];
                load_offsets<V>(ta, v, W, o0);
                PieceT p0;
                if constexpr (V == 1) {
                    const bool two = j1 < Rd;
                    const uint32_t vb = two ? v1 : v, jb = two ? j1 : j;
                    const uint4 t1 = lds128(tb + 16 * jb);
                    uint32_t o1[1];
                    load_offsets<1>(ta, vb, W, o1);
                    PieceT p1;
                    load_piece(p0, sb + t0.x, o0);
                    load_piece(p1, sb + t1.x, o1);
                    store(true, v, t0, p0);
                    store(two, vb, t1, p1);
                    if (two) {                                  // past the second piece
                        v1 += dv;
                        j1 += dj;
                        if (v1 >= W) {
                            v1 -= W;
                            ++j1;
                        }
                    }
                } else {
                    load_piece(p0, sb + t0.x, o0);
                    store(true, v, t0, p0);
                }
                v = v1;
                j = j1;
            }
        } else {
            uint32_t gw = (uint32_t)warp % GW, gr = (uint32_t)warp / GW;
            while (gr < GR) {
                uint32_t v = (gw << pw_lg) + pl, j = (gr << a.r_lg) + rl;
                const bool in = v < W && j < Rd;
                v = in ? v : 0;                                 // (table reads stay inside)
                j = in ? j : 0;
                const uint4 t0 = lds128(tb + 16 * j);
                uint32_t o0[V];
                load_offsets<V>(ta, v, W, o0);
                PieceT p0;
                load_piece(p0, sb + t0.x, o0);
                store(in, v, t0, p0);
                gw += dgw;
                gr += dgr;
                if (gw >= GW) {
                    gw -= GW;
                    ++gr;
                }
            }
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&empty[s]);
    }
    dev::cta_finish(a.cta_times);
}

using BlockFn = void (*)(const BlockArgs);

template <int EB>
BlockFn kernel_of(int v) {
    if constexpr (EB == 1) {
        switch (v) {
        case 16: return &k_block<1, 16>;
        case 8: return &k_block<1, 8>;
        case 4: return &k_block<1, 4>;
        case 2: return &k_block<1, 2>;
        default: return &k_block<1, 1>;
        }
    } else if constexpr (EB == 2) {
        switch (v) {
        case 8: return &k_block<2, 8>;
        case 4: return &k_block<2, 4>;
        case 2: return &k_block<2, 2>;
        default: return &k_block<2, 1>;
        }
    } else if constexpr (EB == 4) {
        switch (v) {
        case 4: return &k_block<4, 4>;
        case 2: return &k_block<4, 2>;
        default: return &k_block<4, 1>;
        }
    } else if constexpr (EB == 8) {
        return v == 2 ? &k_block<8, 2> : &k_block<8, 1>;
    } else {
        return &k_block<16, 1>;
    }
}

template <int CAST>
BlockFn cast_kernel_of(int v) {
    constexpr int SEB = dev::Cast<CAST>::kSrc;
    if constexpr (dev::Cast<CAST>::kDst == 2) {          // pieces of 1, 2, 4 or 8 16-bit elements
        switch (v) {
        case 8: return &k_block<SEB, 8, CAST>;
        case 4: return &k_block<SEB, 4, CAST>;
        case 2: return &k_block<SEB, 2, CAST>;
        default: return &k_block<SEB, 1, CAST>;
        }
    } else {                                            // pieces of 1, 2 or 4 fp32 elements
        switch (v) {
        case 4: return &k_block<SEB, 4, CAST>;
        case 2: return &k_block<SEB, 2, CAST>;
        default: return &k_block<SEB, 1, CAST>;
        }
    }
}

BlockFn block_fn(int eb, int v, int cast) {
    switch (cast) {
    case TL_CAST_F32_TO_BF16: return cast_kernel_of<TL_CAST_F32_TO_BF16>(v);
    case TL_CAST_F32_TO_F16: return cast_kernel_of<TL_CAST_F32_TO_F16>(v);
    case TL_CAST_BF16_TO_F32: return cast_kernel_of<TL_CAST_BF16_TO_F32>(v);
    case TL_CAST_F16_TO_F32: return cast_kernel_of<TL_CAST_F16_TO_F32>(v);
    default: break;
    }
    switch (eb) {
    case 1: return kernel_of<1>(v);
    case 2: return kernel_of<2>(v);
    case 4: return kernel_of<4>(v);
    case 8: return kernel_of<8>(v);
    default: return kernel_of<16>(v);
    }
}

}  // namespace

int block_smem_bytes(const BlockArgs& a) {
    return a.table_off + 4 * ((a.Ld + 3) & ~3) + 16 * a.Rd + 16 * a.Rs;
}

const void* block_kernel(int eb, int v, int cast) {
    return reinterpret_cast<const void*>(block_fn(eb, v, cast));
}

cudaError_t launch_block(int eb, const BlockArgs& a, int grid, cudaStream_t st, bool pdl) {
    return launch_kernel(block_fn(eb, a.V, a.cast), dim3(grid), dim3(32 * (a.cw + 1) * a.groups),
                         block_smem_bytes(a), st, pdl, a);
}

}  // namespace tl
