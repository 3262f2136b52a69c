// k_block.cu -- permutes whose plane (src-contiguous axis a by dst-contiguous axis b)
// is too small for a useful tile: high-rank permutes of short axes (the `B.permute`
// of the TVM "Buffers and memory" page, "Buffer APIs", on tensors such as 12^7 or
// 9^8), where the rows a panel tile moves on one side are a few dozen bytes.
//
// The tile is up to four axes T chosen on the host so that it is a few long
// contiguous runs on both sides: the src run is the chain of T's axes from src
// stride 1, each of src stride the product of the extents before it, and the other
// axes of T index the src runs; the dst run and its index axes likewise from dst
// stride 1.  Each CTA runs a ring of kBlockStages shared-memory stages: every src run
// of a tile is copied as the aligned 16-byte blocks covering it (cp.async, landing at
// the run's own offset inside its first block), and while the copies of the next
// tiles fly, the landed tile is stored along its dst runs, consecutive threads
// writing consecutive dst addresses.  Per-CTA tables built once in shared memory turn
// (dst run j, position i) into (src run, position inside it) with adds only; the
// run pitch is chosen on the host by replaying the store walk's warp reads on the
// bank model of the TVM "permute_layout" page ("Algorithm", step 2).  Element
// offsets follow the strided addressing of "Buffers and memory", "Declaring buffers".
#include "tl_kernels.h"

namespace tl {
namespace {

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

// Copies of one tile into stage `slot`: the 16-byte blocks covering each valid src
// run; the first block's thread records where the run starts in the stage.
template <int EB>
__device__ __forceinline__ void block_issue(const BlockArgs& a, const BlockTile& ti,
                                            uint32_t sbase, const uint4* TR, uint32_t* RB) {
    const uintptr_t base = reinterpret_cast<uintptr_t>(a.src) + (uintptr_t)(ti.so * EB);
    const uint32_t ls = a.ls_inner == a.Ls ? (uint32_t)a.Ls : (uint32_t)a.ls_inner * ti.vc;
    const uint32_t nblk = (uint32_t)a.nblk, n = (uint32_t)a.Rs * nblk;
    for (uint32_t g = threadIdx.x; g < n; g += kBlockThreads) {
        const uint32_t r = dev::div_u32(g, a.d_nblk), k = g - r * nblk;
        const uint4 tr = TR[r];
        if (tr.z >= ti.vc) continue;                    // a run past the tile's chunk
        const int64_t soff = (int64_t)((uint64_t)tr.x | ((uint64_t)tr.y << 32));
        const uintptr_t run = base + (uintptr_t)(soff * EB);
        const uint32_t mis = (uint32_t)(run & 15);
        if (k == 0) RB[r] = r * (uint32_t)a.pitch + mis;
        if (k < ((mis + ls * EB + 15) >> 4))
            cp_async16(sbase + r * (uint32_t)a.pitch + 16 * k, (run & ~uintptr_t(15)) + 16 * k);
    }
}

// Stores one landed tile along its dst runs: element (j, i) of the tile's dst runs
// from the stage at RB[r_i + r_j] + (p_i + p_j) * EB, or, when every src run starts
// at the same offset inside its 16-byte block (umis), at mis0 + T_i + T_j with the
// tables holding r * pitch + p * EB.  Four elements per thread and step, so that
// their table and stage reads overlap.
template <int EB>
__device__ __forceinline__ void block_drain(const BlockArgs& a, const BlockTile& ti,
                                            const uint8_t* st, const uint2* TA, const uint4* TB,
                                            const uint32_t* RB) {
    using T = typename dev::Bits<EB>::T;
    constexpr uint32_t U = 4;
    T* d = reinterpret_cast<T*>(a.dst) + ti.dof;
    const uint32_t Ld = (uint32_t)a.Ld, n = Ld * (uint32_t)a.Rd;
    const uint32_t vc = ti.vc;
    const uint8_t* st0 = st + (reinterpret_cast<uintptr_t>(a.src + ti.so * EB) & 15);
    for (uint32_t f0 = threadIdx.x; f0 < n; f0 += U * kBlockThreads) {
#pragma unroll
        for (uint32_t u = 0; u < U; ++u) {
            const uint32_t f = f0 + u * kBlockThreads;
            if (f >= n) break;
            const uint32_t j = dev::div_u32(f, a.d_Ld), i = f - j * Ld;
            const uint2 ta = TA[i];
            const uint4 tb = TB[j];
            if ((ta.y >> 16) + (tb.y >> 16) >= vc) continue;   // past the tile's chunk
            const int64_t dofs = (int64_t)((uint64_t)tb.z | ((uint64_t)tb.w << 32));
            const uint8_t* sp;
            if (a.umis) {
                sp = st0 + ta.x + tb.x;
            } else {
                const uint32_t r = (ta.y & 0xffffu) + (tb.y & 0xffffu);
                sp = st + RB[r] + (ta.x + tb.x) * EB;
            }
            d[dofs + i] = *reinterpret_cast<const T*>(sp);
        }
    }
}

template <int EB>
__global__ void __launch_bounds__(kBlockThreads) k_block(const BlockArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const uint32_t sbase = dev::smem_addr(smem);
    const uint32_t stage = (uint32_t)a.stage_bytes;
    uint2* TA = reinterpret_cast<uint2*>(smem + a.table_off);
    uint4* TB = reinterpret_cast<uint4*>(TA + ((a.Ld + 1) & ~1));   // 16-byte aligned
    uint4* TR = reinterpret_cast<uint4*>(TB + a.Rd);
    uint32_t* RB = reinterpret_cast<uint32_t*>(TR + a.Rs);     // [kBlockStages][Rs]

    // the tables (from the arguments only: before the dependency wait)
    for (int32_t i = threadIdx.x; i < a.Ld; i += kBlockThreads) {
        int64_t x = i, sp = 0;
        uint32_t r = 0, c = 0;
        for (int k = 0; k < a.nd; ++k) {
            const int64_t dg = x % a.dext[k];
            x /= a.dext[k];
            sp += dg * a.dsp[k];
            r += (uint32_t)dg * (uint32_t)a.drs[k];
            if (k == a.dck) c = (uint32_t)dg;
        }
        TA[i] = make_uint2(a.umis ? r * (uint32_t)a.pitch + (uint32_t)sp * EB : (uint32_t)sp,
                           r | (c << 16));
    }
    for (int32_t j = threadIdx.x; j < a.Rd; j += kBlockThreads) {
        int64_t x = j, sp = 0, dofs = 0;
        uint32_t r = 0, c = 0;
        for (int k = 0; k < a.nj; ++k) {
            const int64_t dg = x % a.jext[k];
            x /= a.jext[k];
            sp += dg * a.jsp[k];
            r += (uint32_t)dg * (uint32_t)a.jrs[k];
            dofs += dg * a.jds[k];
            if (k == a.jck) c = (uint32_t)dg;
        }
        TB[j] = make_uint4(a.umis ? r * (uint32_t)a.pitch + (uint32_t)sp * EB : (uint32_t)sp,
                           r | (c << 16), (uint32_t)(uint64_t)dofs,
                           (uint32_t)((uint64_t)dofs >> 32));
    }
    for (int32_t r = threadIdx.x; r < a.Rs; r += kBlockThreads) {
        int64_t x = r, soff = 0;
        uint32_t c = 0;
        for (int k = 0; k < a.nr; ++k) {
            const int64_t dg = x % a.rext[k];
            x /= a.rext[k];
            soff += dg * a.rss[k];
            if (k == a.rck) c = (uint32_t)dg;
        }
        TR[r] = make_uint4((uint32_t)(uint64_t)soff, (uint32_t)((uint64_t)soff >> 32), c, 0u);
    }
    __syncthreads();
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);

    const int64_t first = blockIdx.x, step = gridDim.x;
    const int64_t mine = first < a.tiles ? (a.tiles - first + step - 1) / step : 0;
    // Every thread commits one group per tile slot (empty groups included), so
    // wait_group counts the same groups in every thread.
    for (int s = 0; s < kBlockStages - 1; ++s) {
        if (s < mine)
            block_issue<EB>(a, block_tile(first + s * step, a), sbase + s * stage, TR,
                            RB + s * a.Rs);
        cp_async_commit();
    }
    uint32_t slot = 0, ahead = kBlockStages - 1;
    for (int64_t i = 0; i < mine; ++i) {
        const int64_t nxt = i + kBlockStages - 1;
        if (nxt < mine)
            block_issue<EB>(a, block_tile(first + nxt * step, a), sbase + ahead * stage, TR,
                            RB + ahead * a.Rs);
        cp_async_commit();
        cp_async_wait<kBlockStages - 1>();           // tile i has landed (this thread's part)
        __syncthreads();                             // ... and every other thread's part
        block_drain<EB>(a, block_tile(first + i * step, a), smem + slot * stage, TA, TB,
                        RB + slot * a.Rs);
        __syncthreads();                             // stage `slot` may be refilled
        slot = slot + 1 == kBlockStages ? 0 : slot + 1;
        ahead = ahead + 1 == kBlockStages ? 0 : ahead + 1;
    }
    cp_async_wait<0>();
    dev::cta_finish(a.cta_times);
}

}  // namespace

int block_smem_bytes(const BlockArgs& a) {
    return a.table_off + 8 * ((a.Ld + 1) & ~1) + 16 * a.Rd + 16 * a.Rs + 4 * kBlockStages * a.Rs;
}

const void* block_kernel(int eb) {
    switch (eb) {
    case 1: return reinterpret_cast<const void*>(&k_block<1>);
    case 2: return reinterpret_cast<const void*>(&k_block<2>);
    case 4: return reinterpret_cast<const void*>(&k_block<4>);
    case 8: return reinterpret_cast<const void*>(&k_block<8>);
    default: return reinterpret_cast<const void*>(&k_block<16>);
    }
}

cudaError_t launch_block(int eb, const BlockArgs& a, int grid, cudaStream_t st, bool pdl) {
    const int smem = block_smem_bytes(a);
    switch (eb) {
    case 1: return launch_kernel(k_block<1>, dim3(grid), dim3(kBlockThreads), smem, st, pdl, a);
    case 2: return launch_kernel(k_block<2>, dim3(grid), dim3(kBlockThreads), smem, st, pdl, a);
    case 4: return launch_kernel(k_block<4>, dim3(grid), dim3(kBlockThreads), smem, st, pdl, a);
    case 8: return launch_kernel(k_block<8>, dim3(grid), dim3(kBlockThreads), smem, st, pdl, a);
    default: return launch_kernel(k_block<16>, dim3(grid), dim3(kBlockThreads), smem, st, pdl, a);
    }
}

}  // namespace tl
