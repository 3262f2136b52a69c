// k_rows.cu -- transposes whose dst runs along b are short (R * EB <= 16 bytes, any
// R >= 2),
// such as the 4 x 32 scale-factor blocks of the TVM "permute_layout" page
// ("Demonstration program") stored as bytes.
//
// Plane: b (extent R, dst stride 1, src stride ss_b) by a (src stride 1, dst
// stride R: the plane is dense in dst), plus batch axes.  A unit is one 16-byte
// column piece of a (16/EB elements): the thread loads it from each of the R
// rows (16-byte loads that use whole sectors), transposes the R x (16/EB) block
// in registers with byte permutes into the R contiguous 16-byte vectors of dst
// the block maps to, and parks them in a per-warp shared-memory stage.  The
// warp then stores the stage back lane by lane, so each store instruction
// writes 512 contiguous bytes whenever consecutive units are adjacent in dst
// (always within a plane, and across planes when the batch is dense).
#include "tl_kernels.h"

namespace tl {
namespace {

// out (R vectors) = in (R rows of 16 bytes) transposed: output element
// f = v * R + b takes row b's element v.
template <int EB, int R>
__device__ __forceinline__ void transpose_block(const uint4 (&in)[R], uint4 (&out)[R]) {
    uint32_t w[R][4];
#pragma unroll
    for (int b = 0; b < R; ++b) {
        w[b][0] = in[b].x; w[b][1] = in[b].y; w[b][2] = in[b].z; w[b][3] = in[b].w;
    }
    uint32_t o[4 * R];
    if constexpr (EB >= 4) {
        constexpr int WPE = EB / 4;          // words per element
#pragma unroll
        for (int W = 0; W < 4 * R; ++W) {
            const int f = W / WPE, q = W % WPE, v = f / R, b = f % R;
            o[W] = w[b][v * WPE + q];
        }
    } else {
#pragma unroll
        for (int W = 0; W < 4 * R; ++W) {
            int sw[4], sb[4], row[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = 4 * W + i, f = p / EB, e = p % EB, v = f / R, b = f % R;
                const int j = v * EB + e;
                row[i] = b;
                sw[i] = j >> 2;
                sb[i] = j & 3;
            }
            const uint32_t t01 = __byte_perm(w[row[0]][sw[0]], w[row[1]][sw[1]],
                                             sb[0] | ((sb[1] + 4) << 4));
            const uint32_t t23 = __byte_perm(w[row[2]][sw[2]], w[row[3]][sw[3]],
                                             sb[2] | ((sb[3] + 4) << 4));
            o[W] = __byte_perm(t01, t23, 0x5410);
        }
    }
#pragma unroll
    for (int k = 0; k < R; ++k) out[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
}

__device__ __forceinline__ void unit_offsets(int64_t u, const RowsArgs& a, int64_t& so,
                                             int64_t& d, int64_t& col) {
    int64_t item;
    so = 0;
    d = 0;
    if (a.use32) {
        const uint32_t q = dev::div_u32((uint32_t)u, a.div_upr);
        col = (int64_t)((uint32_t)u - q * a.div_upr.d);
        uint32_t rem = q;
#pragma unroll
        for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
            if (i < a.n) {
                const uint32_t qq = dev::div_u32(rem, a.div[i]);
                const uint32_t c = rem - qq * a.div[i].d;
                rem = qq;
                so += (int64_t)c * a.ss[i];
                d += (int64_t)c * a.ds[i];
            }
        }
    } else {
        item = u / a.upr;
        col = u - item * a.upr;
#pragma unroll
        for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
            if (i < a.n) {
                const int64_t c = item % a.ext[i];
                item /= a.ext[i];
                so += c * a.ss[i];
                d += c * a.ds[i];
            }
        }
    }
}

// Shared-memory staging of a warp's output: for R a power of two, 16-byte chunk c
// is kept at c ^ (((c >> 3) ^ (c >> 6)) & 7), which spreads both the per-lane writes
// (chunks lane*R + k) and the contiguous read-back (chunks 32*i + lane) over
// distinct bank groups in every 8-lane wavefront; R = 12 keeps c ^ ((c >> 3) & 7)
// (2-way writes, 4-way without).  Other R keep c: an odd stride R already gives 8
// lanes 8 distinct bank groups, and for R = 6, 10, 14 no swizzle of these forms does
// better than the plain 2-way.
template <int R>
__device__ __forceinline__ uint32_t stage_chunk(uint32_t c) {
    if constexpr ((R & (R - 1)) == 0) return c ^ (((c >> 3) ^ (c >> 6)) & 7u);
    if constexpr (R % 4 == 0) return c ^ ((c >> 3) & 7u);
    return c;
}

// Block size and units in flight per thread: the 16-row variant keeps one unit
// of 256 bytes in registers and a 32 KiB stage for 4 warps.
template <int R> __host__ __device__ constexpr int rows_threads() { return R >= 16 ? 128 : 256; }
template <int R> __host__ __device__ constexpr int rows_units() { return R >= 8 ? 1 : 2; }

template <int EB, int R>
__global__ void __launch_bounds__(rows_threads<R>()) k_rows(const RowsArgs a) {
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    dev::cta_start(a.cta_times);
    constexpr int U = rows_units<R>();
    constexpr int kWarps = rows_threads<R>() / 32;
    __shared__ __align__(16) uint4 stage[kWarps][32 * R];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t stage_base = dev::smem_addr(&stage[warp][0]);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    const int64_t gwarp = (int64_t)blockIdx.x * kWarps + warp;
    // Each round a warp takes U groups of 32 consecutive units (warp-uniform loop).
    for (int64_t base = gwarp * 32 * U; base < a.units; base += nwarps * 32 * U) {
        uint4 in[U][R];
        int64_t dofs[U];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            const int64_t u = base + uu * 32 + lane;
            dofs[uu] = -1;
            if (u < a.units) {
                int64_t so, d, col;
                unit_offsets(u, a, so, d, col);
                const uint8_t* s = a.src + so * EB + col * 16;
#pragma unroll
                for (int b = 0; b < R; ++b) in[uu][b] = dev::ldg128(s + b * a.ss_b * EB);
                dofs[uu] = d * EB + col * 16 * R;
            }
        }
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            if (base + uu * 32 >= a.units) break;          // warp-uniform
            uint4 out[R];
            transpose_block<EB, R>(in[uu], out);
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const uint4 v = out[k];
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 stage_base + 16 * stage_chunk<R>(lane * R + k)),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
            }
            __syncwarp();
            // store chunk 32*i + lane: unit (32*i + lane) / R of this group, piece k
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int c = 32 * i + lane;
                const int64_t d = __shfl_sync(0xffffffffu, dofs[uu], c / R);
                const uint4 v = dev::lds128(stage_base + 16 * stage_chunk<R>(c));
                if (d >= 0) dev::stg128(a.dst + d + 16 * (c % R), v);
            }
            __syncwarp();
        }
    }
    dev::cta_finish(a.cta_times);
}

template <int EB, int R>
cudaError_t go(const RowsArgs& a, int grid, int block, cudaStream_t st, bool pdl) {
    if (block != rows_threads<R>()) return cudaErrorInvalidValue;
    return launch_kernel(k_rows<EB, R>, dim3(grid), dim3(block), 0, st, pdl, a);
}

}  // namespace

cudaError_t launch_rows(int eb, int r, const RowsArgs& a, int grid, int block, cudaStream_t st,
                        bool pdl) {
    switch (eb * 100 + r) {
    case 102: return go<1, 2>(a, grid, block, st, pdl);
    case 103: return go<1, 3>(a, grid, block, st, pdl);
    case 104: return go<1, 4>(a, grid, block, st, pdl);
    case 105: return go<1, 5>(a, grid, block, st, pdl);
    case 106: return go<1, 6>(a, grid, block, st, pdl);
    case 107: return go<1, 7>(a, grid, block, st, pdl);
    case 108: return go<1, 8>(a, grid, block, st, pdl);
    case 109: return go<1, 9>(a, grid, block, st, pdl);
    case 110: return go<1, 10>(a, grid, block, st, pdl);
    case 111: return go<1, 11>(a, grid, block, st, pdl);
    case 112: return go<1, 12>(a, grid, block, st, pdl);
    case 113: return go<1, 13>(a, grid, block, st, pdl);
    case 114: return go<1, 14>(a, grid, block, st, pdl);
    case 115: return go<1, 15>(a, grid, block, st, pdl);
    case 116: return go<1, 16>(a, grid, block, st, pdl);
    case 202: return go<2, 2>(a, grid, block, st, pdl);
    case 203: return go<2, 3>(a, grid, block, st, pdl);
    case 204: return go<2, 4>(a, grid, block, st, pdl);
    case 205: return go<2, 5>(a, grid, block, st, pdl);
    case 206: return go<2, 6>(a, grid, block, st, pdl);
    case 207: return go<2, 7>(a, grid, block, st, pdl);
    case 208: return go<2, 8>(a, grid, block, st, pdl);
    case 402: return go<4, 2>(a, grid, block, st, pdl);
    case 403: return go<4, 3>(a, grid, block, st, pdl);
    case 404: return go<4, 4>(a, grid, block, st, pdl);
    case 802: return go<8, 2>(a, grid, block, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tl
