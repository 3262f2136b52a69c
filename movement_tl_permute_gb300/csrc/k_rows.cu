// k_rows.cu -- transposes whose dst runs along b are short (R * EB <= 16 bytes),
// such as the 4 x 32 scale-factor blocks of the TVM "permute_layout" page
// ("Demonstration program") stored as bytes.
//
// Plane: b (extent R, dst stride 1, src stride ss_b) by a (src stride 1, dst
// stride R: the plane is dense in dst), plus batch axes.  A unit is one 16-byte
// column piece of a (16/EB elements): the thread loads it from each of the R
// rows (R coalesced 16-byte loads), transposes the R x (16/EB) block in
// registers with byte permutes, and writes the R contiguous 16-byte vectors of
// dst the block maps to.  No shared memory is involved.
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

template <int EB, int R>
__global__ void __launch_bounds__(256) k_rows(const RowsArgs a) {
    constexpr int U = 2;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u0 < a.units;
         u0 += step * U) {
        uint4 in[U][R];
        int64_t dofs[U];
        bool ok[U];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
            const int64_t u = u0 + uu * step;
            ok[uu] = u < a.units;
            dofs[uu] = 0;
            if (ok[uu]) {
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
            if (!ok[uu]) continue;
            uint4 out[R];
            transpose_block<EB, R>(in[uu], out);
#pragma unroll
            for (int k = 0; k < R; ++k) dev::stg128(a.dst + dofs[uu] + 16 * k, out[k]);
        }
    }
}

template <int EB, int R>
cudaError_t go(const RowsArgs& a, int grid, int block, cudaStream_t st) {
    k_rows<EB, R><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rows(int eb, int r, const RowsArgs& a, int grid, int block, cudaStream_t st) {
    switch (eb * 100 + r) {
    case 102: return go<1, 2>(a, grid, block, st);
    case 104: return go<1, 4>(a, grid, block, st);
    case 108: return go<1, 8>(a, grid, block, st);
    case 116: return go<1, 16>(a, grid, block, st);
    case 202: return go<2, 2>(a, grid, block, st);
    case 204: return go<2, 4>(a, grid, block, st);
    case 208: return go<2, 8>(a, grid, block, st);
    case 402: return go<4, 2>(a, grid, block, st);
    case 404: return go<4, 4>(a, grid, block, st);
    case 802: return go<8, 2>(a, grid, block, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tl
