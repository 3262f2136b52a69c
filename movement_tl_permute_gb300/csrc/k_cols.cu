// k_cols.cu -- transposes whose src runs along a are short (interleaved channels ->
// planes: pixels of A = 2..16 elements, A * EB <= 24 bytes, stored back to back).
//
// Plane: a (extent A, src stride 1, dst stride ds_a: one dst plane per a) by b (src
// stride A: the pixels are dense in src, dst stride 1), plus batch axes.  A unit is
// one 16-byte piece of every dst plane, the N = 16 / EB consecutive b it holds: its
// src is the N pixels' A * 16 contiguous bytes, which the thread loads as A 16-byte
// vectors (read-only path; the A loads of a warp share their cache lines), transposes
// in registers with byte permutes (plane c takes element c of every pixel) and stores
// as A 16-byte vectors, one per plane.  Consecutive threads take consecutive pieces,
// so each store instruction writes 512 contiguous bytes of one plane.  This mirrors
// the register transpose of k_rows.cu (short dst runs) for short src runs.  Element
// offsets follow the strided addressing of the TVM "Buffers and memory" page
// ("Declaring buffers").
#include "tl_kernels.h"

namespace tl {
namespace {

// Plane c's 16-byte piece from the A src vectors in w (A x 4 words, the N pixels
// back to back): its element p is src element p * A + c.
template <int EB, int A>
__device__ __forceinline__ uint4 plane_piece(const uint32_t (&w)[A][4], int c) {
    constexpr int N = 16 / EB;
    uint32_t o[4];
#pragma unroll
    for (int W = 0; W < 4; ++W) {
        if constexpr (EB >= 4) {
            // word W of the piece: element p = W * 4 / EB, its word q
            const int p = W * 4 / EB, q = W % (EB / 4);
            const int byte = (p * A + c) * EB + 4 * q;
            o[W] = w[byte / 16][(byte % 16) / 4];
        } else {
            int sv[4], sw[4], sb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int pb = 4 * W + i, p = pb / EB, e = pb % EB;
                const int byte = (p * A + c) * EB + e;
                sv[i] = byte / 16;
                sw[i] = (byte % 16) / 4;
                sb[i] = byte % 4;
            }
            const uint32_t t01 =
                __byte_perm(w[sv[0]][sw[0]], w[sv[1]][sw[1]], sb[0] | ((sb[1] + 4) << 4));
            const uint32_t t23 =
                __byte_perm(w[sv[2]][sw[2]], w[sv[3]][sw[3]], sb[2] | ((sb[3] + 4) << 4));
            o[W] = __byte_perm(t01, t23, 0x5410);
        }
    }
    static_assert(N * EB == 16, "a piece is 16 bytes");
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// unit u -> src element offset of its first pixel, dst element offset of its piece
// of plane 0
__device__ __forceinline__ void unit_offsets(int64_t u, const ColsArgs& a, int64_t& so,
                                             int64_t& d) {
    so = 0;
    d = 0;
    if (a.use32) {
        const uint32_t q = dev::div_u32((uint32_t)u, a.div_upp);
        const uint32_t col = (uint32_t)u - q * a.div_upp.d;
        so = (int64_t)col * a.n_px * a.A;
        d = (int64_t)col * a.n_px;
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
        int64_t item = u / a.upp;
        const int64_t col = u - item * a.upp;
        so = col * a.n_px * a.A;
        d = col * a.n_px;
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

template <int EB, int A>
__global__ void __launch_bounds__(kColsThreads) k_cols(const ColsArgs a) {
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    const int64_t step = (int64_t)gridDim.x * kColsThreads;
    for (int64_t u = (int64_t)blockIdx.x * kColsThreads + threadIdx.x; u < a.units; u += step) {
        int64_t so, d;
        unit_offsets(u, a, so, d);
        const uint8_t* s = a.src + so * EB;
        uint32_t w[A][4];
#pragma unroll
        for (int j = 0; j < A; ++j) {
            const uint4 v = dev::ldg128(s + 16 * j);
            w[j][0] = v.x;
            w[j][1] = v.y;
            w[j][2] = v.z;
            w[j][3] = v.w;
        }
        uint8_t* dp = a.dst + d * EB;
#pragma unroll
        for (int c = 0; c < A; ++c) dev::stg128(dp + (int64_t)c * a.ds_a * EB, plane_piece<EB, A>(w, c));
    }
}

template <int EB, int A>
cudaError_t go(const ColsArgs& a, int grid, cudaStream_t st, bool pdl) {
    return launch_kernel(k_cols<EB, A>, dim3(grid), dim3(kColsThreads), 0, st, pdl, a);
}

// pixels of A elements, A * EB <= 24 bytes
template <int EB>
cudaError_t go_eb(const ColsArgs& a, int grid, cudaStream_t st, bool pdl) {
    switch (a.A) {
    case 2: return go<EB, 2>(a, grid, st, pdl);
    case 3: return go<EB, 3>(a, grid, st, pdl);
    default: break;
    }
    if constexpr (EB <= 4) {
        switch (a.A) {
        case 4: return go<EB, 4>(a, grid, st, pdl);
        case 5: return go<EB, 5>(a, grid, st, pdl);
        case 6: return go<EB, 6>(a, grid, st, pdl);
        default: break;
        }
    }
    if constexpr (EB <= 2) {
        switch (a.A) {
        case 7: return go<EB, 7>(a, grid, st, pdl);
        case 8: return go<EB, 8>(a, grid, st, pdl);
        case 9: return go<EB, 9>(a, grid, st, pdl);
        case 10: return go<EB, 10>(a, grid, st, pdl);
        case 11: return go<EB, 11>(a, grid, st, pdl);
        case 12: return go<EB, 12>(a, grid, st, pdl);
        default: break;
        }
    }
    if constexpr (EB == 1) {
        switch (a.A) {
        case 13: return go<EB, 13>(a, grid, st, pdl);
        case 14: return go<EB, 14>(a, grid, st, pdl);
        case 15: return go<EB, 15>(a, grid, st, pdl);
        case 16: return go<EB, 16>(a, grid, st, pdl);
        default: break;
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_cols(int eb, const ColsArgs& a, int grid, cudaStream_t st, bool pdl) {
    switch (eb) {
    case 1: return go_eb<1>(a, grid, st, pdl);
    case 2: return go_eb<2>(a, grid, st, pdl);
    case 4: return go_eb<4>(a, grid, st, pdl);
    case 8: return go_eb<8>(a, grid, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tl
