// k_warp.cu -- the warp register-staged permute of the TVM "permute_layout" page
// ("Algorithm", step 3), one warp tile per batch item.
//
// A tile holds 32 * P elements.  In iteration r lane l handles iteration index
// j = r ^ ((l >> shift) & mask), whose coordinates are the row-major
// decomposition of l + 32 * j over the tile extent: phase 1 reads all P elements
// through the src strides into registers, the warp synchronises, phase 2 writes
// them through the dst strides, and the warp synchronises again.  The (shift,
// mask) pair comes from the host bank simulator so that both phases are
// shared-memory bank-conflict-free, and because every read of a tile precedes its
// writes the kernel is correct in place (src == dst, equal per-tile footprints).
#include "tl_kernels.h"
#include "../../include/tl_permute_device.cuh"

namespace tl {
namespace {

template <int EB, int P>
__global__ void __launch_bounds__(128, 4) k_warp(const WarpArgs a) {
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    using T = typename dev::Bits<EB>::T;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    tl_dev::WarpTile ts, td;
    ts.n = td.n = a.tn;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ts.ext[i] = td.ext[i] = (int32_t)(i < a.tn ? a.text[i] : 1);
        ts.str[i] = i < a.tn ? a.tss[i] : 0;
        td.str[i] = i < a.tn ? a.tds[i] : 0;
    }
    const T* src = reinterpret_cast<const T*>(a.src);
    T* dst = reinterpret_cast<T*>(a.dst);
    for (int64_t item = gw; item < a.items; item += nw) {
        int64_t sb = 0, db = 0, rem = item;
#pragma unroll
        for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
            if (i < a.bn) {
                const int64_t c = rem % a.bext[i];
                rem /= a.bext[i];
                sb += c * a.bss[i];
                db += c * a.bds[i];
            }
        }
        // phase 1 reads via src strides, warp barrier, phase 2 writes via dst strides
        tl_dev::warp_permute_layout<P>(dst + db, src + sb, ts, td, a.shift, a.mask);
    }
}

template <int EB, int P>
cudaError_t go(const WarpArgs& a, int grid, int block, cudaStream_t st, bool pdl) {
    return launch_kernel(k_warp<EB, P>, dim3(grid), dim3(block), 0, st, pdl, a);
}

template <int EB>
cudaError_t by_p(int P, const WarpArgs& a, int grid, int block, cudaStream_t st, bool pdl) {
    switch (P) {
    case 1: return go<EB, 1>(a, grid, block, st, pdl);
    case 2: return go<EB, 2>(a, grid, block, st, pdl);
    case 4: return go<EB, 4>(a, grid, block, st, pdl);
    case 8: return go<EB, 8>(a, grid, block, st, pdl);
    case 16: if constexpr (EB <= 8) return go<EB, 16>(a, grid, block, st, pdl); break;
    case 32: if constexpr (EB <= 4) return go<EB, 32>(a, grid, block, st, pdl); break;
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_warp(int eb, int P, const WarpArgs& a, int grid, int block, cudaStream_t st,
                        bool pdl) {
    switch (eb) {
    case 1: return by_p<1>(P, a, grid, block, st, pdl);
    case 2: return by_p<2>(P, a, grid, block, st, pdl);
    case 4: return by_p<4>(P, a, grid, block, st, pdl);
    case 8: return by_p<8>(P, a, grid, block, st, pdl);
    case 16: return by_p<16>(P, a, grid, block, st, pdl);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tl
