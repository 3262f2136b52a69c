// k_generic.cu -- the correctness floor: any layout pair, one element per step, or
// 16 bytes of dst per step when dst's innermost axis is contiguous (gathers from
// strided views).
//
// Flat index f runs over the canonical shape in dst order (axes sorted by dst
// stride, so consecutive threads write neighbouring elements); its coordinates
// are decoded with per-axis divisions and applied to both stride vectors
// (offset = sum c[i] * stride[i], TVM docs "Buffers and memory", "Declaring
// buffers").
#include "tl_kernels.h"

namespace tl {
namespace {

// CK: the checked run -- each element's byte ranges are compared with the buffer
// sizes first; an element outside is skipped and TL_ERR_BOUNDS recorded.
// CAST (TL_CAST_*): each element converted on the way (EB is the source's width;
// dst offsets count destination elements).
template <int EB, int VM, bool CK, int CAST = TL_CAST_NONE>
__global__ void __launch_bounds__(256) k_generic(const GenericArgs a) {
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t f = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; f < a.total; f += step) {
        int64_t so = 0, d = 0;
        if (a.use32) {
            uint32_t rem = (uint32_t)f;
#pragma unroll
            for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
                if (i < a.n) {
                    const uint32_t q = dev::div_u32(rem, a.div[i]);
                    const uint32_t c = rem - q * a.div[i].d;
                    rem = q;
                    so += (int64_t)c * a.ss[i];
                    d += (int64_t)c * a.ds[i];
                }
            }
        } else {
            int64_t rem = f;
#pragma unroll
            for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
                if (i < a.n) {
                    const int64_t c = rem % a.ext[i];
                    rem /= a.ext[i];
                    so += c * a.ss[i];
                    d += c * a.ds[i];
                }
            }
        }
        if constexpr (CK) {
            const bool in = (a.src_bytes <= 0 || (so + 1) * EB <= a.src_bytes) &&
                            (a.dst_bytes <= 0 || (d + 1) * EB <= a.dst_bytes);
            if (!in) {
                dev::report(a.status, TL_ERR_BOUNDS);
                continue;
            }
        }
        if constexpr (CAST != TL_CAST_NONE) {
            using C = dev::Cast<CAST>;
            const uint32_t x = C::kSrc == 4 ? *reinterpret_cast<const uint32_t*>(a.src + so * 4)
                                            : *reinterpret_cast<const uint16_t*>(a.src + so * 2);
            const uint32_t y = C::cvt(x);
            if constexpr (C::kDst == 4) *reinterpret_cast<uint32_t*>(a.dst + d * 4) = y;
            else *reinterpret_cast<uint16_t*>(a.dst + d * 2) = (uint16_t)y;
        } else if constexpr (VM == 0) {
            dev::copy_elem<EB>(a.dst + d * EB, a.src + so * EB);
        } else {
            using T = typename dev::Bits<EB>::T;
            constexpr int V = 16 / EB;
            union {
                uint4 v;
                T e[V];
            } u;
            // gather V strided elements, one 16-byte store
#pragma unroll
            for (int k = 0; k < V; ++k)
                u.e[k] = *reinterpret_cast<const T*>(a.src + (so + k * a.vstep) * EB);
            dev::stg128(a.dst + d * EB, u.v);
        }
    }
}

}  // namespace

template <int EB>
cudaError_t launch_generic(const GenericArgs& a, int grid, int block, cudaStream_t st, bool pdl) {
    if (a.checked)
        return launch_kernel(k_generic<EB, 0, true>, dim3(grid), dim3(block), 0, st, pdl, a);
    if constexpr (EB < 16) {
        if (a.vmode == 1)
            return launch_kernel(k_generic<EB, 1, false>, dim3(grid), dim3(block), 0, st, pdl, a);
    }
    return launch_kernel(k_generic<EB, 0, false>, dim3(grid), dim3(block), 0, st, pdl, a);
}

cudaError_t launch_generic_cast(int cast, const GenericArgs& a, int grid, int block,
                               cudaStream_t st, bool pdl) {
    switch (cast) {
    case TL_CAST_F32_TO_BF16:
        return launch_kernel(k_generic<4, 0, false, TL_CAST_F32_TO_BF16>, dim3(grid), dim3(block),
                             0, st, pdl, a);
    case TL_CAST_F32_TO_F16:
        return launch_kernel(k_generic<4, 0, false, TL_CAST_F32_TO_F16>, dim3(grid), dim3(block),
                             0, st, pdl, a);
    case TL_CAST_BF16_TO_F32:
        return launch_kernel(k_generic<2, 0, false, TL_CAST_BF16_TO_F32>, dim3(grid), dim3(block),
                             0, st, pdl, a);
    case TL_CAST_F16_TO_F32:
        return launch_kernel(k_generic<2, 0, false, TL_CAST_F16_TO_F32>, dim3(grid), dim3(block),
                             0, st, pdl, a);
    }
    return cudaErrorInvalidValue;
}

template cudaError_t launch_generic<1>(const GenericArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_generic<2>(const GenericArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_generic<4>(const GenericArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_generic<8>(const GenericArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_generic<16>(const GenericArgs&, int, int, cudaStream_t, bool);

}  // namespace tl
