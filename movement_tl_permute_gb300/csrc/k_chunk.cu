// k_chunk.cu -- permutes whose innermost axis is contiguous on both sides.
//
// After canonicalisation the common stride-1 chain (the contiguous chunk of the
// TVM "copy_async -> dsmem" page, "Algorithm" step 1) is one row of `vpr`
// vectors of VB bytes; the remaining axes (in dst order) place each row.  A
// group of G = 2^log2g lanes copies one row; consecutive groups take consecutive
// rows, so a warp writes one contiguous run of dst.  Each thread keeps U rows in
// flight before it stores.
#include "tl_kernels.h"

namespace tl {
namespace {

template <int VB> struct Vec;
template <> struct Vec<1> { using T = uint8_t; };
template <> struct Vec<2> { using T = uint16_t; };
template <> struct Vec<4> { using T = uint32_t; };
template <> struct Vec<8> { using T = uint2; };
template <> struct Vec<16> { using T = uint4; };

template <int VB>
__device__ __forceinline__ typename Vec<VB>::T ld(const uint8_t* p) {
    if constexpr (VB == 16) return dev::ldg128(p);
    else return __ldg(reinterpret_cast<const typename Vec<VB>::T*>(p));
}

template <int VB>
__device__ __forceinline__ void st(uint8_t* p, const typename Vec<VB>::T& v) {
    if constexpr (VB == 16) dev::stg128(p, v);
    else *reinterpret_cast<typename Vec<VB>::T*>(p) = v;
}

// Byte offsets of row r on both sides.
__device__ __forceinline__ void row_offsets(int64_t r, const ChunkArgs& a, int64_t& so,
                                            int64_t& d) {
    so = 0;
    d = 0;
    if (a.use32) {
        uint32_t rem = (uint32_t)r;
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
#pragma unroll
        for (int i = TL_MAX_DIMS - 1; i >= 0; --i) {
            if (i < a.n) {
                const int64_t c = r % a.ext[i];
                r /= a.ext[i];
                so += c * a.ss[i];
                d += c * a.ds[i];
            }
        }
    }
}

template <int VB>
__global__ void __launch_bounds__(256) k_chunk(const ChunkArgs a) {
    constexpr int U = 4;
    using T = typename Vec<VB>::T;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t G = 1LL << a.log2g;
    const int64_t gid = gtid >> a.log2g;
    const int64_t lig = gtid & (G - 1);
    const int64_t ngroups = ((int64_t)gridDim.x * blockDim.x) >> a.log2g;
    for (int64_t row0 = gid; row0 < a.rows; row0 += ngroups * U) {
        int64_t so[U], d[U];
        bool ok[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = row0 + u * ngroups;
            ok[u] = r < a.rows;
            so[u] = d[u] = 0;
            if (ok[u]) row_offsets(r, a, so[u], d[u]);
        }
        for (int64_t c = lig; c < a.vpr; c += G) {
            T v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (ok[u]) v[u] = ld<VB>(a.src + so[u] + c * VB);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (ok[u]) st<VB>(a.dst + d[u] + c * VB, v[u]);
        }
    }
}

}  // namespace

template <int VB>
cudaError_t launch_chunk(const ChunkArgs& a, int grid, int block, cudaStream_t st) {
    k_chunk<VB><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

template cudaError_t launch_chunk<1>(const ChunkArgs&, int, int, cudaStream_t);
template cudaError_t launch_chunk<2>(const ChunkArgs&, int, int, cudaStream_t);
template cudaError_t launch_chunk<4>(const ChunkArgs&, int, int, cudaStream_t);
template cudaError_t launch_chunk<8>(const ChunkArgs&, int, int, cudaStream_t);
template cudaError_t launch_chunk<16>(const ChunkArgs&, int, int, cudaStream_t);

}  // namespace tl
