// k_chunk.cu -- permutes whose innermost axis is contiguous on both sides.
//
// After canonicalisation the common stride-1 chain (the contiguous chunk of the
// TVM "copy_async -> dsmem" page, "Algorithm" step 1) is one row of `vpr`
// vectors of VB bytes; the remaining axes (in dst order) place each row.  A
// group of G = 2^log2g lanes copies one row; consecutive groups take consecutive
// rows, so a warp writes one contiguous run of dst.  A group takes U consecutive
// rows at a time: it decodes the first row's coordinates and steps the
// innermost outer axis for the others, and each lane keeps two vectors of each
// of the U rows in flight before it stores.
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

// Destination vector bytes for a source vector of VB bytes.
template <int CAST, int VB> struct DstVec {
    static constexpr int kBytes = VB / dev::Cast<CAST>::kSrc * dev::Cast<CAST>::kDst;
};
template <int VB> struct DstVec<TL_CAST_NONE, VB> { static constexpr int kBytes = VB; };

// The converted vector of a cast: the VB / ES source elements of v, each converted
// (ES, ED: source and destination element bytes).
template <int CAST, int VB>
__device__ __forceinline__ auto convert_vec(const typename Vec<VB>::T& v) {
    using C = dev::Cast<CAST>;
    constexpr int N = VB / C::kSrc, DVB = N * C::kDst;
    uint32_t in[(VB + 3) / 4] = {};
    __builtin_memcpy(in, &v, VB);
    uint32_t out[(DVB + 3) / 4] = {};
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const uint32_t x = C::kSrc == 4 ? in[k] : (in[k / 2] >> (16 * (k & 1))) & 0xFFFFu;
        const uint32_t y = C::cvt(x);
        if constexpr (C::kDst == 4) out[k] = y;
        else out[k / 2] |= y << (16 * (k & 1));
    }
    typename Vec<DVB>::T r;
    __builtin_memcpy(&r, out, DVB);
    return r;
}

// CAST (TL_CAST_*): each element converted on the way; VB is the source vector, the
// destination vector holds as many elements (row offsets are bytes of each side).
template <int VB, int CAST = TL_CAST_NONE>
__global__ void __launch_bounds__(256) k_chunk(const ChunkArgs a) {
    dev::grid_dependency_wait();
    dev::allow_dependent_launch();
    constexpr int U = 4;        // consecutive rows per group and round
    using T = typename Vec<VB>::T;
    constexpr int DVB = DstVec<CAST, VB>::kBytes;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t G = 1LL << a.log2g;
    const int64_t gid = gtid >> a.log2g;
    const int64_t lig = gtid & (G - 1);
    const int64_t ngroups = ((int64_t)gridDim.x * blockDim.x) >> a.log2g;
    // innermost outer axis: consecutive rows usually differ only there
    const int last = a.n - 1;
    const int64_t ext_last = a.n > 0 ? a.ext[last] : 1;
    const int64_t ss_last = a.n > 0 ? a.ss[last] : 0, ds_last = a.n > 0 ? a.ds[last] : 0;
    for (int64_t q = gid; q * U < a.rows; q += ngroups) {
        const int64_t r0 = q * U;
        int64_t so[U], d[U];
        bool ok[U];
        row_offsets(r0, a, so[0], d[0]);
        int64_t c_last = a.n > 0 ? r0 % ext_last : 0;
        ok[0] = true;
#pragma unroll
        for (int u = 1; u < U; ++u) {
            ok[u] = r0 + u < a.rows;
            if (c_last + 1 < ext_last) {            // step the innermost axis
                ++c_last;
                so[u] = so[u - 1] + ss_last;
                d[u] = d[u - 1] + ds_last;
            } else {                                // carry: decode afresh
                c_last = 0;
                so[u] = d[u] = 0;
                if (ok[u]) row_offsets(r0 + u, a, so[u], d[u]);
            }
        }
        // two vectors per lane and row: columns c0 and c0 + G
        for (int64_t c0 = lig; c0 < a.vpr; c0 += 2 * G) {
            const bool two = c0 + G < a.vpr;
            T v0[U], v1[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!ok[u]) continue;
                v0[u] = ld<VB>(a.src + so[u] + c0 * VB);
                if (two) v1[u] = ld<VB>(a.src + so[u] + (c0 + G) * VB);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!ok[u]) continue;
                if constexpr (CAST == TL_CAST_NONE) {
                    st<VB>(a.dst + d[u] + c0 * VB, v0[u]);
                    if (two) st<VB>(a.dst + d[u] + (c0 + G) * VB, v1[u]);
                } else {
                    st<DVB>(a.dst + d[u] + c0 * DVB, convert_vec<CAST, VB>(v0[u]));
                    if (two) st<DVB>(a.dst + d[u] + (c0 + G) * DVB, convert_vec<CAST, VB>(v1[u]));
                }
            }
        }
    }
}

}  // namespace

template <int VB>
cudaError_t launch_chunk(const ChunkArgs& a, int grid, int block, cudaStream_t st, bool pdl) {
    return launch_kernel(k_chunk<VB>, dim3(grid), dim3(block), 0, st, pdl, a);
}

// the cast kernels: source vectors of 4, 2 or 1 elements
cudaError_t launch_chunk_cast(int cast, int vb, const ChunkArgs& a, int grid, int block,
                              cudaStream_t st, bool pdl) {
#define TL_CC(C, V)                                                                        \
    if (cast == C && vb == V)                                                              \
        return launch_kernel(k_chunk<V, C>, dim3(grid), dim3(block), 0, st, pdl, a);
    TL_CC(TL_CAST_F32_TO_BF16, 16) TL_CC(TL_CAST_F32_TO_BF16, 8) TL_CC(TL_CAST_F32_TO_BF16, 4)
    TL_CC(TL_CAST_F32_TO_F16, 16) TL_CC(TL_CAST_F32_TO_F16, 8) TL_CC(TL_CAST_F32_TO_F16, 4)
    TL_CC(TL_CAST_BF16_TO_F32, 8) TL_CC(TL_CAST_BF16_TO_F32, 4) TL_CC(TL_CAST_BF16_TO_F32, 2)
    TL_CC(TL_CAST_F16_TO_F32, 8) TL_CC(TL_CAST_F16_TO_F32, 4) TL_CC(TL_CAST_F16_TO_F32, 2)
#undef TL_CC
    return cudaErrorInvalidValue;
}

template cudaError_t launch_chunk<1>(const ChunkArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_chunk<2>(const ChunkArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_chunk<4>(const ChunkArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_chunk<8>(const ChunkArgs&, int, int, cudaStream_t, bool);
template cudaError_t launch_chunk<16>(const ChunkArgs&, int, int, cudaStream_t, bool);

}  // namespace tl
