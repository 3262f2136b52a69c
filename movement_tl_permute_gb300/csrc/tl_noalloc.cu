// tl_noalloc.cu -- tl_permute_tile_noalloc: the TMA tile transpose for callers
// that cannot allocate device memory.
//
// The tile kernel's only scratch is a 4-byte status word that it writes when
// one of its bounded waits expires.  tl_permute_ex takes that word from the
// caller (opts.dev_status), which means a cudaMalloc somewhere.  This entry point
// instead keeps the word in a file-scope __device__ array that lives as long as
// the library is loaded, so a call allocates nothing.
//
// The array's name is a host-side stand-in in host code, not a device address:
// its device address is fetched once per device with cudaGetSymbolAddress (the
// first call on each device does this set-up, with that device current) and then
// passed to the kernel.  The address is kept for the life of the process, so the
// entry point is not for use on a device after a cudaDeviceReset of it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tl_permute.h"

namespace {

static __device__ __align__(256) int32_t g_tile_scratch[TL_NOALLOC_SCRATCH_BYTES / 4];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use).
int scratch_address(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tile_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return TL_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return TL_OK;
}

}  // namespace

extern "C" TL_API int tl_permute_tile_noalloc(const void* src, void* dst, int ndim,
                                              const int64_t* shape, const int64_t* src_strides,
                                              const int64_t* dst_strides, int elem_bytes,
                                              tl_stream_t stream, int32_t* host_status) {
    // Scratch this launch needs: the tile kernel's single status word.
    const size_t needed = sizeof(int32_t);
    if (needed > TL_NOALLOC_SCRATCH_BYTES) return TL_ERR_BOUNDS;

    // Validate and plan first (host only), so a rejected call touches no device state.
    // The plan is cached: the launch below reuses it instead of planning again.
    tl_plan_info info;
    tl_permute_opts opts{};
    opts.flags = TL_PATH_TILE;
    int rc = tl_plan(src, dst, ndim, shape, src_strides, dst_strides, elem_bytes, &opts, &info);
    if (rc != TL_OK) return rc;

    int32_t* status = nullptr;
    rc = scratch_address(&status);
    if (rc != TL_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, needed, st) != cudaSuccess) return TL_ERR_CUDA;
    opts.dev_status = status;
    rc = tl_permute_ex(src, dst, ndim, shape, src_strides, dst_strides, elem_bytes, stream, &opts);
    if (rc != TL_OK) return rc;
    if (host_status &&
        cudaMemcpyAsync(host_status, status, needed, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return TL_ERR_CUDA;
    return TL_OK;
}
