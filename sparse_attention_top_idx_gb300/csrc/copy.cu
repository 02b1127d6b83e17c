// copy.cu -- idx_copy: a copy kernel for staging a decode step's inputs and
// results between pinned host memory and the device (a library utility, not
// part of the indexer's computation).  On a GPU that reaches host memory over
// a coherent link, a kernel whose CTAs load 16-byte words of the host buffer
// moves a few hundred kilobytes much faster than the copy engine does, and it
// joins the score calls' programmatic launches: it may be scheduled while the
// previous kernel finishes and waits for it before touching memory.
#include <cuda_runtime.h>

#include "dsaidx.h"
#include "internal.h"

namespace {

__global__ void __launch_bounds__(256) copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                   int64_t n16) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

// The address a kernel uses for p: device memory as it is, mapped pinned host
// memory through its device alias, pageable host memory only where the device
// reads host page tables.  Null when a kernel cannot use p.
const void* device_view(const void* p, int dev) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    int pageable = 0;
    if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccessUsesHostPageTables, dev) != cudaSuccess)
        return nullptr;
    return pageable ? p : nullptr;
}

}  // namespace

extern "C" idx_status idx_copy(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return IDX_OK;
    if (!dst || !src || (reinterpret_cast<uintptr_t>(dst) & 15u) || (reinterpret_cast<uintptr_t>(src) & 15u) ||
        (bytes & 15u))
        return IDX_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IDX_ERR_CUDA;
    void* d = const_cast<void*>(device_view(dst, dev));
    const void* s = device_view(src, dev);
    if (!d || !s) return IDX_ERR_INVALID_ARG;
    const int64_t n16 = static_cast<int64_t>(bytes / 16);
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 2 * sms) blocks = 2 * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_kernel, static_cast<uint4*>(d), static_cast<const uint4*>(s), n16) ==
                   cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}
