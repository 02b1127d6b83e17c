// decode_static.cu -- the decode score + top-k call for callers that cannot
// allocate device memory.  Its scratch (per-sequence tickets, histograms,
// flags and the candidate buffer that idx_score_topk_decode keeps in the
// caller's workspace) lives in a fixed array in the library's own device
// memory instead, so the caller passes only inputs and outputs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dsaidx.h"
#include "internal.h"

namespace {

// Largest scratch a call may need; every GPU that loads the library holds this
// much device memory until the process exits.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch, per device and context.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// (with that device current) and cached together with the context it was
// looked up in: a context that was destroyed and created again on the device
// (cudaDeviceReset, for instance) has its module loaded anew, so a different
// current context looks the address up again.
std::mutex g_scratch_mu;
constexpr int kMaxDevices = 64;
struct ScratchAddr {
    CUcontext ctx = nullptr;
    void* addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    return fn;
}

idx_status scratch_of_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return IDX_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current();
    if (get == nullptr || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    ScratchAddr& e = g_scratch_addr[dev];
    if (e.addr == nullptr || e.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return IDX_ERR_CUDA;
        e.addr = p;
        e.ctx = ctx;
    }
    *out = e.addr;
    return IDX_OK;
}

}  // namespace

extern "C" idx_status idx_score_topk_decode_static(const idx_cache* cache, const void* q_bf16_dev,
                                                   const float* w_dev, const int32_t* block_table_dev,
                                                   int max_blocks_per_seq, const int32_t* seq_lens_dev,
                                                   int batch, int max_seq_len, int heads, int topk,
                                                   int32_t* out_idx_dev, float* out_score_dev, void* stream) {
    if (!cache) return IDX_ERR_INVALID_ARG;
    const size_t need = idx_workspace_bytes_decode(cache, batch, max_seq_len, heads, topk);
    if (need == 0)   // invalid or unsupported shape: the regular call reports which
        return idx_score_topk_decode(cache, q_bf16_dev, w_dev, block_table_dev, max_blocks_per_seq,
                                     seq_lens_dev, batch, max_seq_len, heads, topk, out_idx_dev,
                                     out_score_dev, nullptr, 0, stream);
    if (need > kStaticScratchBytes) return IDX_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    const idx_status s = scratch_of_current_device(&scratch);
    if (s != IDX_OK) return s;
    // The scratch keeps whatever the previous call left; the counters,
    // histograms and status word must start at zero, so clear the part used.
    if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return IDX_ERR_CUDA;
    return idx_score_topk_decode(cache, q_bf16_dev, w_dev, block_table_dev, max_blocks_per_seq, seq_lens_dev,
                                 batch, max_seq_len, heads, topk, out_idx_dev, out_score_dev, scratch, need,
                                 stream);
}
