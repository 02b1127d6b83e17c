// ktimer.cu -- opt-in per-kernel timing of the score calls: CUDA events
// recorded on the call's stream before and after every kernel the calls
// launch, so that a benchmark can time each kernel of a multi-kernel call
// (the prefill scoring kernel apart from its row selection).  Off by default;
// a library utility, not part of the indexer's computation.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "dsaidx.h"
#include "internal.h"

namespace {

struct KernelTimer {
    std::mutex mu;
    std::vector<cudaEvent_t> ev;   // before/after pairs, in launch order
    size_t used = 0;
};
KernelTimer g_kt;

void destroy_all() {
    for (cudaEvent_t e : g_kt.ev) cudaEventDestroy(e);
    g_kt.ev.clear();
    g_kt.used = 0;
}

}  // namespace

namespace dsaidx {

void kt_mark(cudaStream_t st) {
    std::lock_guard<std::mutex> lock(g_kt.mu);
    if (g_kt.used < g_kt.ev.size()) cudaEventRecord(g_kt.ev[g_kt.used++], st);
}

}  // namespace dsaidx

extern "C" int idx_kernel_timing(int capacity) {
    std::lock_guard<std::mutex> lock(g_kt.mu);
    destroy_all();
    if (capacity <= 0) return 0;
    if (capacity > 4096) capacity = 4096;
    g_kt.ev.resize(static_cast<size_t>(capacity) * 2);
    for (size_t i = 0; i < g_kt.ev.size(); ++i) {
        if (cudaEventCreate(&g_kt.ev[i]) != cudaSuccess) {
            g_kt.ev.resize(i);
            destroy_all();
            return -1;
        }
    }
    return capacity;
}

extern "C" int idx_kernel_times(float* out_ms, int max) {
    std::lock_guard<std::mutex> lock(g_kt.mu);
    const int n = static_cast<int>(g_kt.used / 2);
    int w = 0;
    for (int i = 0; i < n && w < max; ++i) {
        if (cudaEventSynchronize(g_kt.ev[2 * i + 1]) != cudaSuccess) return -1;
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, g_kt.ev[2 * i], g_kt.ev[2 * i + 1]) != cudaSuccess) return -1;
        if (out_ms) out_ms[w] = ms;
        ++w;
    }
    g_kt.used = 0;
    return w;
}
