// decode.cu -- launch of the fused decode score + top-k kernel: a grid of
// persistent 8-CTA thread-block clusters that take the batch's sequence
// segments in turn (decode_kernel.cuh).
#include <mutex>

#include "decode_kernel.cuh"

namespace dsaidx {

namespace {

constexpr int kMaxDevices = 64;

// A kernel of the decode kernel's shape (threads, registers, dynamic shared
// memory) that allocates no TMEM: the occupancy calculator counts one CTA per
// SM for a kernel that allocates TMEM, while two CTAs of 128 TMEM columns
// each do share an SM (measured on GB300), so clusters are counted on this
// stand-in.
__global__ void __maxnreg__(120) decode_shape_probe(int* sink) {
    if (sink) sink[threadIdx.x] = 0;
}

struct ClusterFit {
    std::mutex mu;
    int n[kMaxDevices] = {};
};

// Clusters of the decode shape that fit on the device at once (queried once
// per device and key format, like the shared-memory limit, so that later
// calls -- including calls captured into a graph -- make no runtime query).
cudaError_t resident_clusters(int smem, int dev, ClusterFit& fit, int* out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(fit.mu);
    int* cached = fit.n;
    if (cached[dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(decode_shape_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kDecCl, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kDecCl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, decode_shape_probe, &cfg);
        if (e != cudaSuccess) return e;
        cached[dev] = n > 0 ? n : 1;
    }
    *out = cached[dev];
    return cudaSuccess;
}

template <bool kFp8, int kBs>
cudaError_t launch_decode_t(const idx_cache* c, const ScoreParams& p, int64_t units_bound, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    static ClusterFit clusters;
    const DecPlan plan = dec_plan(kFp8);
    auto kern = decode_kernel<kFp8, kBs>;
    cudaError_t e = set_smem_once(kern, plan.total, attr_done);
    if (e != cudaSuccess) return e;
    int fit = 1;
    e = resident_clusters(plan.total, c->device, clusters, &fit);
    if (e != cudaSuccess) return e;
    // persistent clusters: at most those that fit at once (and never more
    // than the workspace's slow-path scratch provides for)
    int64_t g = units_bound < fit ? units_bound : fit;
    if (g > kDecMaxClusters(c->num_sms)) g = kDecMaxClusters(c->num_sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(g) * kDecCl, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.total);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kDecCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the set-up may overlap the previous kernel (the kernel waits for it,
    // griddepcontrol.wait, before it reads anything that kernel writes)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    kt_mark(st);
    e = cudaLaunchKernelEx(&cfg, kern, c->tmap, p);
    kt_mark(st);
    return e;
}

}  // namespace

// Segments of the longest sequence; every sequence takes at most that many
// units (an empty or invalid one takes one).
DecodeGeom decode_geometry(const idx_cache* c, int batch, int max_seq_len) {
    (void)c;
    (void)batch;
    DecodeGeom g{};
    g.cluster = kDecCl;
    g.chunk = max_seq_len > 0 ? dec_chunk(max_seq_len) : kTileKeys;
    g.nseg_max = max_seq_len > 0 ? dec_nseg(max_seq_len) : 1;
    return g;
}

cudaError_t launch_decode(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    const int64_t units_bound = static_cast<int64_t>(p.batch) * p.nseg_max;
    if (units_bound <= 0) return cudaSuccess;
    const bool fp8 = c->key_dtype == IDX_KEY_FP8_E4M3;
    if (fp8 && c->block_size == 64) return launch_decode_t<true, 64>(c, p, units_bound, st);
    if (fp8 && c->block_size == 32) return launch_decode_t<true, 32>(c, p, units_bound, st);
    if (!fp8 && c->block_size == 64) return launch_decode_t<false, 64>(c, p, units_bound, st);
    return launch_decode_t<false, 32>(c, p, units_bound, st);
}

}  // namespace dsaidx

#ifdef DSAIDX_PHASE_STAMPS
// Diagnostic build only: copies the phase stamps (kPhaseCtas x kPhaseUnits x
// kPhaseSlots nanosecond values, 0 = not reached) to host memory `out` and,
// with clear != 0, zeroes them on the device.  Returns 0 on success.
extern "C" int idx_phase_stamps(unsigned long long* out, int clear) {
    if (out && cudaMemcpyFromSymbol(out, dsaidx::g_phase, sizeof(dsaidx::g_phase)) != cudaSuccess) return 1;
    if (clear) {
        static unsigned long long zero[dsaidx::kPhaseCtas][dsaidx::kPhaseUnits][dsaidx::kPhaseSlots];
        if (cudaMemcpyToSymbol(dsaidx::g_phase, zero, sizeof(zero)) != cudaSuccess) return 1;
    }
    return 0;
}
#endif
