// decode.cu -- launch of the fused decode score + top-k kernel as thread-block
// clusters (one cluster per segment of a sequence).
#include "score_kernel.cuh"

namespace dsaidx {

namespace {

constexpr int kDecodeCluster = kCl;   // portable cluster size

template <bool kFp8, int kBs>
cudaError_t launch_decode_t(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    const SmemPlan plan = make_plan(kFp8, 1, p.chunk);
    auto kern = score_kernel<kFp8, kBs, 1>;
    // the limit is raised once to the largest plan this key format uses
    int most = make_plan(kFp8, 1, kFp8 ? 8192 : 2048).total;
    const int mid = make_plan(kFp8, 1, 4096).total;
    if (kFp8 && mid > most) most = mid;
    cudaError_t e = set_smem_once(kern, most, attr_done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.batch) * p.nseg_max * p.cluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(plan.total);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, c->tmap, p);
}

}  // namespace

// One cluster of 8 CTAs per sequence segment.  A CTA scores at most `chunk`
// keys: the longest sequence's share of its cluster rounded up to the 128-key
// tile, at most 8192 (fp8) or 2048 (bf16) keys so that the chunk's scores stay
// in shared memory; sequences longer than 8 chunks take several segments.
DecodeGeom decode_geometry(const idx_cache* c, int batch, int max_seq_len) {
    (void)batch;
    DecodeGeom g{};
    g.cluster = kDecodeCluster;
    const int cap = (c->key_dtype == IDX_KEY_FP8_E4M3) ? 8192 : 2048;
    int64_t per = (static_cast<int64_t>(max_seq_len) + g.cluster - 1) / g.cluster;
    per = (per + kTileKeys - 1) / kTileKeys * kTileKeys;
    if (per < kTileKeys) per = kTileKeys;
    g.chunk = static_cast<int>(per < cap ? per : cap);
    const int64_t seglen = static_cast<int64_t>(g.cluster) * g.chunk;
    int64_t nseg = (static_cast<int64_t>(max_seq_len) + seglen - 1) / seglen;
    g.nseg_max = static_cast<int>(nseg < 1 ? 1 : nseg);
    return g;
}

cudaError_t launch_decode(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    const bool fp8 = c->key_dtype == IDX_KEY_FP8_E4M3;
    if (fp8 && c->block_size == 64) return launch_decode_t<true, 64>(c, p, st);
    if (fp8 && c->block_size == 32) return launch_decode_t<true, 32>(c, p, st);
    if (!fp8 && c->block_size == 64) return launch_decode_t<false, 64>(c, p, st);
    return launch_decode_t<false, 32>(c, p, st);
}

}  // namespace dsaidx
