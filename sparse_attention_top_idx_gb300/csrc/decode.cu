// decode.cu -- launch of the fused decode score + top-k kernel.
#include "score_kernel.cuh"

namespace dsaidx {

namespace {

template <bool kFp8, int kBs>
cudaError_t launch_decode_t(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    const SmemPlan plan = make_plan(kFp8, 1, p.chunk);
    auto kern = score_kernel<kFp8, kBs, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.total);
    if (e != cudaSuccess) return e;
    const int grid = p.batch * p.max_chunks;
    kern<<<grid, kThreads, plan.total, st>>>(c->tmap, p);
    return cudaGetLastError();
}

}  // namespace

// Keys per decode CTA: enough CTAs for two per SM over the bound batch *
// max_seq_len, a multiple of the 128-key tile, between 512 and 8192 (fp8) or
// 2048 (bf16) keys so that two CTAs (stages, scores, histogram) fit per SM.
int decode_chunk(const idx_cache* c, int batch, int max_seq_len) {
    const int cap = (c->key_dtype == IDX_KEY_FP8_E4M3) ? 8192 : 2048;
    const double slots = 2.0 * (c->num_sms > 0 ? c->num_sms : 1);
    double est = static_cast<double>(batch) * static_cast<double>(max_seq_len) / slots;
    int64_t ch = static_cast<int64_t>(est + 0.999999);
    ch = (ch + kTileKeys - 1) / kTileKeys * kTileKeys;
    if (ch < 512) ch = 512;
    if (ch > cap) ch = cap;
    return static_cast<int>(ch);
}

cudaError_t launch_decode(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    const bool fp8 = c->key_dtype == IDX_KEY_FP8_E4M3;
    if (fp8 && c->block_size == 64) return launch_decode_t<true, 64>(c, p, st);
    if (fp8 && c->block_size == 32) return launch_decode_t<true, 32>(c, p, st);
    if (!fp8 && c->block_size == 64) return launch_decode_t<false, 64>(c, p, st);
    return launch_decode_t<false, 32>(c, p, st);
}

}  // namespace dsaidx
