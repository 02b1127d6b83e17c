// api.cu -- the C ABI of libdsaidx (declared in include/dsaidx.h): argument
// checks, pool TMA descriptors, workspace carving and kernel dispatch.  No
// device memory is allocated here and no stream is synchronised (except in
// idx_read_device_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>

#include "common.cuh"
#include "dsaidx.h"
#include "internal.h"

using dsaidx::align_up;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool same_device(const idx_cache* c) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == c->device;
}

// Decode workspace layout: the status header, the unit counters, per
// sequence a ticket and a flag, the clusters' slow-path score scratch and,
// when a sequence can take several segments, per sequence an 8192-bin
// histogram and nseg_max runs of topk composites.
struct DecodeWs {
    size_t ctr, seqflag, ucount, scratch, ghist, runs, total;
    int64_t runs_cap;   // composites per sequence
    dsaidx::DecodeGeom geom;
};
DecodeWs decode_ws(const idx_cache* c, int batch, int max_seq_len, int topk) {
    DecodeWs w{};
    w.geom = dsaidx::decode_geometry(c, batch, max_seq_len);
    const size_t nb = static_cast<size_t>(batch);
    const bool multi = w.geom.nseg_max > 1;
    w.runs_cap = multi ? static_cast<int64_t>(w.geom.nseg_max) * topk : 0;
    // clusters launched: at most one per unit and at most kDecMaxClusters
    const int64_t units = static_cast<int64_t>(batch) * w.geom.nseg_max;
    const int64_t maxcl = dsaidx::kDecMaxClusters(c->num_sms);
    const size_t clusters = static_cast<size_t>(units < maxcl ? units : maxcl);
    size_t o = dsaidx::kWsHeaderBytes;
    w.ctr = o;      o = align_up(o + nb * 4, 256);
    w.seqflag = o;  o = align_up(o + nb * 4, 256);
    w.ucount = o;   o = align_up(o + 8, 256);
    w.scratch = o;  o = align_up(o + clusters * dsaidx::kDecCl * static_cast<size_t>(w.geom.chunk) * 4, 256);
    w.ghist = o;    o = align_up(o + (multi ? nb * dsaidx::kGHistWords * 4 : 0), 256);
    w.runs = o;     o = align_up(o + nb * static_cast<size_t>(w.runs_cap) * 8, 256);
    w.total = o;
    return w;
}

// Prefill workspace layout.
struct PrefillWs {
    size_t rowflag, scores, total;
    int64_t stride;
};
PrefillWs prefill_ws(int total_q, int max_seq_len) {
    PrefillWs w{};
    w.stride = static_cast<int64_t>(align_up(static_cast<size_t>(max_seq_len > 0 ? max_seq_len : 1), 4));
    size_t o = dsaidx::kWsHeaderBytes;
    w.rowflag = o;  o = align_up(o + static_cast<size_t>(total_q) * 4, 256);
    w.scores = o;   o = align_up(o + static_cast<size_t>(total_q) * static_cast<size_t>(w.stride) * 4, 256);
    w.total = o;
    return w;
}

bool valid_dtype(int d) { return d == IDX_KEY_FP8_E4M3 || d == IDX_KEY_BF16; }

// Limit of the decode kernel's pipeline waits; idx_test_set_wait_limit
// shortens it (and makes the MMA issuer withhold one signal) for the test of
// the timeout path.
std::atomic<unsigned long long> g_test_wait_ns{dsaidx::kWaitLimitNs};

}  // namespace

extern "C" {

size_t idx_block_bytes(int key_dtype, int block_size, int head_dim) {
    if (!valid_dtype(key_dtype) || head_dim != IDX_HEAD_DIM) return 0;
    if (block_size != 32 && block_size != 64) return 0;
    return key_dtype == IDX_KEY_FP8_E4M3 ? static_cast<size_t>(block_size) * (128 + 4)
                                        : static_cast<size_t>(block_size) * 256;
}

idx_status idx_cache_create(idx_cache** out, void* pool_dev, int64_t num_blocks, int block_size,
                            int head_dim, int key_dtype) {
    if (!out || !pool_dev) return IDX_ERR_INVALID_ARG;
    if (!valid_dtype(key_dtype) || (block_size != 32 && block_size != 64)) return IDX_ERR_INVALID_ARG;
    if (head_dim != IDX_HEAD_DIM) return IDX_ERR_UNSUPPORTED;
    if (num_blocks < 1 || num_blocks >= (int64_t(1) << 31)) return IDX_ERR_INVALID_ARG;
    if (!aligned(pool_dev, 256)) return IDX_ERR_INVALID_ARG;
    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return IDX_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return IDX_ERR_CUDA;
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return IDX_ERR_CUDA;
    idx_cache* c = new (std::nothrow) idx_cache;
    if (!c) return IDX_ERR_CUDA;
    std::memset(c, 0, sizeof(*c));
    c->pool = static_cast<uint8_t*>(pool_dev);
    c->num_blocks = num_blocks;
    c->block_size = block_size;
    c->key_dtype = key_dtype;
    c->block_bytes = static_cast<int64_t>(idx_block_bytes(key_dtype, block_size, head_dim));
    c->device = dev;
    c->num_sms = sms;
    const bool fp8 = key_dtype == IDX_KEY_FP8_E4M3;
    // 3-D view of the pool: (byte or element within a key row, row within the
    // block, block).  Boxes are one block of rows by 128 bytes, 128-byte swizzled.
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(block_size), static_cast<cuuint64_t>(num_blocks)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(fp8 ? 128 : 256),
                             static_cast<cuuint64_t>(c->block_bytes)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(fp8 ? 128 : 64), static_cast<cuuint32_t>(block_size), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&c->tmap, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     pool_dev, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        delete c;
        return IDX_ERR_CUDA;
    }
    *out = c;
    return IDX_OK;
}

void idx_cache_destroy(idx_cache* cache) { delete cache; }

namespace {
idx_status store_keys_common(const idx_cache* cache, const void* k_bf16_dev, const int64_t* slot_mapping_dev,
                             int64_t n, int32_t* status_dev, unsigned flags, void* stream) {
    if (!cache || n < 0 || (flags & ~(IDX_STORE_ROTATE | IDX_STORE_FP4_ROUNDTRIP)) != 0u) return IDX_ERR_INVALID_ARG;
    if (n == 0) return IDX_OK;
    if (!k_bf16_dev || !slot_mapping_dev || !aligned(k_bf16_dev, 16) || !aligned(slot_mapping_dev, 8))
        return IDX_ERR_INVALID_ARG;
    if (!same_device(cache)) return IDX_ERR_INVALID_ARG;
    cudaError_t e = dsaidx::launch_store(cache, k_bf16_dev, slot_mapping_dev, n, status_dev, flags,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}
}  // namespace

idx_status idx_store_keys(const idx_cache* cache, const void* k_bf16_dev, const int64_t* slot_mapping_dev,
                          int64_t n, int32_t* status_dev, void* stream) {
    return store_keys_common(cache, k_bf16_dev, slot_mapping_dev, n, status_dev, 0u, stream);
}

idx_status idx_store_keys_rotated(const idx_cache* cache, const void* k_bf16_dev, const int64_t* slot_mapping_dev,
                                  int64_t n, int32_t* status_dev, void* stream) {
    return store_keys_common(cache, k_bf16_dev, slot_mapping_dev, n, status_dev, IDX_STORE_ROTATE, stream);
}

idx_status idx_store_keys_ex(const idx_cache* cache, const void* k_bf16_dev, const int64_t* slot_mapping_dev,
                             int64_t n, unsigned flags, int32_t* status_dev, void* stream) {
    return store_keys_common(cache, k_bf16_dev, slot_mapping_dev, n, status_dev, flags, stream);
}

idx_status idx_gather_blocks(const idx_cache* cache, const int32_t* block_table_dev, int max_blocks_per_seq,
                             const int32_t* seq_lens_dev, int batch, void* dst_pool_dev, int32_t* status_dev,
                             void* stream) {
    if (!cache || batch < 0 || max_blocks_per_seq < 1) return IDX_ERR_INVALID_ARG;
    if (batch == 0) return IDX_OK;
    if (!block_table_dev || !seq_lens_dev || !dst_pool_dev || !aligned(dst_pool_dev, 16)) return IDX_ERR_INVALID_ARG;
    if (!same_device(cache)) return IDX_ERR_INVALID_ARG;
    cudaError_t e = dsaidx::launch_gather(cache, block_table_dev, max_blocks_per_seq, seq_lens_dev, batch,
                                          dst_pool_dev, status_dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

size_t idx_workspace_bytes_decode(const idx_cache* cache, int batch, int max_seq_len, int heads, int topk) {
    if (!cache || batch < 0 || max_seq_len < 0 || heads != dsaidx::kHeads) return 0;
    if (topk < 1 || topk > IDX_MAX_TOPK) return 0;
    return decode_ws(cache, batch, max_seq_len, topk).total;
}

idx_status idx_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream) {
    if (!workspace_dev || ws_bytes < dsaidx::kWsHeaderBytes) return IDX_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace_dev, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? IDX_OK
               : IDX_ERR_CUDA;
}

idx_status idx_score_topk_decode(const idx_cache* cache, const void* q_bf16_dev, const float* w_dev,
                                 const int32_t* block_table_dev, int max_blocks_per_seq,
                                 const int32_t* seq_lens_dev, int batch, int max_seq_len, int heads,
                                 int topk, int32_t* out_idx_dev, float* out_score_dev, void* workspace_dev,
                                 size_t ws_bytes, void* stream) {
    return idx_score_topk_decode_slots(cache, q_bf16_dev, w_dev, block_table_dev, max_blocks_per_seq,
                                       seq_lens_dev, batch, max_seq_len, heads, topk, out_idx_dev, out_score_dev,
                                       nullptr, workspace_dev, ws_bytes, stream);
}

idx_status idx_score_topk_decode_slots(const idx_cache* cache, const void* q_bf16_dev, const float* w_dev,
                                       const int32_t* block_table_dev, int max_blocks_per_seq,
                                       const int32_t* seq_lens_dev, int batch, int max_seq_len, int heads,
                                       int topk, int32_t* out_idx_dev, float* out_score_dev,
                                       int64_t* out_slot_dev, void* workspace_dev, size_t ws_bytes, void* stream) {
    if (!cache) return IDX_ERR_INVALID_ARG;
    if (out_slot_dev && !aligned(out_slot_dev, 8)) return IDX_ERR_INVALID_ARG;
    if (heads != dsaidx::kHeads) return IDX_ERR_UNSUPPORTED;
    if (batch < 0 || max_seq_len < 0 || topk < 1 || topk > IDX_MAX_TOPK || max_blocks_per_seq < 1)
        return IDX_ERR_INVALID_ARG;
    if (batch == 0) return IDX_OK;
    if (!q_bf16_dev || !w_dev || !block_table_dev || !seq_lens_dev || !out_idx_dev || !workspace_dev)
        return IDX_ERR_INVALID_ARG;
    if (!aligned(q_bf16_dev, 16) || !aligned(w_dev, 16) || !aligned(workspace_dev, 256))
        return IDX_ERR_INVALID_ARG;
    if (!same_device(cache)) return IDX_ERR_INVALID_ARG;
    const DecodeWs ws = decode_ws(cache, batch, max_seq_len, topk);
    if (ws_bytes < ws.total) return IDX_ERR_WORKSPACE_TOO_SMALL;
    if (static_cast<int64_t>(batch) * ws.geom.nseg_max >= (int64_t(1) << 31)) return IDX_ERR_INVALID_ARG;
    uint8_t* base = static_cast<uint8_t*>(workspace_dev);
    dsaidx::ScoreParams p{};
    p.q = static_cast<const uint16_t*>(q_bf16_dev);
    p.w = w_dev;
    p.block_table = block_table_dev;
    p.seq_lens = seq_lens_dev;
    p.pool = cache->pool;
    p.num_blocks = cache->num_blocks;
    p.block_bytes = cache->block_bytes;
    p.mbps = max_blocks_per_seq;
    p.batch = batch;
    p.max_seq_len = max_seq_len;
    p.topk = topk;
    p.chunk = ws.geom.chunk;
    p.cluster = ws.geom.cluster;
    p.nseg_max = ws.geom.nseg_max;
    p.out_idx = out_idx_dev;
    p.out_score = out_score_dev;
    p.out_slot = out_slot_dev;
    p.block_size = cache->block_size;
    p.status = reinterpret_cast<int32_t*>(base);
    p.ctr = reinterpret_cast<uint32_t*>(base + ws.ctr);
    p.seqflag = reinterpret_cast<uint32_t*>(base + ws.seqflag);
    p.ghist = reinterpret_cast<uint32_t*>(base + ws.ghist);
    p.cand = reinterpret_cast<uint64_t*>(base + ws.runs);
    p.cand_cap = ws.runs_cap;
    p.ucount = reinterpret_cast<uint32_t*>(base + ws.ucount);
    p.scratch = reinterpret_cast<float*>(base + ws.scratch);
    p.wait_ns = g_test_wait_ns.load(std::memory_order_relaxed);
    p.withhold = p.wait_ns != dsaidx::kWaitLimitNs ? 1 : 0;
    cudaError_t e = dsaidx::launch_decode(cache, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

size_t idx_workspace_bytes_prefill(const idx_cache* cache, int batch, int total_q, int max_seq_len, int heads,
                                   int topk) {
    if (!cache || batch < 0 || total_q < 0 || max_seq_len < 0 || heads != dsaidx::kHeads) return 0;
    if (topk < 1 || topk > IDX_MAX_TOPK) return 0;
    return prefill_ws(total_q, max_seq_len).total;
}

idx_status idx_score_topk_prefill(const idx_cache* cache, const void* q_bf16_dev, const float* w_dev,
                                  const int32_t* cu_seqlens_q_dev, const int32_t* seq_lens_dev,
                                  const int32_t* block_table_dev, int max_blocks_per_seq, int batch,
                                  int total_q, int max_seq_len, int heads, int topk, int32_t* out_idx_dev,
                                  float* out_score_dev, void* workspace_dev, size_t ws_bytes, void* stream) {
    return idx_score_topk_prefill_slots(cache, q_bf16_dev, w_dev, cu_seqlens_q_dev, seq_lens_dev, block_table_dev,
                                        max_blocks_per_seq, batch, total_q, max_seq_len, heads, topk, out_idx_dev,
                                        out_score_dev, nullptr, workspace_dev, ws_bytes, stream);
}

idx_status idx_score_topk_prefill_slots(const idx_cache* cache, const void* q_bf16_dev, const float* w_dev,
                                        const int32_t* cu_seqlens_q_dev, const int32_t* seq_lens_dev,
                                        const int32_t* block_table_dev, int max_blocks_per_seq, int batch,
                                        int total_q, int max_seq_len, int heads, int topk, int32_t* out_idx_dev,
                                        float* out_score_dev, int64_t* out_slot_dev, void* workspace_dev,
                                        size_t ws_bytes, void* stream) {
    if (!cache) return IDX_ERR_INVALID_ARG;
    if (out_slot_dev && !aligned(out_slot_dev, 8)) return IDX_ERR_INVALID_ARG;
    if (heads != dsaidx::kHeads) return IDX_ERR_UNSUPPORTED;
    if (batch < 0 || batch > 4096 || total_q < 0 || max_seq_len < 0 || topk < 1 || topk > IDX_MAX_TOPK ||
        max_blocks_per_seq < 1)
        return IDX_ERR_INVALID_ARG;
    if (batch == 0 || total_q == 0) return IDX_OK;
    if (!q_bf16_dev || !w_dev || !cu_seqlens_q_dev || !seq_lens_dev || !block_table_dev || !out_idx_dev ||
        !workspace_dev)
        return IDX_ERR_INVALID_ARG;
    if (!aligned(q_bf16_dev, 16) || !aligned(w_dev, 16) || !aligned(workspace_dev, 256))
        return IDX_ERR_INVALID_ARG;
    if (!same_device(cache)) return IDX_ERR_INVALID_ARG;
    const PrefillWs ws = prefill_ws(total_q, max_seq_len);
    if (ws_bytes < ws.total) return IDX_ERR_WORKSPACE_TOO_SMALL;
    uint8_t* base = static_cast<uint8_t*>(workspace_dev);
    dsaidx::ScoreParams p{};
    p.q = static_cast<const uint16_t*>(q_bf16_dev);
    p.w = w_dev;
    p.block_table = block_table_dev;
    p.seq_lens = seq_lens_dev;
    p.cu_q = cu_seqlens_q_dev;
    p.pool = cache->pool;
    p.num_blocks = cache->num_blocks;
    p.block_bytes = cache->block_bytes;
    p.mbps = max_blocks_per_seq;
    p.batch = batch;
    p.max_seq_len = max_seq_len;
    p.topk = topk;
    p.chunk = 0;
    p.cluster = 1;
    p.nseg_max = 0;
    p.total_q = total_q;
    p.num_groups = (total_q + dsaidx::kPrefillQT - 1) / dsaidx::kPrefillQT + batch;
    p.out_idx = out_idx_dev;
    p.out_score = out_score_dev;
    p.out_slot = out_slot_dev;
    p.block_size = cache->block_size;
    p.status = reinterpret_cast<int32_t*>(base);
    p.rowflag = reinterpret_cast<uint32_t*>(base + ws.rowflag);
    p.scores = reinterpret_cast<float*>(base + ws.scores);
    p.score_stride = ws.stride;
    p.wait_ns = dsaidx::kWaitLimitNs;
    cudaError_t e = dsaidx::launch_prefill(cache, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? IDX_OK : IDX_ERR_CUDA;
}

idx_status idx_read_device_status(const void* workspace_dev, void* stream, int32_t* code_out) {
    if (!workspace_dev || !code_out) return IDX_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return IDX_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, workspace_dev, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return IDX_ERR_CUDA;
    *code_out = v;
    return IDX_OK;
}

idx_status idx_test_set_wait_limit(unsigned long long limit_ns) {
    if (limit_ns == 0 || limit_ns > dsaidx::kWaitLimitNs) limit_ns = dsaidx::kWaitLimitNs;
    g_test_wait_ns.store(limit_ns, std::memory_order_relaxed);
    return IDX_OK;
}

const char* idx_status_str(idx_status s) {
    switch (s) {
        case IDX_OK: return "ok";
        case IDX_ERR_INVALID_ARG: return "invalid argument";
        case IDX_ERR_UNSUPPORTED: return "unsupported configuration";
        case IDX_ERR_CUDA: return "CUDA error";
        case IDX_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case IDX_ERR_DEVICE_CHECK: return "device-side check failed";
        case IDX_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
