// internal.h -- host/device structures shared between the C ABI layer and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "dsaidx.h"

struct idx_cache {
    uint8_t* pool;
    int64_t num_blocks;
    int block_size;
    int key_dtype;          // IDX_KEY_FP8_E4M3 or IDX_KEY_BF16
    int64_t block_bytes;
    int device;
    int num_sms;
    CUtensorMap tmap;       // 3-D view (row bytes/elements, rows in block, block) of the pool
};

namespace dsaidx {

constexpr int kThreads = 256;        // decode scoring and selection kernels
constexpr int kPrefillThreads = 640; // prefill scoring: 16 epilogue warps
constexpr int kTileKeys = 128;       // keys per MMA tile (M)
constexpr int kPrefillQT = 4;        // queries per prefill CTA (N = 64 * 4 = 256)
constexpr int kBidWindow = 256;      // block ids the TMA producer warp prefetches at a time

// Parameters of the scoring kernels (decode fused top-k, prefill scores).
struct ScoreParams {
    const uint16_t* q;           // bf16 bits [rows, 64, 128]
    const float* w;              // [rows, 64]
    const int32_t* block_table;  // [batch, mbps]
    const int32_t* seq_lens;     // [batch]
    const int32_t* cu_q;         // [batch + 1] (prefill)
    const uint8_t* pool;
    int64_t num_blocks;
    int64_t block_bytes;
    int mbps;
    int batch;
    int max_seq_len;
    int topk;
    int chunk;                   // decode: largest chunk of keys per CTA (multiple of 128)
    int cluster;                 // decode: CTAs per cluster (one sequence segment)
    int nseg_max;                // decode: segments of the longest sequence
    int total_q;                 // prefill
    int num_groups;              // prefill: grid bound on query groups
    int32_t* out_idx;
    float* out_score;
    // workspace
    int32_t* status;
    uint32_t* ctr;               // decode: [batch] completed-chunk tickets
    uint32_t* ghist;             // decode: [batch, 4096] histogram of published candidates
    uint32_t* seqflag;           // decode: [batch] device-check flags
    uint32_t* seqcnt;            // decode: [batch] candidates published per sequence
    uint64_t* cand;              // decode: [batch, cand_cap] composites
    int64_t cand_cap;            // decode: nseg_max * cluster * chunk (>= every seq_len)
    float* scores;               // prefill: [total_q, score_stride]
    int64_t score_stride;
    uint32_t* rowflag;           // prefill: [total_q]
};

// Shared-memory plan of the scoring kernel for (fp8, queries per CTA, chunk).
struct SmemPlan {
    int stages, a_stage_bytes, q_bytes, n_cols;
    int a_off, recv_off, recv_bytes, q_off, scale_off, w_off, hist_off, raw_off, bid_off, misc_off, bar_off;
    int total;   // bytes to request (includes 1 KB of alignment slack)
};

// Decode keeps two CTAs per SM (<= ~112 KB each for fp8 keys): while the
// chunk's scores take <= 16 KB, three key stages and a 16 KB area that
// receives the other CTAs' histogram slices at the end (cluster_select);
// three stages for larger chunks.  The raw query rows are staged where the
// decode scores later go (or, for prefill, in a 64 KB region of their own).
__host__ __device__ inline SmemPlan make_plan(bool fp8, int qt, int chunk) {
    SmemPlan p{};
    p.n_cols = 64 * qt;
    p.stages = (qt == 1) ? (fp8 ? 3 : 2) : (fp8 ? 4 : 2);
    p.recv_bytes = (qt == 1 && fp8 && chunk <= 4096) ? 16384 : 0;
    p.a_stage_bytes = fp8 ? 16384 : 32768;
    p.q_bytes = p.n_cols * (fp8 ? 128 : 256);
    const int raw_bytes = (qt == 1) ? (chunk * 4 > 16384 ? chunk * 4 : 16384) : qt * 16384;
    int o = 0;
    p.a_off = o;       o += p.stages * p.a_stage_bytes;
    p.recv_off = o;    o += p.recv_bytes;
    p.q_off = o;       o += p.q_bytes;
    p.scale_off = o;   o += fp8 ? p.stages * 512 : 0;
    p.w_off = o;       o += p.n_cols * 4;
    p.hist_off = o;    o += (qt == 1) ? 4096 * 4 : 0;
    p.raw_off = o;     o += raw_bytes;
    p.bid_off = o;     o += kBidWindow * 4;  // prefetched block ids
    p.misc_off = o;    o += 4096;            // selection scratch, flags, group scan
    p.bar_off = o;     o += 512;             // mbarriers
    p.total = o + 1024;
    return p;
}

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device
// (the first call for each device sets it; later calls, including calls made
// while a stream is being captured into a graph, skip the runtime call).
template <class Kern>
inline cudaError_t set_smem_once(Kern kern, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Kernel launchers (one per translation unit).
cudaError_t launch_store(const idx_cache* c, const void* k, const int64_t* slots, int64_t n,
                         int32_t* status, cudaStream_t st);
cudaError_t launch_decode(const idx_cache* c, const ScoreParams& p, cudaStream_t st);
cudaError_t launch_prefill(const idx_cache* c, const ScoreParams& p, cudaStream_t st);

// Decode geometry for a batch shape: clusters of `cluster` CTAs, each CTA
// scoring at most `chunk` keys, `nseg_max` cluster segments per sequence.
struct DecodeGeom {
    int cluster, chunk, nseg_max;
};
DecodeGeom decode_geometry(const idx_cache* c, int batch, int max_seq_len);

}  // namespace dsaidx
