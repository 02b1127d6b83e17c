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
    int64_t* out_slot;           // nullable: physical slot of each selected key (-1 pads)
    int block_size;              // tokens per pool block (the slot translation)
    // workspace
    int32_t* status;
    uint32_t* ctr;               // decode: [batch] completed-segment tickets
    uint32_t* ghist;             // decode: [batch, kGHistWords] bin counts of the segments' runs
    uint32_t* seqflag;           // decode: [batch] a segment failed a device check
    uint64_t* cand;              // decode: [batch, cand_cap] the segments' sorted top-k runs
    int64_t cand_cap;            // decode: nseg_max * topk composites per sequence
    float* scores;               // prefill: [total_q, score_stride]
    int64_t score_stride;
    uint32_t* rowflag;           // prefill: [total_q]
    uint32_t* ucount;            // decode: [2] units drawn, clusters done (zero between calls)
    float* scratch;              // decode: per cluster kDecCl * chunk scores (slow path)
    unsigned long long wait_ns;  // limit of the pipeline waits (normally 2 s)
    int withhold;                // test hook: 1 = the MMA issuer withholds its first accumulator signal
};

// ---------------------------------------------------------------------------
// decode geometry (host and device agree on it)
// ---------------------------------------------------------------------------
constexpr int kDecCl = 8;               // CTAs per cluster (one sequence segment)
constexpr int kDecChunkMax = 8192;      // keys one CTA scores per segment
// Per-sequence histogram of the segments' runs (score key >> 19); word
// kGHistBins holds the largest bin of any run entry plus one (0: none).
constexpr int kGHistBins = 8192;
constexpr int kGHistWords = kGHistBins + 32;

// Keys per CTA for a sequence of S > 0 keys: its share of a cluster rounded up
// to the 128-key tile, at most kDecChunkMax.
__host__ __device__ inline int dec_chunk(int S) {
    int per = (S + kDecCl - 1) / kDecCl;
    per = (per + kTileKeys - 1) / kTileKeys * kTileKeys;
    if (per < kTileKeys) per = kTileKeys;
    return per < kDecChunkMax ? per : kDecChunkMax;
}
// Segments (clusters' worth of chunks) of a sequence of S > 0 keys.
__host__ __device__ inline int dec_nseg(int S) {
    const int64_t seglen = static_cast<int64_t>(kDecCl) * dec_chunk(S);
    const int64_t n = (static_cast<int64_t>(S) + seglen - 1) / seglen;
    return n < 1 ? 1 : static_cast<int>(n);
}
// Work units of a sequence: its segments, or one unit that writes the -1 row
// of an empty sequence or of one whose length is out of range.
__host__ __device__ inline int dec_units(int S, int max_seq_len) {
    return (S > 0 && S <= max_seq_len) ? dec_nseg(S) : 1;
}

// Shared-memory plan of the decode kernel: three key stages (after the
// stream: the selection's scratch), the B tile right after them (1024-byte
// aligned for the 128-byte swizzle), one region that holds in turn this CTA's
// staged bf16 query rows and the chunk's 16-bit histogram (during the stream)
// and the pool of every CTA's candidates (during the selection), the chunk's
// scores, the cluster's histogram windows, w', block ids, scratch and
// barriers.  fp8: 114,832 bytes, two CTAs per SM; bf16: one.
struct DecPlan {
    int stages, a_stage_bytes, a_off, raw_off, sc_off, win_off, pool_off, q_off, w_off, bid_off, misc_off, bar_off,
        total;
};
constexpr int kDecMiscBytes = 1536;
__host__ __device__ inline DecPlan dec_plan(bool fp8) {
    DecPlan p{};
    p.stages = 3;
    p.a_stage_bytes = fp8 ? 16384 : 32768;
    int o = 0;
    p.a_off = o;      o += p.stages * p.a_stage_bytes;
    p.q_off = o;      o += 64 * (fp8 ? 128 : 256);
    p.raw_off = o;    o += 16384;                      // 2 KB query rows + w / 16 KB histogram / 16 KB pool
    p.pool_off = p.raw_off;
    p.sc_off = o;     o += kDecChunkMax * 4 + 16;
    p.win_off = o;    o += kDecCl * 528;
    p.w_off = o;      o += 64 * 4;
    p.bid_off = o;    o += kDecChunkMax / 32 * 4;      // block ids of one chunk
    p.misc_off = o;   o += kDecMiscBytes;
    p.bar_off = o;    o += 256;
    p.total = o + 1024;
    return p;
}
static_assert(3 * 16384 >= 4096 * 4 + 4096 * 8, "the selection scratch fits the fp8 key stages");
constexpr int kDecMaxClusters(int sms) { return 2 * sms / kDecCl; }   // two CTAs per SM at most

// Shared-memory plan of the prefill scoring kernel (kPrefillQT queries per
// CTA): key stages (seven of fp8 codes, two of bf16 keys; the epilogue reads
// the fp8 key scales from the pool, so a stage holds codes only and is free
// once the MMA has read it), the B tile, head weights, the staged bf16 query
// rows, block ids, scratch and barriers (at most 8 stages).
struct SmemPlan {
    int stages, a_stage_bytes, q_bytes, n_cols;
    int a_off, q_off, scale_off, w_off, raw_off, bid_off, misc_off, bar_off;
    int total;   // bytes to request (includes 1 KB of alignment slack)
};
__host__ __device__ inline SmemPlan make_plan(bool fp8, int qt, int chunk) {
    (void)chunk;
    SmemPlan p{};
    p.n_cols = 64 * qt;
    p.stages = fp8 ? 7 : 2;
    p.a_stage_bytes = fp8 ? 16384 : 32768;
    p.q_bytes = p.n_cols * (fp8 ? 128 : 256);
    int o = 0;
    p.a_off = o;       o += p.stages * p.a_stage_bytes;
    p.q_off = o;       o += p.q_bytes;
    p.scale_off = o;   // no scale ring
    p.w_off = o;       o += p.n_cols * 4;
    p.raw_off = o;     o += qt * 16384;
    p.bid_off = o;     o += kBidWindow * 4;  // prefetched block ids
    p.misc_off = o;    o += 4096;            // scratch, flags, group scan
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
                         int32_t* status, unsigned flags, cudaStream_t st);   // IDX_STORE_* flags
cudaError_t launch_decode(const idx_cache* c, const ScoreParams& p, cudaStream_t st);
cudaError_t launch_prefill(const idx_cache* c, const ScoreParams& p, cudaStream_t st);
cudaError_t launch_gather(const idx_cache* c, const int32_t* block_table, int mbps, const int32_t* seq_lens,
                          int batch, void* dst, int32_t* status, cudaStream_t st);
// Per-kernel timing hook (ktimer.cu): records the next event when timing is on.
void kt_mark(cudaStream_t st);

// Decode geometry for a batch shape: clusters of `cluster` CTAs, chunks of at
// most `chunk` keys, at most `nseg_max` segments (work units) per sequence.
struct DecodeGeom {
    int cluster, chunk, nseg_max;
};
DecodeGeom decode_geometry(const idx_cache* c, int batch, int max_seq_len);

}  // namespace dsaidx
