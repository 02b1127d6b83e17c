// score_kernel.cuh -- the indexer scoring kernel for sm_103a.
//
// score[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])  (fp32 accumulation), the
// compressed query-key relevance score of "The Hypothesis That Refused to Die"
// (section "The Context"), computed from the paged index-key cache the way the
// paged MQA logits of "DeepSeek-V4 index_topk=1024 sparse indexer can't recall
// verbatim lines" (ROCm/ATOM issue #1507, section "How it was isolated") read
// it: straight from the paged blocks through the block table.
//
// Work units:
//   decode  (kQT = 1, 256 threads): a chunk of one sequence's keys against
//                      its 64 query heads (N = 64); the 8 CTAs of a sequence
//                      segment form a thread-block cluster that selects the
//                      top-k together (cluster_select.cuh);
//   prefill (kQT = 4, 640 threads): up to 4 consecutive query rows of one
//                      sequence against every key they can see (N = 256);
//                      scores go to the workspace for the row select kernel.
// The contraction D[s, (t, h)] = sum_d k[s, d] q[t, h, d] runs on the 5th-gen
// tensor cores: M = 128 keys (A, K-major, TMA-loaded 64- or 32-row boxes of the
// paged blocks, 128-byte swizzle), N = 64 * kQT query-heads (B, quantised by
// the CTA itself into shared memory), K = 128, fp32 accumulators in TMEM
// (two buffers so the epilogue of tile i overlaps the MMA of tile i + 1).
// fp8 keys use kind::f8f6f4 (e4m3 x e4m3), bf16 keys kind::f16.
//
// Warp roles: warp 0 lane 0 starts the query rows' bulk copy, then issues the
// key TMA (the warp prefetches block ids; in decode lane 0 of warp 3 issues
// the second half of every tile's blocks); the other warps quantise the
// queries into the B tile (decode: warps 4..7, then warps 1, 2 and 4..7 send
// them to the cluster); warp 1 owns TMEM and its lane 0 issues the MMAs;
// warps 4.. (decode 4, prefill 16: one per TMEM lane quadrant and query, one
// key row per thread) run the epilogue ks[s] * sum_h w'[t, h] * max(D, 0)
// with the query's head weights held in registers.
#pragma once

#include <cuda_bf16.h>

#include "cluster_select.cuh"
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace dsaidx {

struct KernelShared {
    uint32_t tmem_base;
    int abort;          // a role gave up on a bounded wait
    int bad;            // a block id failed its check
    uint32_t ticket;
    int unit_b, key_begin, key_end, seq_len, nrows, row0, nq;
    int seg, nseg;      // decode: segment of the sequence and segments in it
    int pos[kPrefillQT];
    ClusterSmem cs;     // decode: the cluster selection's shared state
    uint32_t merge_last;   // decode: this cluster merges the sequence's runs (pushed by rank 0)
    SelectSmem sel;
    uint32_t grp[kThreads];   // prefill: group-count scan (first 256 threads)
};
static_assert(sizeof(KernelShared) <= 4096, "KernelShared must fit the misc region");

// e4m3 encode of two fp32 values (lo = a, hi = b) by the hardware convert.
__device__ __forceinline__ uint32_t cvt_e4m3x2_pair(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a K-major operand
// tile stored with the 128-byte swizzle (1024-byte aligned tile base).
__device__ __forceinline__ int sw128_off(int r, int c) {
    return (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4);
}

// Copy a 4096-bin histogram from global memory (bypassing L1) into shared
// memory: four independent 16-byte loads per thread of a 256-thread block.
__device__ __forceinline__ void copy_hist_global(uint32_t* dst, const uint32_t* src) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(s4 + u * 256 + threadIdx.x);
#pragma unroll
    for (int u = 0; u < 4; ++u) d4[u * 256 + threadIdx.x] = v[u];
}

// One quarter (32 elements, `part` 0..3) of query row r, staged in shared
// memory as bf16, turned into its B-tile content.  fp8: per row scale
// sq = amax / 448 (IEEE; the four lanes of gmask share the row and reduce
// amax), codes e4m3(q / sq) with the quotient correctly rounded, returned as
// two 16-byte chunks (row chunks 2 part and 2 part + 1), w' = w * sq; amax = 0
// gives zero codes.  bf16: the 64 bytes as four chunks (B-tile half part / 2,
// chunks 4 (part & 1) .. +3), w' = w.  A missing row (have = false) gives
// zero chunks and w' = 0.
template <bool kFp8>
__device__ __forceinline__ float quant_row_part(const uint8_t* raw_row, int part, bool have, float wv,
                                                unsigned gmask, uint4 (&out)[4]) {
    uint4 v[4];
    if (have) {
        const uint4* src = reinterpret_cast<const uint4*>(raw_row + part * 64);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = src[i];
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
        wv = 0.0f;
    }
    if constexpr (!kFp8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[i] = v[i];
        return wv;
    } else {
        float x[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * i + 2 * e] = __uint_as_float(w4[e] << 16);
                x[8 * i + 2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
        const float sq = __fdiv_rn(amax, 448.0f);
        const DivBy div(sq);
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (amax != 0.0f) {
                const float y0 = div(x[4 * i + 0]), y1 = div(x[4 * i + 1]);
                const float y2 = div(x[4 * i + 2]), y3 = div(x[4 * i + 3]);
                c[i] = cvt_e4m3x2_pair(y0, y1) | (cvt_e4m3x2_pair(y2, y3) << 16);
            } else {
                c[i] = 0;
            }
        }
        out[0] = make_uint4(c[0], c[1], c[2], c[3]);
        out[1] = make_uint4(c[4], c[5], c[6], c[7]);
        return wv * sq;
    }
}

// One sixteenth (8 elements, `part` 0..15) of query row r (bf16, staged in
// shared memory) turned into its B-tile bytes, written to qtile (a tile of
// `rows` rows): the same encoding as quant_row_part with the 16 lanes of
// gmask sharing the row (the row's amax reduced over them).  Returns w' of
// the row (w * sq for fp8, w for bf16).
template <bool kFp8>
__device__ __forceinline__ float quant_row_sixteenth(const uint8_t* raw_row, int part, float wv, unsigned gmask,
                                                     uint8_t* qtile, int r, int rows) {
    const uint4 v = reinterpret_cast<const uint4*>(raw_row)[part];
    if constexpr (!kFp8) {
        *reinterpret_cast<uint4*>(qtile + (part >> 3) * (rows * 128) + sw128_off(r, part & 7)) = v;
        return wv;
    } else {
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = __uint_as_float(w4[e] << 16);
            x[2 * e + 1] = __uint_as_float(w4[e] & 0xFFFF0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, o));
        const float sq = __fdiv_rn(amax, 448.0f);
        uint32_t c0 = 0, c1 = 0;
        if (amax != 0.0f) {
            const DivBy div(sq);
            c0 = cvt_e4m3x2_pair(div(x[0]), div(x[1])) | (cvt_e4m3x2_pair(div(x[2]), div(x[3])) << 16);
            c1 = cvt_e4m3x2_pair(div(x[4]), div(x[5])) | (cvt_e4m3x2_pair(div(x[6]), div(x[7])) << 16);
        }
        *reinterpret_cast<uint2*>(qtile + sw128_off(r, part >> 1) + (part & 1) * 8) = make_uint2(c0, c1);
        return wv * sq;
    }
}

// Byte offset in the B tile of chunk i (0..3) produced by quant_row_part.
template <bool kFp8>
__device__ __forceinline__ int qchunk_off(int r, int part, int i, int rows) {
    if constexpr (kFp8) return sw128_off(r, 2 * part + i);
    else return (part >> 1) * (rows * 128) + sw128_off(r, (part & 1) * 4 + i);
}

// All query rows of a CTA (prefill), staged as raw [nrows][64][128] bf16 with
// their head weights in wq: builds the B tile and turns wq into w'.  Row
// n = j * 64 + h; rows of missing queries (j >= nrows) get zero codes and zero
// weight.  Four consecutive threads per row; t / nthreads: this thread's index
// among the nthreads doing the work.
template <bool kFp8, int kQT>
__device__ __forceinline__ void prep_queries(const uint8_t* raw, int nrows, uint8_t* qtile, float* wq,
                                             int t, int nthreads) {
    constexpr int kRows = 64 * kQT;
    constexpr int kChunks = kFp8 ? 2 : 4;
    const int part = t & 3;
    const unsigned gmask = 0xFu << (threadIdx.x & 28);   // the 4 lanes sharing a row
    for (int r = t >> 2; r < kRows; r += nthreads / 4) {
        const bool have = (r >> 6) < nrows;
        const float wv = have ? wq[r] : 0.0f;
        __syncwarp(gmask);   // every lane of the row has read wq[r]
        uint4 out[4];
        const float wn = quant_row_part<kFp8>(raw + static_cast<size_t>(r) * 256, part, have, wv, gmask, out);
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
            *reinterpret_cast<uint4*>(qtile + qchunk_off<kFp8>(r, part, i, kRows)) = out[i];
        if (part == 0) wq[r] = wn;
    }
}

// Clusters a decode sequence of S keys takes: its segments of `cluster`
// chunks, each chunk the sequence's share of its cluster rounded up to the
// tile and capped at p.chunk keys; one for an invalid or empty sequence (it
// writes the -1 outputs).
__device__ __forceinline__ int decode_clusters_of(int S, const ScoreParams& p, int CL) {
    if (S <= 0 || S > p.max_seq_len) return 1;
    const int chunk = min(p.chunk, ((S + CL - 1) / CL + kTileKeys - 1) / kTileKeys * kTileKeys);
    return (S + CL * chunk - 1) / (CL * chunk);
}

// Two decode CTAs share an SM only at <= 124 registers per thread (measured
// with the occupancy API on GB300: 126 already limits it to one), hence the
// explicit cap for the decode instantiation.
template <int kQT>
struct RegCap {
    static constexpr int value = (kQT == 1) ? 120 : 96;    // 96 * 640 threads fits one SM
};
template <int kQT>
struct BlockDim {
    static constexpr int value = (kQT == 1) ? kThreads : kPrefillThreads;
};

template <bool kFp8, int kBs, int kQT>
__global__ void __launch_bounds__(BlockDim<kQT>::value, 1) __maxnreg__(RegCap<kQT>::value)
    score_kernel(const __grid_constant__ CUtensorMap tmap, const ScoreParams p) {
    constexpr bool kDecode = (kQT == 1);
    constexpr int kBlock = BlockDim<kQT>::value;
    constexpr int kEpiWarps = kDecode ? 4 : 16;            // one per (TMEM lane quadrant, query)
    constexpr int kQPer = kQT / (kEpiWarps / 4);           // queries per epilogue warp
    constexpr int kN = 64 * kQT;
    constexpr int kBlocksPerTile = kTileKeys / kBs;
    constexpr int kKSteps = kFp8 ? 4 : 8;
    constexpr uint32_t kBlockTx = kFp8 ? (kBs * 128 + kBs * 4) : (kBs * 256);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemPlan plan = make_plan(kFp8, kQT, p.chunk);
    const int kStages = plan.stages;
    uint8_t* a_tiles = smem + plan.a_off;
    uint8_t* qtile = smem + plan.q_off;
    float* scales = reinterpret_cast<float*>(smem + plan.scale_off);
    float* wq = reinterpret_cast<float*>(smem + plan.w_off);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + plan.hist_off);
    uint8_t* raw = smem + plan.raw_off;                     // staged query rows (bf16)
    float* cscores = reinterpret_cast<float*>(smem + plan.raw_off);   // decode: the chunk's scores
    KernelShared* ks = reinterpret_cast<KernelShared*>(smem + plan.misc_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
    uint64_t* full = bars;                 // [stages] TMA -> MMA
    uint64_t* empty = bars + 4;            // [stages] MMA (+ epilogue) -> TMA
    uint64_t* tfull = bars + 8;            // [2] MMA -> epilogue
    uint64_t* tempty = bars + 10;          // [2] epilogue -> MMA
    uint64_t* mdone = bars + 12;           // MMA drain at exit
    uint64_t* qbar = bars + 13;            // query rows staged
    uint64_t* qready = bars + 14;          // decode: every rank's query rows written here
    uint64_t* cbar = bars + 15;            // decode: [kClBars] barriers of the segment selection
    uint64_t* cbar2 = cbar + kClBars;      // decode: [kClBars] barriers of the sequence merge
    uint64_t* rdone = cbar2 + kClBars;     // decode: every CTA of the cluster wrote its run part
    uint64_t* rlast = rdone + 1;           // decode: the cluster learnt whether it merges
    uint64_t* bready = rlast + 1;          // decode: the chunk's block ids are in shared memory

    const int tid = threadIdx.x;
    const int warp = warp_id(), lane = lane_id();
    int32_t* status = p.status;

    // ------------------------------------------------------------ work unit
    if constexpr (kDecode) {
        // cluster (b, seg) of p.cluster CTAs; CTA `rank` takes the rank-th chunk
        // of the segment.  Every CTA of a cluster sees the same (b, seg).
        const int CL = p.cluster;
        const int rank = static_cast<int>(cluster_rank());
        const int cid = blockIdx.x / CL;
        int b = cid, seg = 0;
        if (p.nseg_max > 1) {
            // The grid has nseg_max clusters per sequence; the clusters of the
            // sequences' real segments take its first ids, sequence by sequence
            // (an invalid or empty sequence takes one, which writes its -1
            // outputs), and the rest leave at once without delaying them.
            const int per = (p.batch + kThreads - 1) / kThreads;
            int mine = 0;
            for (int i = 0; i < per; ++i) {
                const int bb = tid * per + i;
                if (bb < p.batch) mine += decode_clusters_of(p.seq_lens[bb], p, CL);
            }
            int incl = mine;   // inclusive scan over the warp
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) ks->grp[warp] = static_cast<uint32_t>(incl);
            if (tid == 0) ks->unit_b = -1;
            __syncthreads();
            int before = 0, total = 0;
            for (int w = 0; w < kThreads / 32; ++w) {
                const int t = static_cast<int>(ks->grp[w]);
                if (w < warp) before += t;
                total += t;
            }
            const int excl = before + incl - mine;
            if (cid >= excl && cid < excl + mine) {
                int acc = excl;
                for (int i = 0; i < per; ++i) {
                    const int bb = tid * per + i;
                    const int nc = decode_clusters_of(p.seq_lens[bb], p, CL);
                    if (cid < acc + nc) {
                        ks->unit_b = bb;
                        ks->seg = cid - acc;
                        break;
                    }
                    acc += nc;
                }
            }
            __syncthreads();
            (void)total;
            if (ks->unit_b < 0) return;   // the whole cluster leaves together
            b = ks->unit_b;
            seg = ks->seg;
            __syncthreads();
        }
        const int S = p.seq_lens[b];
        const bool valid = S >= 0 && S <= p.max_seq_len;
        int chunk = kTileKeys, nseg = 0;
        if (valid && S > 0) {
            chunk = min(p.chunk, ((S + CL - 1) / CL + kTileKeys - 1) / kTileKeys * kTileKeys);
            nseg = (S + CL * chunk - 1) / (CL * chunk);
        }
        if (!(valid && S > 0)) {
            if (seg == 0 && rank == 0) {
                if (!valid && tid == 0) set_status(status, IDX_ERR_DEVICE_CHECK);
                for (int j = tid; j < p.topk; j += kThreads) {
                    p.out_idx[static_cast<int64_t>(b) * p.topk + j] = -1;
                    if (p.out_score) p.out_score[static_cast<int64_t>(b) * p.topk + j] = -INFINITY;
                }
            }
            return;   // the whole cluster leaves together
        }
        if (seg >= nseg) return;   // the whole cluster leaves together
        if (tid == 0) {
            ks->unit_b = b;
            ks->seg = seg;
            ks->nseg = nseg;
            ks->seq_len = S;
            ks->key_begin = min(S, seg * CL * chunk + rank * chunk);
            ks->key_end = min(S, ks->key_begin + chunk);
            ks->row0 = b;
            ks->nrows = 1;
        }
    } else {
        // group g of up to 4 rows of one sequence; longest rows first
        const int g = gridDim.x - 1 - blockIdx.x;
        uint32_t mine = 0;
        const int per = (p.batch + kThreads - 1) / kThreads;   // the first 256 threads scan
        for (int i = 0; i < per && tid < kThreads; ++i) {
            const int bb = tid * per + i;
            if (bb < p.batch) {
                const int nq = p.cu_q[bb + 1] - p.cu_q[bb];
                mine += static_cast<uint32_t>((max(nq, 0) + kQT - 1) / kQT);
            }
        }
        if (tid < kThreads) ks->grp[tid] = mine;
        __syncthreads();
        if (tid == 0) {
            uint32_t acc = 0;
            for (int i = 0; i < kThreads; ++i) {
                const uint32_t v = ks->grp[i];
                ks->grp[i] = acc;   // exclusive prefix
                acc += v;
            }
            ks->unit_b = (static_cast<uint32_t>(g) < acc) ? -2 : -1;
        }
        __syncthreads();
        if (ks->unit_b == -1) return;
        {
            // the thread whose range holds g finds the sequence
            const uint32_t lo = tid < kThreads ? ks->grp[tid] : 0u;
            if (tid < kThreads && mine > 0 && static_cast<uint32_t>(g) >= lo && static_cast<uint32_t>(g) < lo + mine) {
                uint32_t acc = lo;
                for (int i = 0; i < per; ++i) {
                    const int bb = tid * per + i;
                    if (bb >= p.batch) break;
                    const int nq = p.cu_q[bb + 1] - p.cu_q[bb];
                    const uint32_t ng = static_cast<uint32_t>((max(nq, 0) + kQT - 1) / kQT);
                    if (static_cast<uint32_t>(g) < acc + ng) {
                        const int i0 = (g - static_cast<int>(acc)) * kQT;
                        const int S = p.seq_lens[bb];
                        ks->unit_b = bb;
                        ks->nq = nq;
                        ks->row0 = p.cu_q[bb] + i0;
                        ks->nrows = min(kQT, nq - i0);
                        ks->seq_len = S;
                        ks->key_begin = 0;
                        for (int j = 0; j < kQT; ++j) ks->pos[j] = S - nq + i0 + j;
                        ks->key_end = S - nq + i0 + ks->nrows;   // last visible key + 1
                        break;
                    }
                    acc += ng;
                }
            }
        }
        __syncthreads();
        const int S = ks->seq_len;
        if (S > p.max_seq_len || ks->nq > S) {
            if (tid == 0) set_status(status, IDX_ERR_DEVICE_CHECK);
            if (tid < ks->nrows) atomicOr(&p.rowflag[ks->row0 + tid], 1u);
            return;
        }
    }
    __syncthreads();

    const int key_begin = ks->key_begin, key_end = ks->key_end, seq_b = ks->unit_b;
    const int ntiles = key_end > key_begin ? (key_end - key_begin + kTileKeys - 1) / kTileKeys : 0;

    // ------------------------------------------------------------ set-up
    // Warp 0: lane 0 starts the query rows' load first (decode: this rank's
    // share of the 64 head rows; prefill: every row) with their head weights,
    // so its latency overlaps the rest of the set-up; lanes 1..3 initialise
    // the other barriers in parallel.
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(qbar, 1);
            fence_mbar_init();
            const uint64_t pol_q = policy_evict_first();
            const int r0 = kDecode ? static_cast<int>(cluster_rank()) * (64 / p.cluster) : 0;
            const int nr = kDecode ? 64 / p.cluster : ks->nrows * 64;
            const int64_t g0 = static_cast<int64_t>(ks->row0) * 64 + r0;
            mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(nr) * (kHeadDim * 2 + 4));
            bulk_load(raw + static_cast<size_t>(r0) * kHeadDim * 2, p.q + g0 * kHeadDim,
                      static_cast<uint32_t>(nr) * kHeadDim * 2, qbar, pol_q);
            bulk_load(wq + r0, p.w + g0, static_cast<uint32_t>(nr) * 4, qbar, pol_q);
            tma_prefetch_desc(&tmap);
            ks->abort = 0;
            ks->bad = 0;
            ks->cs.dead = 0;
        } else if (lane == 1) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kFp8 ? 1 + kEpiWarps : 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], kEpiWarps);
            }
            mbar_init(mdone, 1);
            fence_mbar_init();
        } else if (lane == 2) {
            if constexpr (kDecode) {
                // qready completes when the query bytes have arrived
                // (st.async); the selection's barriers: see cluster_select
                mbar_init(qready, 1);
                cluster_select_init(cbar);
                fence_mbar_init();
                mbar_arrive_expect_tx(qready, 64 * (kFp8 ? 128 : 256) + 64 * 4);
                cluster_select_expect(cbar);
            }
        } else if (lane == 3) {
            if constexpr (kDecode) {
                cluster_select_init(cbar2);
                mbar_init(rdone, kCl);
                mbar_init(rlast, 1);
                mbar_init(bready, 1);
                fence_mbar_init();
                cluster_select_expect(cbar2);
                mbar_arrive_expect_tx(rlast, 4);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(&ks->tmem_base, 2 * kN);
        tmem_relinquish();
    }
    if constexpr (kDecode) {
        for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // every CTA of the cluster has its barriers and histogram ready before any
    // CTA touches another's shared memory: arrive now, wait after the local
    // query quantisation below
    if constexpr (kDecode) cluster_arrive();
    const uint32_t tmem = ks->tmem_base;

    // The query rows are in flight since the set-up; warps 0 and 3 (decode)
    // start streaming keys at once.  Decode: each rank of the cluster
    // quantises 64 / cluster of the 64 head rows (warps 4..7) and warps 1, 2
    // and 4..7 send them, as one contiguous run of the 128-byte swizzled B
    // tile (row r is bytes [128 r, 128 r + 128)) plus the rows' weights, to
    // every rank as st.async counted on that rank's qready.  Prefill: warps
    // 1..19 build the whole tile and meet on a named barrier.
    int qrow0 = 0, qrows = 0;
    if constexpr (kDecode) {
        qrows = 64 / p.cluster;
        qrow0 = static_cast<int>(cluster_rank()) * qrows;
        // 16 threads per row (warps 4..7) quantise this rank's rows
        for (int i = tid - 128; i >= 0 && i < qrows * 16; i += kThreads - 128) {
            const int r = qrow0 + (i >> 4), part = i & 15;
            const unsigned gmask = 0xFFFFu << (threadIdx.x & 16);
            if (!mbar_wait(qbar, 0, status, &ks->abort)) ks->abort = 1;
            const float wn = quant_row_sixteenth<kFp8>(raw + static_cast<size_t>(r) * 256, part, wq[r], gmask,
                                                       qtile, r, 64);
            if (part == 0) wq[r] = wn;
        }
        // warps 1, 2 and 4..7 meet on a named barrier and then on the cluster
        // barrier; warps 0 and 3 go straight to the key loads (they touch only
        // this CTA's shared memory) and wait on the cluster barrier after
        // their loops
        if (warp != 0 && warp != 3) {
            asm volatile("bar.sync 1, %0;" ::"r"(kThreads - 64) : "memory");
            cluster_wait();
            const int run = qrows * 128 / 16;                  // 16-byte chunks per half
            const int per_rank = run * (kFp8 ? 1 : 2) + qrows * 4 / 16;
            const int sender = warp < 3 ? tid - 32 : tid - 64;  // 0 .. kThreads - 65
            for (int j = sender; j < per_rank * p.cluster; j += kThreads - 64) {
                const int rk = j / per_rank, c = j - rk * per_rank;
                const uint32_t qb = dsmem_addr(qready, static_cast<uint32_t>(rk));
                const uint8_t* src;
                if (c < run * (kFp8 ? 1 : 2)) {
                    const int half = c / run, cc = c - half * run;
                    src = qtile + half * (64 * 128) + qrow0 * 128 + cc * 16;
                } else {
                    src = reinterpret_cast<const uint8_t*>(wq + qrow0) + (c - run * (kFp8 ? 1 : 2)) * 16;
                }
                dsmem_st_async_v4(dsmem_addr(src, static_cast<uint32_t>(rk)), *reinterpret_cast<const uint4*>(src), qb);
            }
        }
    } else if (warp != 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(qbar, 0, status, &ks->abort))) ks->abort = 1;
        prep_queries<kFp8, kQT>(raw, ks->nrows, qtile, wq, tid - 32, kBlock - 32);
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, %0;" ::"r"(kBlock - 32) : "memory");
    }

    // ------------------------------------------------------------ main loop
    if (warp == 0) {
        // Warp 0: the whole warp loads the block ids of up to kBidWindow
        // blocks at a time into shared memory, then lane 0 alone issues the
        // key TMA of every tile whose blocks lie in that window (the chunk
        // starts on a tile boundary and the window holds whole tiles), with
        // the stage and phase kept as running counters.  The issue loop is a
        // single thread's dependent chain and was the decode loop's limit, so
        // in decode (one window holds a whole chunk) it is split: lane 0 of
        // warp 0 takes the first half of every tile's blocks and counts the
        // tile's bytes, lane 0 of warp 3 the second half (see below).
        int* bids = reinterpret_cast<int*>(smem + plan.bid_off);
        const uint64_t pol = kDecode ? policy_evict_first() : policy_evict_last();
        const int lb_begin = key_begin / kBs;
        const int lb_end = (key_end + kBs - 1) / kBs;
        const int* bt_row = p.block_table + static_cast<int64_t>(seq_b) * p.mbps;
        int t = 0;   // tiles issued
        bool ok = true;
        for (int w0 = lb_begin; ok && w0 < lb_end; w0 += kBidWindow) {
            const int wn = min(kBidWindow, lb_end - w0);
            __syncwarp();
            for (int i = lane; i < wn; i += 32) bids[i] = (w0 + i < p.mbps) ? bt_row[w0 + i] : -1;
            __syncwarp();
            if constexpr (kDecode) {
                if (lane == 0) mbar_arrive(bready);
            }
            if (lane == 0) {
                int s = t % kStages;
                uint32_t ph = static_cast<uint32_t>(t / kStages) & 1u;
                for (int b0 = 0; b0 < wn; b0 += kBlocksPerTile) {
                    if (t >= kStages && !mbar_wait(&empty[s], ph ^ 1u, status, &ks->abort)) {
                        ok = false;
                        break;
                    }
                    int phys[kBlocksPerTile];
                    uint32_t bytes = 0;
#pragma unroll
                    for (int j = 0; j < kBlocksPerTile; ++j) {
                        phys[j] = -1;
                        if (b0 + j < wn) {
                            const int pb = bids[b0 + j];
                            if (pb < 0 || pb >= p.num_blocks) {
                                ks->bad = 1;
                                set_status(status, IDX_ERR_DEVICE_CHECK);
                            } else {
                                phys[j] = pb;
                                bytes += kBlockTx;
                            }
                        }
                    }
                    uint8_t* a_s = a_tiles + s * plan.a_stage_bytes;
                    mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
                    for (int j = 0; j < (kDecode ? kBlocksPerTile / 2 : kBlocksPerTile); ++j) {
                        if (phys[j] < 0) continue;
                        if constexpr (kFp8) {
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, phys[j], pol);
                            bulk_load(scales + s * 128 + j * kBs,
                                      p.pool + static_cast<int64_t>(phys[j]) * p.block_bytes + kBs * 128,
                                      kBs * 4, &full[s], pol);
                        } else {
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, phys[j], pol);
                            tma_load_3d(a_s + 16384 + j * kBs * 128, &tmap, &full[s], 64, 0, phys[j], pol);
                        }
                    }
                    ++t;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            t = __shfl_sync(0xffffffffu, t, 0);
        }
        if (lane == 0) {
            // copies still in flight (only when a wait gave up) must land before exit
            for (int u = max(0, t - kStages); u < t; ++u)
                mbar_wait(&full[u % kStages], static_cast<uint32_t>(u / kStages) & 1u, status, nullptr);
            mbar_wait(qbar, 0, status, nullptr);
        }
        __syncwarp();
        if constexpr (kDecode) cluster_wait();
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = idesc_make(kFp8, kTileKeys, kN);
        const uint32_t q_base = smem_u32(qtile);
        if constexpr (kDecode) {
            // the B tile was written by the cluster's ranks
            if (!mbar_wait_cluster(qready, 0, status)) ks->abort = 1;
            fence_proxy_async_smem();
        }
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % kStages;
            const uint32_t ph = static_cast<uint32_t>(t / kStages) & 1u;
            const int a = t & 1;
            const uint32_t aph = static_cast<uint32_t>(t >> 1) & 1u;
            if (!mbar_wait(&full[s], ph, status, &ks->abort)) break;
            if (t >= 2 && !mbar_wait(&tempty[a], aph ^ 1u, status, &ks->abort)) break;
            tc_fence_after();
            const uint32_t a_base = smem_u32(a_tiles + s * plan.a_stage_bytes);
            const uint32_t d = tmem + static_cast<uint32_t>(a * kN);
#pragma unroll
            for (int k = 0; k < kKSteps; ++k) {
                uint32_t ao, bo;
                if constexpr (kFp8) {
                    ao = k * 32;
                    bo = k * 32;
                } else {
                    ao = (k >> 2) * 16384 + (k & 3) * 32;
                    bo = (k >> 2) * (kN * 128) + (k & 3) * 32;
                }
                if constexpr (kFp8)
                    mma_fp8(d, sdesc_sw128(a_base + ao), sdesc_sw128(q_base + bo), idesc, k > 0);
                else
                    mma_bf16(d, sdesc_sw128(a_base + ao), sdesc_sw128(q_base + bo), idesc, k > 0);
            }
            mma_commit(&empty[s]);
            mma_commit(&tfull[a]);
        }
        // every MMA issued above has finished once mdone completes
        mma_commit(mdone);
        mbar_wait(mdone, 0, status, nullptr);
    } else if (kDecode && warp == 3) {
        // Decode: the second key issuer, for the second half of every tile's
        // blocks (warp 0 counts the whole tile's bytes, so these copies may
        // land before its expect-tx: the phase cannot complete before that
        // arrival).  A decode chunk is at most 8192 keys, at most 256 blocks
        // of 32 keys: one window of block ids holds it all.
        static_assert(8192 / 32 <= kBidWindow, "one block-id window per decode chunk");
        if (lane == 0 && ntiles > 0) {
            const int* bids = reinterpret_cast<const int*>(smem + plan.bid_off);
            const uint64_t pol = policy_evict_first();
            const int nblk = (key_end + kBs - 1) / kBs - key_begin / kBs;
            int t = 0;   // tiles issued
            if (mbar_wait(bready, 0, status, &ks->abort)) {
                int s = 0;
                uint32_t ph = 0;
                for (int b0 = 0; b0 < nblk; b0 += kBlocksPerTile) {
                    if (t >= kStages && !mbar_wait(&empty[s], ph ^ 1u, status, &ks->abort)) break;
                    uint8_t* a_s = a_tiles + s * plan.a_stage_bytes;
#pragma unroll
                    for (int j = kBlocksPerTile / 2; j < kBlocksPerTile; ++j) {
                        const int pb = b0 + j < nblk ? bids[b0 + j] : -1;
                        if (pb < 0 || pb >= p.num_blocks) continue;   // warp 0 flags a bad id
                        if constexpr (kFp8) {
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, pb, pol);
                            bulk_load(scales + s * 128 + j * kBs,
                                      p.pool + static_cast<int64_t>(pb) * p.block_bytes + kBs * 128, kBs * 4,
                                      &full[s], pol);
                        } else {
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, pb, pol);
                            tma_load_3d(a_s + 16384 + j * kBs * 128, &tmap, &full[s], 64, 0, pb, pol);
                        }
                    }
                    ++t;
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // copies still in flight (only when a wait gave up) must land before exit
            for (int u = max(0, t - kStages); u < t; ++u)
                mbar_wait(&full[u % kStages], static_cast<uint32_t>(u / kStages) & 1u, status, nullptr);
        }
        __syncwarp();
        cluster_wait();
    } else if (warp >= 4) {
        // epilogue: one key row per thread; warp w reads TMEM lane quadrant
        // w % 4 and queries j0 .. j0 + kQPer - 1 of the tile
        const int qd = warp & 3;
        const int row = qd * 32 + lane;
        const int j0 = ((warp - 4) >> 2) * kQPer;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
        if constexpr (kDecode) {
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(qready, 0, status))) ks->abort = 1;   // w'
        }
        // one query per warp: its 64 head weights stay in registers for the
        // whole loop, and TMEM is read 16 columns at a time to make room.
        // (Reloading them per tile made the shared-memory load pipe the
        // prefill kernel's limit: a broadcast load fills the 32 lanes'
        // registers at 128 bytes per wavefront, 64 wavefronts per warp-tile.)
        static_assert(kQPer == 1, "one query per epilogue warp");
        unsigned long long wr[32];
        const unsigned long long* wq2 = reinterpret_cast<const unsigned long long*>(wq + j0 * 64);
#pragma unroll
        for (int i = 0; i < 32; ++i) wr[i] = wq2[i];
        int vis_rows = 0, vis_pos = 0;
        int64_t out_row = 0;
        if constexpr (!kDecode) {
            vis_rows = ks->nrows;
            vis_pos = j0 < vis_rows ? ks->pos[j0] : -1;
            out_row = static_cast<int64_t>(ks->row0 + j0) * p.score_stride;
        }
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % kStages;
            const uint32_t ph = static_cast<uint32_t>(t / kStages) & 1u;
            const int a = t & 1;
            const uint32_t aph = static_cast<uint32_t>(t >> 1) & 1u;
            // waits are combined over the warp so that every lane leaves together
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[a], aph, status, &ks->abort))) break;
            tc_fence_after();
            float kscale = 1.0f;
            if constexpr (kFp8) {
                if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, status, &ks->abort))) break;
                kscale = scales[s * 128 + row];
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            // sum_h w'[h] * max(D[h], 0): even and odd heads in the two lanes of
            // a packed fp32 pair, added at the end
            float res[kQPer];
            {
                // max(D, 0) as D + |D| = 2 max(D, 0) exactly: an add with an
                // absolute-value operand on the FMA pipe (the ALU pipe, where
                // a max goes, was the epilogue's busiest; moving all 64 there
                // measured fastest, and one accumulator chain faster than
                // two), the factor 2 removed at the end (exact); 16 heads
                // per TMEM load
                unsigned long long acc = 0ull;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[16];
                    tmem_ld16(lane_base + static_cast<uint32_t>(a * kN + j0 * 64 + 16 * c), v);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        acc = f2_fma(wr[8 * c + i],
                                     f2_pack(v[2 * i] + fabsf(v[2 * i]), v[2 * i + 1] + fabsf(v[2 * i + 1])), acc);
                }
                const float2 pr = f2_unpack(acc);
                res[0] = kscale * (0.5f * (pr.x + pr.y));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
            const int key = key_begin + t * kTileKeys + row;
            if constexpr (kDecode) {
                const bool valid = key < key_end;
                const uint32_t kk = score_key(res[0]);
                if (valid) cscores[key - key_begin] = res[0];
                hist_add_warp(hist, key_bin(kk), valid);
            } else {
                if (key <= vis_pos) p.scores[out_row + key] = res[0];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 2 * kN);

    if constexpr (!kDecode) {
        if (ks->bad || ks->abort) {
            if (tid < ks->nrows) atomicOr(&p.rowflag[ks->row0 + tid], 1u);
        }
        return;
    } else {
        // ------------------------------------------------ cluster top-k
        // The segment's exact top-k by the whole cluster.  A one-segment
        // sequence writes its outputs directly.  A longer one writes each
        // segment's sorted top-k to the workspace (a run of k composites,
        // zero-padded); the last cluster of the sequence to finish then merges
        // the runs with a second selection over them.
        const int b = seq_b;
        const int n = key_end - key_begin;
        const int k = p.topk;
        const bool single = ks->nseg == 1;
        const uint32_t rank = cluster_rank();
        int32_t* oi = p.out_idx + static_cast<int64_t>(b) * k;
        float* os = p.out_score ? p.out_score + static_cast<int64_t>(b) * k : nullptr;
        uint64_t* runs_b = p.cand + static_cast<int64_t>(b) * p.cand_cap;
        uint64_t* run = runs_b + static_cast<int64_t>(ks->seg) * k;
        uint64_t* lists = reinterpret_cast<uint64_t*>(a_tiles);   // 3 x kClCap composites
        ClusterBufs B{hist,
                      reinterpret_cast<uint32_t*>(qtile),
                      reinterpret_cast<uint32_t*>(lists),
                      reinterpret_cast<uint32_t*>(lists + kClCap),
                      lists,
                      lists + kClCap,
                      lists + 2 * kClCap,
                      cbar,
                      plan.recv_bytes ? reinterpret_cast<uint32_t*>(smem + plan.recv_off) : nullptr};
        // the chunk's scores as (score key, key index): four scores per load,
        // two loads in flight per iteration, the same trip count in every lane
        auto walk_keys = [&](auto f) {
            const float4* c4 = reinterpret_cast<const float4*>(cscores);
            const int nj = (n + 3) / 4;
            const int njr = (nj + kThreads - 1) / kThreads * kThreads;
#pragma unroll 2
            for (int j = tid; j < njr; j += kThreads) {
                const float4 x = j < nj ? c4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                const int i = 4 * j;
                f(score_key(x.x), key_begin + i, i < n);
                f(score_key(x.y), key_begin + i + 1, i + 1 < n);
                f(score_key(x.z), key_begin + i + 2, i + 2 < n);
                f(score_key(x.w), key_begin + i + 3, i + 3 < n);
            }
        };
        auto walk = [&](auto f) {
            walk_keys([&](uint32_t key, int idx, bool v) { f(make_comp(key, idx), v); });
        };
        auto collect_keys = [&](uint32_t kthr, uint64_t* dst, uint32_t cap, uint64_t* seg, uint32_t* wsum) {
            return block_collect_keys(walk_keys, kthr, dst, cap, seg, wsum);
        };
        auto emit_out = [&](int r, uint64_t c) {
            oi[r] = comp_index(c);
            if (os) os[r] = key_score(comp_key(c));
        };
        auto pad_out = [&](int count) {
            for (int j = max(count, 0) + tid; j < k; j += kThreads) {
                oi[j] = -1;
                if (os) os[j] = -INFINITY;
            }
        };
        // one selection (one copy of its code) for both cases
        const int count = cluster_select(
            walk, collect_keys,
            [&](int r, uint64_t c) {
                if (single) emit_out(r, c);
                else run[r] = c;
            },
            B, k, ks->bad != 0 || ks->abort != 0, &ks->cs, status);
        if (single) {
            if (rank == 0) pad_out(count);
            return;
        }
        if (rank == 0) {
            if (count < 0) {
                if (tid == 0) atomicOr(p.seqflag + b, 1u);
            } else {
                for (int j = count + tid; j < k; j += kThreads) run[j] = 0ull;
            }
        }
        // the cluster's run is written: rank 0 takes the sequence's ticket and
        // tells every CTA whether this cluster is the last one
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            fence_acq_rel_cluster();
            mbar_arrive_remote(dsmem_addr(rdone, 0));
        }
        if (rank == 0) {
            if (!mbar_wait_cluster(rdone, 0, status)) ks->abort = 1;
            if (tid < kCl) {
                uint32_t last = 0;
                if (tid == 0) {
                    __threadfence();
                    last = (atomicAdd(p.ctr + b, 1u) == static_cast<uint32_t>(ks->nseg - 1)) ? 1u : 0u;
                }
                last = __shfl_sync(0xffu, last, 0);
                dsmem_st_async_u32(dsmem_addr(&ks->merge_last, static_cast<uint32_t>(tid)), last,
                                   dsmem_addr(rlast, static_cast<uint32_t>(tid)));
            }
        }
        if (!mbar_wait_cluster(rlast, 0, status) || ks->merge_last == 0u) return;

        // ------------------------------------------------ sequence merge (last cluster)
        // CTA r takes entries r, r + 8, r + 16, ... of every run, so each CTA
        // holds about an eighth of the candidates; they are staged in shared
        // memory where its scores were (zero entries are padding).
        __threadfence();
        const int nseg = ks->nseg;
        const int per_run = (k - static_cast<int>(rank) + kCl - 1) / kCl;
        const int m = nseg * per_run;
        const int cap_stage = (plan.bid_off - plan.raw_off) / 8;   // the scores region
        uint64_t* staged = reinterpret_cast<uint64_t*>(cscores);
        const bool fits = m <= cap_stage;
        auto run_entry = [&](int i) {
            const int j = i / per_run;
            const int e = static_cast<int>(rank) + (i - j * per_run) * kCl;
            return static_cast<uint64_t>(
                __ldcg(reinterpret_cast<const unsigned long long*>(runs_b) + static_cast<int64_t>(j) * k + e));
        };
        if (fits) {
#pragma unroll 4
            for (int i = tid; i < m; i += kThreads) staged[i] = run_entry(i);
        }
        const int mround = (m + kThreads - 1) / kThreads * kThreads;
        auto walk_runs = [&](auto f) {
            for (int i = tid; i < mround; i += kThreads) {
                uint64_t c = 0ull;
                if (i < m) c = fits ? staged[i] : run_entry(i);
                f(c, c != 0ull);
            }
        };
        for (int i = tid; i < kHistBins; i += kThreads) hist[i] = 0;
        __syncthreads();
        walk_runs([&](uint64_t c, bool v) { hist_add_warp(hist, key_bin(comp_key(c)), v); });
        const uint32_t flagged = __ldcg(p.seqflag + b);
        B.cbar = cbar2;
        auto collect_runs = [&](uint32_t kthr, uint64_t* dst, uint32_t cap, uint64_t* seg, uint32_t* wsum) {
            const uint64_t thr = static_cast<uint64_t>(kthr) << 32;
            return block_collect_warp(walk_runs, [&](uint64_t c) { return c >= thr; }, dst, cap, seg, wsum);
        };
        const int total = cluster_select(walk_runs, collect_runs, emit_out, B, k, flagged != 0u, &ks->cs, status);
        if (rank == 0) {
            pad_out(total);
            if (tid == 0) {
                p.ctr[b] = 0;
                p.seqflag[b] = 0;
                p.seqcnt[b] = 0;
            }
        }
    }
}

}  // namespace dsaidx
