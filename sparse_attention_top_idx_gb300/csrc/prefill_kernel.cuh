// prefill_kernel.cuh -- the causal-chunk scoring kernel for sm_103a.
//
// score[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])  (fp32 accumulation), the
// compressed query-key relevance score of "The Hypothesis That Refused to Die"
// (section "The Context"), for the query rows of a causal chunk
// (_score_topk_prefill in "DeepSeek-V4 index_topk=1024 sparse indexer can't
// recall verbatim lines", ROCm/ATOM issue #1507, section "Root cause found"),
// read straight from the paged blocks through the block table the way that
// issue's paged MQA logits read them (section "How it was isolated").
//
// Work unit: a group of up to kPrefillQT = 4 consecutive query rows of one
// sequence against every key they can see (N = 256 query-heads), groups with
// the longest rows first.  The contraction D[s, (t, h)] = sum_d k[s, d]
// q[t, h, d] runs on the 5th-gen tensor cores: M = 128 keys (A, K-major,
// TMA-loaded 64- or 32-row boxes of the paged blocks, 128-byte swizzle), N =
// 256 (B, quantised by the CTA itself into shared memory), K = 128, fp32
// accumulators in TMEM (two buffers so the epilogue of tile i overlaps the MMA
// of tile i + 1).  fp8 keys use kind::f8f6f4 (e4m3 x e4m3), bf16 keys
// kind::f16.
//
// Warp roles (640 threads): warp 0 lane 0 starts the query rows' bulk copy,
// then the warp prefetches block ids and lane 0 issues the key TMA; warps
// 1..19 quantise the queries into the B tile; warp 1 owns TMEM and its lane 0
// issues the MMAs; warps 4..19 (one per TMEM lane quadrant and query; each
// lane sums a quarter of the heads of four key rows, then the four lanes of
// a row group combine theirs) run the epilogue ks[s] * sum_h w'[t, h] *
// max(D, 0) with the head weights held in registers and write the causally
// visible scores to the workspace for the row select kernel.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "headsum.cuh"
#include "internal.h"
#include "qprep.cuh"
#include "topk.cuh"

namespace dsaidx {

struct PrefillShared {
    uint32_t tmem_base;
    int abort;          // a role gave up on a bounded wait
    int bad;            // a block id failed its check
    int unit_b, key_begin, key_end, seq_len, nrows, row0, nq;
    int pos[kPrefillQT];
    uint32_t grp[kThreads];   // group-count scan (first 256 threads)
};
static_assert(sizeof(PrefillShared) <= 4096, "PrefillShared must fit the misc region");

template <bool kFp8, int kBs>
__global__ void __maxnreg__(96)
    prefill_score_kernel(const __grid_constant__ CUtensorMap tmap, const ScoreParams p) {
    constexpr int kQT = kPrefillQT;
    constexpr int kBlock = kPrefillThreads;
    constexpr int kEpiWarps = 16;                          // per (TMEM buffer, lane quadrant, query pair)
    constexpr int kN = 64 * kQT;
    constexpr int kBlocksPerTile = kTileKeys / kBs;
    constexpr int kKSteps = kFp8 ? 4 : 8;
    constexpr uint32_t kBlockTx = kFp8 ? (kBs * 128) : (kBs * 256);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const SmemPlan plan = make_plan(kFp8, kQT, 0);
    const int kStages = plan.stages;
    uint8_t* a_tiles = smem + plan.a_off;
    uint8_t* qtile = smem + plan.q_off;
    float* wq = reinterpret_cast<float*>(smem + plan.w_off);
    uint8_t* raw = smem + plan.raw_off;                     // staged query rows (bf16)
    PrefillShared* ks = reinterpret_cast<PrefillShared*>(smem + plan.misc_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
    uint64_t* full = bars;                 // [stages] TMA -> MMA
    uint64_t* empty = bars + 8;            // [stages] MMA -> TMA
    uint64_t* tfull = bars + 16;           // [2] MMA -> epilogue
    uint64_t* tempty = bars + 18;          // [2] epilogue -> MMA
    uint64_t* mdone = bars + 20;           // MMA drain at exit
    uint64_t* qbar = bars + 21;            // query rows staged

    const int tid = threadIdx.x;
    const int warp = warp_id(), lane = lane_id();
    int32_t* status = p.status;

    // ------------------------------------------------------------ work unit
    // group g of up to 4 rows of one sequence; longest rows first
    {
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
    // Warp 0: lane 0 starts the query rows' load first with their head
    // weights, so its latency overlaps the rest of the set-up; lane 1
    // initialises the other barriers in parallel.
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(qbar, 1);
            fence_mbar_init();
            const uint64_t pol_q = policy_evict_first();
            const int nr = ks->nrows * 64;
            const int64_t g0 = static_cast<int64_t>(ks->row0) * 64;
            mbar_arrive_expect_tx(qbar, static_cast<uint32_t>(nr) * (kHeadDim * 2 + 4));
            bulk_load(raw, p.q + g0 * kHeadDim, static_cast<uint32_t>(nr) * kHeadDim * 2, qbar, pol_q);
            bulk_load(wq, p.w + g0, static_cast<uint32_t>(nr) * 4, qbar, pol_q);
            tma_prefetch_desc(&tmap);
            ks->abort = 0;
            ks->bad = 0;
        } else if (lane == 1) {
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(&tfull[a], 1);
                mbar_init(&tempty[a], kEpiWarps / 2);
            }
            mbar_init(mdone, 1);
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc(&ks->tmem_base, 2 * kN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ks->tmem_base;

    // The query rows are in flight since the set-up; warps 1..19 build the B
    // tile and meet on a named barrier while warp 0 starts the key loads.
    if (warp != 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(qbar, 0, status, &ks->abort))) ks->abort = 1;
        prep_queries<kFp8, kQT>(raw, ks->nrows, qtile, wq, tid - 32, kBlock - 32);
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, %0;" ::"r"(kBlock - 32) : "memory");
    }

    // ------------------------------------------------------------ main loop
    if (warp == 0) {
        // The whole warp loads the block ids of up to kBidWindow blocks at a
        // time into shared memory, then lane 0 alone issues the key TMA of
        // every tile whose blocks lie in that window (the window holds whole
        // tiles), with the stage and phase kept as running counters.
        int* bids = reinterpret_cast<int*>(smem + plan.bid_off);
        const uint64_t pol = policy_evict_last();
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
            if (lane == 0) {
                int s = t % kStages;
                uint32_t ph = static_cast<uint32_t>(t / kStages) & 1u;
                for (int b0 = 0; b0 < wn; b0 += kBlocksPerTile) {
                    if (t >= kStages && !mbar_wait(&empty[s], ph ^ 1u, status, &ks->abort, p.wait_ns)) {
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
                    for (int j = 0; j < kBlocksPerTile; ++j) {
                        if (phys[j] < 0) continue;
                        if constexpr (kFp8) {
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, phys[j], pol);
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
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        constexpr uint32_t idesc = idesc_make(kFp8, kTileKeys, kN);
        const uint32_t q_base = smem_u32(qtile);
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % kStages;
            const uint32_t ph = static_cast<uint32_t>(t / kStages) & 1u;
            const int a = t & 1;
            const uint32_t aph = static_cast<uint32_t>(t >> 1) & 1u;
            if (!mbar_wait(&full[s], ph, status, &ks->abort, p.wait_ns)) break;
            if (t >= 2 && !mbar_wait(&tempty[a], aph ^ 1u, status, &ks->abort, p.wait_ns)) break;
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
    } else if (warp >= 4) {
        // epilogue: two groups of 8 warps, group g taking the tiles of TMEM
        // buffer g (tiles t = g, g + 2, ...), so that one group works while
        // the other waits for its next accumulator.  Epilogue warp e = w - 4
        // reads TMEM lane quadrant qd = w % 4 (32 keys) for queries
        // 2 (e / 8) and 2 (e / 8) + 1 of the group; each lane keeps the
        // weights of its 16 heads of both queries in registers (reloading
        // the second query's per tile measured 4 % slower than the spill of
        // 24 bytes that holding both costs; key scales in a shared-memory ring
        // instead of the prefetch below, 15 % slower) and writes the scores
        // of quadrant row head_sum_row(lane).
        const int e = warp - 4;
        const int qd = warp & 3;
        const int g = (e >> 2) & 1;
        const int jq = 2 * (e >> 3);
        const int orow = qd * 32 + head_sum_row(lane);
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
        unsigned long long wr0[8], wr1[8];
        load_head_weights(wq + jq * 64, lane, wr0);
        load_head_weights(wq + (jq + 1) * 64, lane, wr1);
        const int vis0 = jq < ks->nrows ? ks->pos[jq] : -1;
        const int vis1 = jq + 1 < ks->nrows ? ks->pos[jq + 1] : -1;
        float* out0 = p.scores + static_cast<int64_t>(ks->row0 + jq) * p.score_stride;
        float* out1 = out0 + p.score_stride;
        // key scale of this lane's key in tile t, read from the pool (0 past
        // the keys or for a bad block id, whose rows are flagged anyway)
        const int* bt_row = p.block_table + static_cast<int64_t>(seq_b) * p.mbps;
        auto scale_of = [&](int t) -> float {
            if constexpr (!kFp8) {
                return 1.0f;
            } else {
                const int key = key_begin + t * kTileKeys + orow;
                if (t >= ntiles || key >= key_end || key / kBs >= p.mbps) return 0.0f;
                const int pb = __ldg(bt_row + key / kBs);
                if (pb < 0 || pb >= p.num_blocks) return 0.0f;
                return __ldg(reinterpret_cast<const float*>(p.pool + static_cast<int64_t>(pb) * p.block_bytes +
                                                            kBs * 128) + (key % kBs));
            }
        };
        float sc0 = scale_of(g);
        for (int t = g; t < ntiles; t += 2) {
            const uint32_t aph = static_cast<uint32_t>(t >> 1) & 1u;
            const float kscale = sc0;
            sc0 = scale_of(t + 2);
            // waits are combined over the warp so that every lane leaves together
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[g], aph, status, &ks->abort, p.wait_ns))) break;
            tc_fence_after();
            const uint32_t col = lane_base + static_cast<uint32_t>(g * kN + jq * 64);
            const float h0 = head_sum_rows(col, wr0, lane, [] {});
            // every TMEM read of the buffer by this warp has completed when release runs
            const float h1 = head_sum_rows(col + 64, wr1, lane, [&] {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[g]);
            });
            const int key = key_begin + t * kTileKeys + orow;
            if (key <= vis0) out0[key] = kscale * (0.5f * h0);
            if (key <= vis1) out1[key] = kscale * (0.5f * h1);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 2 * kN);
    if (ks->bad || ks->abort) {
        if (tid < ks->nrows) atomicOr(&p.rowflag[ks->row0 + tid], 1u);
    }
}

}  // namespace dsaidx
