// decode_kernel.cuh -- fused decode score + top-k for sm_103a (one query per
// sequence, every key of the sequence visible).
//
// score[s] = sum_h w[h] * ReLU(q[h] . k[s])  (fp32 accumulation), the
// compressed query-key score of "The Hypothesis That Refused to Die" (section
// "The Context"), read straight from the paged index-key cache the way the
// paged MQA logits of "DeepSeek-V4 index_topk=1024 sparse indexer can't
// recall verbatim lines" (ROCm/ATOM issue #1507, section "How it was
// isolated") read it, followed by that section's per-row top-k
// (top_k_per_row_decode) in the same kernel: the scores stay on chip.
//
// Work decomposition.  A sequence of S keys is cut into segments of up to
// kDecCl chunks; a chunk (at most kDecChunkMax keys, a multiple of the
// 128-key tile) is scored by one CTA.  The grid is a set of persistent
// thread-block clusters of kDecCl CTAs that take the segments (units) of the
// flattened list over all sequences: cluster c starts with unit c and then
// takes units from a counter in the workspace (rank 0 draws the next unit
// while the current one is selected and sends it to the cluster), so no
// cluster is launched idle and clusters that start late find less work.
//
// One unit, in every CTA of the cluster (warp roles):
//   warp 0     lane 0 starts the copy of this CTA's 8 of the sequence's 64
//              bf16 query rows and their head weights, the warp loads the
//              chunk's block ids, then lane 0 issues one TMA box per paged
//              block (64 or 32 rows of 128 bytes, 128-byte swizzle) into a
//              ring of stages;
//   warp 1     owns TMEM; lane 0 issues tcgen05.mma (M = 128 keys, N = 64
//              heads, K = 128) into a double-buffered fp32 accumulator;
//   warps 2-5  quantise this CTA's 8 query rows into its 1 KB block of the B
//              operand (16 lanes per row) and send the block and the rows'
//              w' to the other 7 CTAs (bulk shared-to-shared copies counted
//              on their query barrier), so the B tile is built once per
//              cluster;
//   warps 4-7  run the epilogue (head_sum_rows: each lane sums 16 of the 64
//              heads of four key rows from .16x256b TMEM loads, a shuffle
//              step leaves it one row's sum), ks[s] * sum_h w'[h] * max(D, 0)
//              with the head weights in registers and the key scale loaded
//              from the cache two tiles ahead; the score goes to shared memory
//              and into a histogram of the chunk at 1/16 octave (score key >> 19).
// Selection, by the 8 CTAs together with two one-way exchanges (st.async,
// counted on the receiver's mbarrier; a remote shared-memory load would cost
// a round trip):
//   1. every CTA sends every CTA its window: the 256 histogram bins below its
//      largest score, its key count and largest key (528 bytes);
//   2. every CTA sums the windows over the 256 bins below the segment's
//      largest: the bin of the segment's k-th largest score (the boundary)
//      and, per bin at or above it, every CTA's count, so the place of each
//      bin's entries in a bin-major pool (bins from the top, CTAs in rank
//      order within a bin) is known to every CTA;
//   3. every CTA writes each of its candidates (scores in bins at or above
//      the boundary) to its place in every CTA's pool: nothing is sorted;
//   4. every CTA ranks one eighth of the pool -- the entries of higher bins
//      plus the larger entries of the same bin -- and writes those of rank
//      < k to the output (or the segment's run).
// A crowded boundary bin (many equal or nearly equal scores) takes a slower
// path: the chunks' scores go through a per-cluster global scratch to one
// CTA, which selects with radix refinement (segsel.cuh).  A sequence longer
// than one segment writes each segment's sorted top-k as a run and its bin
// counts (and largest bin) to the sequence's histogram in the workspace; the
// CTA that ends the sequence's last segment (a ticket) merges: the histogram
// gives the boundary bin and, runs being sorted, only each run's prefix at or
// above it is read.
//
// Every mbarrier wait is bounded (%globaltimer); a wait that runs out sets
// IDX_ERR_TIMEOUT, the CTA stops streaming (draining its copies and MMAs),
// keeps taking part in the cluster protocol with flagged (-1) results, frees
// TMEM and exits.  Within a cluster, one hardware cluster barrier per unit
// orders the reuse of the receive areas.
#pragma once

#include "common.cuh"
#include "headsum.cuh"
#include "internal.h"
#include "qprep.cuh"
#include "segsel.cuh"
#include "topk.cuh"

namespace dsaidx {

// Phase stamps (a diagnostic build only, -DDSAIDX_PHASE_STAMPS): %globaltimer
// at the phase boundaries of the first kPhaseUnits units of every CTA, read
// back by idx_phase_stamps (decode.cu) and printed by the package's phases
// module.  Slots: 0 kernel entry, 1 set-up done, 2 unit located, 3 query rows
// landed, 4 B tile complete, 5 first key tile landed, 6 stream done,
// 7 window sent, 8 windows received, 9 boundary known, 10 pool complete,
// 11 ranks written, 12 unit end, 13 loop done, 14 exit.
constexpr int kPhaseCtas = 2048;
constexpr int kPhaseUnits = 4;
constexpr int kPhaseSlots = 16;
#ifdef DSAIDX_PHASE_STAMPS
__device__ unsigned long long g_phase[kPhaseCtas][kPhaseUnits][kPhaseSlots];
#define DSAIDX_PHASE(it, slot)                                                   \
    do {                                                                         \
        if ((it) < kPhaseUnits && blockIdx.x < kPhaseCtas)                       \
            g_phase[blockIdx.x][(it)][(slot)] = global_timer_ns();               \
    } while (0)
#else
#define DSAIDX_PHASE(it, slot) \
    do {                       \
    } while (0)
#endif

struct DecShared {
    uint32_t tmem_base;
    int abort;              // a pipeline wait of this CTA gave up (sticky)
    int bad;                // this unit: a block id failed its check
    int ub, useg, uS;       // the located unit: sequence, segment, its length
    uint32_t unext[2];      // next units, sent by rank 0
    uint32_t last;          // this CTA ends its sequence (merges)
    uint32_t emax[4];       // epilogue warps' largest score keys
    uint32_t nmine;         // crowded bins listed for the ranking
    int cnt[kDecCl];        // the CTAs' candidate counts (-1: not known from the window)
    uint32_t scan[kThreads / 32];
    SegSelSmem sel;
};
static_assert(sizeof(DecShared) <= kDecMiscBytes, "DecShared must fit the misc region");

template <bool kFp8, int kBs>
__global__ void __maxnreg__(120) decode_kernel(const __grid_constant__ CUtensorMap tmap, const ScoreParams p) {
    constexpr int kN = 64;                                // B rows: the 64 heads
    constexpr int kBlocksPerTile = kTileKeys / kBs;
    constexpr int kKSteps = kFp8 ? 4 : 8;                 // K = 128 in steps of 32 bytes
    constexpr uint32_t kBoxBytes = kBs * 128;             // one TMA box: a block's code rows (or half rows)
    constexpr int kQuantThreads = kThreads - 64;          // warps 2..7 take part in the query stage
    constexpr int kQRows = kN / kDecCl;                   // query rows each CTA quantises
    // bytes each other CTA sends: its rows' block of the B tile (each K-half
    // for bf16) and their w'
    constexpr uint32_t kQPushBytes = kQRows * 128 * (kFp8 ? 1 : 2) + kQRows * 4;
    static_assert(kQRows == 8, "one 8-row swizzle atom (1 KB) of the B tile per CTA");
    constexpr int kEpiWarps = 4;
    constexpr uint32_t kWinBytes = kWinWords * 4;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const DecPlan plan = dec_plan(kFp8);
    const int kStages = plan.stages;
    uint8_t* a_tiles = smem + plan.a_off;
    uint8_t* raw = smem + plan.raw_off;                                 // staged bf16 query rows
    float* wraw = reinterpret_cast<float*>(raw + kQRows * kHeadDim * 2);
    uint32_t* chist = reinterpret_cast<uint32_t*>(raw);                 // the chunk's 16-bit histogram (aliased)
    float* csc = reinterpret_cast<float*>(smem + plan.sc_off);          // this chunk's scores
    uint32_t* win = reinterpret_cast<uint32_t*>(smem + plan.win_off);   // [kDecCl][kWinWords]
    uint64_t* pool = reinterpret_cast<uint64_t*>(smem + plan.pool_off); // the cluster's candidates, bin-major
    uint8_t* qtile = smem + plan.q_off;
    float* wq = reinterpret_cast<float*>(smem + plan.w_off);
    int* bids = reinterpret_cast<int*>(smem + plan.bid_off);
    DecShared* ks = reinterpret_cast<DecShared*>(smem + plan.misc_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + plan.bar_off);
    uint64_t* full = bars;            // [stages] TMA -> MMA
    uint64_t* empty = bars + 4;       // [stages] MMA -> TMA
    uint64_t* tfull = bars + 8;       // [2] MMA -> epilogue
    uint64_t* tempty = bars + 10;     // [2] epilogue -> MMA
    uint64_t* mdone = bars + 12;      // MMA drain after a timeout
    uint64_t* qbar = bars + 13;       // query rows and weights staged
    uint64_t* qready = bars + 14;     // B tile and w' written (one arrive per query-stage warp)
    uint64_t* wbar = bars + 15;       // every other CTA's window has arrived
    uint64_t* lbar = bars + 16;       // every other CTA's candidates have arrived
    uint64_t* ubar = bars + 17;       // [2] the next unit has arrived
    uint64_t* rbar = bars + 19;       // coordinating CTA: every CTA wrote its part of the unit
    // after the stream the key stages hold the selection's tables and scratch
    // (slow path, merge: the chunk's scores are in global scratch or done with)
    uint32_t* shist = reinterpret_cast<uint32_t*>(csc);                 // [4096] selection histogram
    uint64_t* sbuf = reinterpret_cast<uint64_t*>(a_tiles);              // [4096] selection buffer

    const int tid = threadIdx.x;
    const int warp = warp_id(), lane = lane_id();
    const uint32_t rank = cluster_rank();
    if (tid == 0) DSAIDX_PHASE(0, 0);
    // a kernel launched next with programmatic serialization (the next key
    // store) may be scheduled now; it waits for this grid to finish before it
    // touches anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int cl = static_cast<int>(blockIdx.x) / kDecCl;
    const int ncl = static_cast<int>(gridDim.x) / kDecCl;
    int32_t* status = p.status;
    const unsigned long long wlim = p.wait_ns;   // limit of the pipeline waits

    // ------------------------------------------------------------ set-up (once)
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(qbar, 1);
            mbar_init(qready, kQuantThreads / 32 + 1);   // + the arrival that expects the other CTAs' rows
            mbar_init(wbar, 1);
            mbar_init(lbar, 1);
            mbar_init(&ubar[0], 1);
            mbar_init(&ubar[1], 1);
            mbar_init(rbar, kDecCl);
            fence_mbar_init();
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
                mbar_init(&tempty[a], kEpiWarps);
            }
            mbar_init(mdone, 1);
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc(&ks->tmem_base, 2 * kN);
        tmem_relinquish();
    }
    // every CTA's barriers are initialised before any CTA sends it anything
    // (the first unit's query rows): a whole-cluster barrier, its wait after
    // the scan below
    cluster_arrive();
    // units per sequence, scanned over the block: thread t holds sequences
    // [t * per, t * per + per) and the exclusive prefix of their units; with
    // one sequence per thread it keeps that sequence's length
    const int per = (p.batch + kThreads - 1) / kThreads;
    int mine_u = 0, myS = 0;
    for (int i = 0; i < per; ++i) {
        const int bb = tid * per + i;
        if (bb < p.batch) {
            myS = __ldg(p.seq_lens + bb);
            mine_u += dec_units(myS, p.max_seq_len);
        }
    }
    int excl = mine_u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, excl, o);
        if (lane >= o) excl += y;
    }
    if (lane == 31) ks->scan[warp] = static_cast<uint32_t>(excl);
    excl -= mine_u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int total = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        const int t = static_cast<int>(ks->scan[w]);
        if (w < warp) excl += t;
        total += t;
    }
    const uint32_t tmem = ks->tmem_base;
    cluster_wait();
    // the first half of the per-unit barrier (its wait follows the stream)
    cluster_arrive();
    if (tid == 0) DSAIDX_PHASE(0, 1);

    // Launched with programmatic serialization, the set-up above may overlap
    // the previous kernel in the stream (the key store); nothing below runs
    // before that grid has finished and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint32_t tcnt = 0;   // tiles streamed by this CTA so far (stage, phase and accumulator)
    uint32_t qcnt = 0;   // query loads (qbar / qready phases)
    uint32_t scnt = 0;   // window exchanges (wbar phases)
    uint32_t lcnt = 0;   // list exchanges (lbar phases)
    uint32_t mcnt = 0;   // MMA drains (mdone phases)
    uint32_t rcnt = 0;   // units this CTA coordinated with an rbar round (rbar phases)
    uint32_t issued = 0; // tiles whose copies the producer has issued (running)

    int u = cl;
    for (uint32_t it = 0; u < total; ++it) {
        // read before the barrier below: no wait of this unit can have set it yet
        const bool aborted = ks->abort != 0;
        // ------------------------------------------------ locate the unit
        if (mine_u > 0 && u >= excl && u < excl + mine_u) {
            int acc = excl;
            for (int i = 0; i < per; ++i) {
                const int bb = tid * per + i;
                const int S = per == 1 ? myS : __ldg(p.seq_lens + bb);
                const int nu = dec_units(S, p.max_seq_len);
                if (u < acc + nu) {
                    ks->ub = bb;
                    ks->useg = u - acc;
                    ks->uS = S;
                    break;
                }
                acc += nu;
            }
        }
        if (tid == 0) mbar_arrive_expect_tx(&ubar[(it + 1) & 1u], 4u);   // the next unit's id
        __syncthreads();
        const int b = ks->ub, seg = ks->useg, S = ks->uS;
        if (tid == 0) DSAIDX_PHASE(it, 2);
        const bool valid = S >= 0 && S <= p.max_seq_len;
        const bool live = valid && S > 0;
        const int chunk = live ? dec_chunk(S) : kTileKeys;
        const int nseg = live ? dec_nseg(S) : 1;
        const int seg_begin = seg * kDecCl * chunk;
        const int seg_end = live ? min(S, seg_begin + kDecCl * chunk) : seg_begin;
        const int key_begin = min(seg_end, seg_begin + static_cast<int>(rank) * chunk);
        const int key_end = min(seg_end, key_begin + chunk);
        const int nkeys = key_end - key_begin;
        const int ntiles = (nkeys + kTileKeys - 1) / kTileKeys;
        const bool run = live && !aborted;   // the same value in every thread
        const int lb0 = key_begin / kBs;
        const uint32_t lead = static_cast<uint32_t>(u % kDecCl);   // the unit's coordinating CTA

        if (live) {
            if (warp == 0) {
                if (lane == 0) {
                    ks->bad = 0;
                    // this CTA's query rows (the other CTAs send the rest of the B tile)
                    const uint64_t pol_q = policy_evict_last();   // other clusters may read them too
                    const int64_t row0 = static_cast<int64_t>(b) * kN + static_cast<int64_t>(rank) * kQRows;
                    mbar_arrive_expect_tx(qbar, kQRows * kHeadDim * 2 + kQRows * 4);
                    bulk_load(raw, p.q + row0 * kHeadDim, kQRows * kHeadDim * 2, qbar, pol_q);
                    bulk_load(wraw, p.w + row0, kQRows * 4, qbar, pol_q);
                }
                // the chunk's block ids (a chunk spans at most kDecChunkMax / 32 blocks)
                const int nblk = (key_end + kBs - 1) / kBs - lb0;
                const int* bt_row = p.block_table + static_cast<int64_t>(b) * p.mbps;
                if (run) {
                    for (int i = lane; i < nblk; i += 32) bids[i] = (lb0 + i < p.mbps) ? __ldg(bt_row + lb0 + i) : -1;
                    __syncwarp();
                    // hand the ids to the epilogue warps (their key-scale loads)
                    asm volatile("bar.arrive 2, %0;" ::"r"(32 + 32 * kEpiWarps) : "memory");
                }
                if (run && lane == 0) {
                    // the key stream starts once the query rows have landed: issued
                    // together, the whole grid's first key tiles (several MB) would
                    // queue ahead of the query copies and hold up the MMAs
                    mbar_wait(qbar, qcnt & 1u, status, &ks->abort, wlim);
                    const uint64_t pol = policy_evict_first();
                    uint32_t T = issued;
                    int s = static_cast<int>(T % kStages);
                    uint32_t ph = (T / kStages) & 1u;
                    for (int t = 0; t < ntiles; ++t) {
                        if (T >= static_cast<uint32_t>(kStages) &&
                            !mbar_wait(&empty[s], ph ^ 1u, status, &ks->abort, wlim))
                            break;
                        int phys[kBlocksPerTile];
                        uint32_t nbox = 0;
#pragma unroll
                        for (int j = 0; j < kBlocksPerTile; ++j) {
                            phys[j] = -1;
                            const int bi = t * kBlocksPerTile + j;
                            if (bi < nblk) {
                                const int pb = bids[bi];
                                if (pb < 0 || pb >= p.num_blocks) {
                                    ks->bad = 1;
                                    set_status(status, IDX_ERR_DEVICE_CHECK);
                                } else {
                                    phys[j] = pb;
                                    ++nbox;
                                }
                            }
                        }
                        uint8_t* a_s = a_tiles + s * plan.a_stage_bytes;
                        mbar_arrive_expect_tx(&full[s], nbox * kBoxBytes * (kFp8 ? 1u : 2u));
#pragma unroll
                        for (int j = 0; j < kBlocksPerTile; ++j) {
                            if (phys[j] < 0) continue;
                            tma_load_3d(a_s + j * kBs * 128, &tmap, &full[s], 0, 0, phys[j], pol);
                            if constexpr (!kFp8)
                                tma_load_3d(a_s + 16384 + j * kBs * 128, &tmap, &full[s], 64, 0, phys[j], pol);
                        }
                        ++T;
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    issued = T;
                }
                issued = __shfl_sync(0xffffffffu, issued, 0);
            } else if (warp == 1) {
                if (run && lane == 0) {
                    constexpr uint32_t idesc = idesc_make(kFp8, kTileKeys, kN);
                    const uint32_t q_base = smem_u32(qtile);
                    if (mbar_wait(qready, qcnt & 1u, status, &ks->abort, wlim)) {
                        fence_proxy_async_smem();
                        for (int t = 0; t < ntiles; ++t) {
                            const uint32_t T = tcnt + static_cast<uint32_t>(t);
                            const int s = static_cast<int>(T % kStages);
                            const uint32_t ph = (T / kStages) & 1u;
                            const int a = static_cast<int>(T & 1u);
                            const uint32_t aph = (T >> 1) & 1u;
                            if (!mbar_wait(&full[s], ph, status, &ks->abort, wlim)) break;
                            if (t == 0) DSAIDX_PHASE(it, 5);
                            if (T >= 2 && !mbar_wait(&tempty[a], aph ^ 1u, status, &ks->abort, wlim)) break;
                            tc_fence_after();
                            const uint32_t a_base = smem_u32(a_tiles + s * plan.a_stage_bytes);
                            const uint32_t d = tmem + static_cast<uint32_t>(a * kN);
#pragma unroll
                            for (int k = 0; k < kKSteps; ++k) {
                                if constexpr (kFp8) {
                                    mma_fp8(d, sdesc_sw128(a_base + k * 32), sdesc_sw128(q_base + k * 32), idesc,
                                            k > 0);
                                } else {
                                    const uint32_t ao = (k >> 2) * 16384 + (k & 3) * 32;
                                    const uint32_t bo = (k >> 2) * (kN * 128) + (k & 3) * 32;
                                    mma_bf16(d, sdesc_sw128(a_base + ao), sdesc_sw128(q_base + bo), idesc, k > 0);
                                }
                            }
                            mma_commit(&empty[s]);
                            // (test hook: the first accumulator's signal is withheld, so the
                            // epilogue's bounded wait runs out)
                            if (!(p.withhold && T == 0)) mma_commit(&tfull[a]);
                        }
                    }
                }
                __syncwarp();
            } else {
                // warps 2..5: this CTA's 8 rows of the B tile, 16 lanes per row,
                // then the rows' block and w' to the other CTAs
                if (warp < 6) {
                    if (tid == 64) mbar_arrive_expect_tx(qready, (kDecCl - 1) * kQPushBytes);
                    const bool have = __all_sync(0xffffffffu, mbar_wait(qbar, qcnt & 1u, status, &ks->abort, wlim));
                    if (tid == 64) DSAIDX_PHASE(it, 3);
                    const int rl = (tid - 64) >> 4, part = tid & 15;
                    const int r = static_cast<int>(rank) * kQRows + rl;
                    if (have) {
                        const float wn = quant_row_sixteenth<kFp8>(raw + static_cast<size_t>(rl) * kHeadDim * 2, part,
                                                                   wraw[rl], 0xffffffffu, qtile, r, kN);
                        if (part == 0) wq[r] = wn;
                    }
                    // the rows' bytes are visible to the copies and to this CTA's MMAs
                    fence_proxy_async_smem();
                    asm volatile("bar.sync 4, 128;" ::: "memory");
                    if (warp == 2 && lane < kDecCl - 1 && have) {
                        const uint32_t dst = static_cast<uint32_t>(lane) + (static_cast<uint32_t>(lane) >= rank ? 1u : 0u);
                        const uint32_t bar = dsmem_addr(qready, dst);
                        uint8_t* blk = qtile + rank * 1024u;
                        bulk_copy_to_cta(dsmem_addr(blk, dst), blk, 1024u, bar);
                        if constexpr (!kFp8) bulk_copy_to_cta(dsmem_addr(blk + kN * 128, dst), blk + kN * 128, 1024u, bar);
                        bulk_copy_to_cta(dsmem_addr(wq + rank * kQRows, dst), wq + rank * kQRows, kQRows * 4u, bar);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(qready);
                // the staged rows are consumed (the histogram takes their place)
                asm volatile("bar.sync 3, %0;" ::"r"(kQuantThreads) : "memory");
                if (warp >= 4 && run) {
                    // epilogue; first the chunk histogram (where the query rows were) is cleared
                    {
                        uint4* h4 = reinterpret_cast<uint4*>(chist);
                        for (int i = tid - 128; i < 4096 / 4; i += 128) h4[i] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    // block ids in place, histogram cleared
                    asm volatile("bar.sync 2, %0;" ::"r"(32 + 32 * kEpiWarps) : "memory");
                    const int qd = warp & 3;
                    const int row = qd * 32 + head_sum_row(lane);   // the row this lane scores
                    const uint32_t lane_base = tmem + (static_cast<uint32_t>(qd * 32) << 16);
                    // every CTA's w' has arrived (the MMA waits on the same phase)
                    const bool qok = __all_sync(0xffffffffu, mbar_wait(qready, qcnt & 1u, status, &ks->abort, wlim));
                    if (tid == 128) DSAIDX_PHASE(it, 4);
                    unsigned long long wr[8];
                    load_head_weights(wq, lane, wr);
                    // key scale of this thread's key in tile t (0 past the chunk or for a bad id)
                    auto scale_of = [&](int t) -> float {
                        if constexpr (!kFp8) {
                            return 1.0f;
                        } else {
                            const int key = key_begin + t * kTileKeys + row;
                            if (t >= ntiles || key >= key_end) return 0.0f;
                            const int pb = bids[key / kBs - lb0];
                            if (pb < 0 || pb >= p.num_blocks) return 0.0f;
                            return __ldg(reinterpret_cast<const float*>(p.pool + static_cast<int64_t>(pb) * p.block_bytes +
                                                                        kBs * 128) + (key % kBs));
                        }
                    };
                    float sc0 = scale_of(0), sc1 = scale_of(1);
                    uint32_t kmax = 0u;
                    for (int t = 0; qok && t < ntiles; ++t) {
                        const uint32_t T = tcnt + static_cast<uint32_t>(t);
                        const int a = static_cast<int>(T & 1u);
                        const uint32_t aph = (T >> 1) & 1u;
                        const float kscale = sc0;
                        sc0 = sc1;
                        sc1 = scale_of(t + 2);
                        // waits are combined over the warp so that every lane leaves together
                        if (!__all_sync(0xffffffffu, mbar_wait(&tfull[a], aph, status, &ks->abort, wlim))) break;
                        tc_fence_after();
                        // every TMEM read of the buffer has completed when release runs
                        const float hs = head_sum_rows(lane_base + static_cast<uint32_t>(a * kN), wr, lane, [&] {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[a]);
                        });
                        const float res = kscale * (0.5f * hs);
                        const int i = t * kTileKeys + row;
                        if (i < nkeys) {
                            csc[i] = res;
                            const uint32_t key = score_key(res);
                            kmax = max(kmax, key);
                            const uint32_t wb = win_bin(key);
                            atomicAdd(&chist[wb >> 1], 1u << ((wb & 1u) * 16u));
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
                    if (lane == 0) ks->emax[warp - 4] = kmax;
                    if (tid == 128) DSAIDX_PHASE(it, 6);
                }
            }
            ++qcnt;
            if (run) tcnt += static_cast<uint32_t>(ntiles);
        }
        __syncthreads();
        // a wait gave up during this unit: let every copy and MMA this CTA
        // issued land before its shared memory is reused (full limit)
        if (ks->abort) {
            if (warp == 0 && lane == 0) {
                for (uint32_t T = issued > static_cast<uint32_t>(kStages) ? issued - kStages : 0u; T < issued; ++T)
                    mbar_wait(&full[T % kStages], (T / kStages) & 1u, status, nullptr);
            }
            if (warp == 1 && lane == 0) {
                mma_commit(mdone);
                mbar_wait(mdone, mcnt & 1u, status, nullptr);
            }
            ++mcnt;
            __syncthreads();
        }
        // every CTA of the cluster finished its previous unit: the receive
        // areas are free
        cluster_wait();
        if (rank == 0 && tid == 0) {
            // draw the unit after this one and send it to the cluster
            const uint32_t nx = static_cast<uint32_t>(ncl) + atomicAdd(p.ucount, 1u);
            for (uint32_t r = 0; r < static_cast<uint32_t>(kDecCl); ++r)
                dsmem_st_async_u32(dsmem_addr(&ks->unext[(it + 1) & 1u], r), nx, dsmem_addr(&ubar[(it + 1) & 1u], r));
            if (nx >= static_cast<uint32_t>(total)) {
                // this cluster is done: the last cluster to finish resets the counters
                if (atomicAdd(p.ucount + 1, 1u) == static_cast<uint32_t>(ncl - 1)) {
                    p.ucount[0] = 0u;
                    p.ucount[1] = 0u;
                }
            }
        }

        if (live) {
            const bool flagged_me = ks->bad != 0 || ks->abort != 0;
            // ------------------------------------ 1. windows to every CTA
            uint32_t* mywin = win + rank * kWinWords;
            if (tid == 0) mbar_arrive_expect_tx(wbar, (kDecCl - 1) * kWinBytes);
            {
                uint32_t hi = 0u;
#pragma unroll
                for (int w = 0; w < 4; ++w) hi = max(hi, ks->emax[w]);
                const uint32_t anchor = run ? win_bin(hi) : 0u;
                if (tid < kWinBins / 2) {
                    uint32_t word = 0u;
                    if (run) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int bn = static_cast<int>(anchor) - (kWinBins - 1) + 2 * tid + hh;
                            const uint32_t c = bn >= 0 ? (chist[bn >> 1] >> ((bn & 1) * 16)) & 0xFFFFu : 0u;
                            word |= c << (16 * hh);
                        }
                    }
                    mywin[kWinHead + tid] = word;
                }
                if (tid == 0) {
                    mywin[0] = anchor;
                    mywin[1] = run ? static_cast<uint32_t>(nkeys) : 0u;
                    mywin[2] = run ? hi : 0u;
                    mywin[3] = flagged_me ? 1u : 0u;
                }
            }
            __syncthreads();
            {
                constexpr int kPieces = kWinWords / 4;   // 16-byte pieces of a window
                for (int j = tid; j < (kDecCl - 1) * kPieces; j += kThreads) {
                    const int q = j / kPieces, c = j - q * kPieces;
                    const uint32_t dst = static_cast<uint32_t>(q) + (static_cast<uint32_t>(q) >= rank ? 1u : 0u);
                    const uint4 v = reinterpret_cast<const uint4*>(mywin)[c];
                    dsmem_st_async_v4(dsmem_addr(mywin, dst) + 16u * c, v, dsmem_addr(wbar, dst));
                }
            }
            if (tid == 0) DSAIDX_PHASE(it, 7);
            const bool wok = __syncthreads_and(mbar_wait_cluster(wbar, scnt & 1u, status, 2 * kWaitLimitNs));
            if (tid == 0) DSAIDX_PHASE(it, 8);
            ++scnt;
            // ------------------------------------ 2. boundary bin, counts, offsets
            // (the same decision in every CTA: a CTA failed a check or gave up a wait)
            int wflag = 0;
            for (int r = 0; r < kDecCl; ++r) wflag |= static_cast<int>(win[r * kWinWords + 3]);
            if (!wok) wflag = 1;
            int flag = wflag;   // this CTA's view: also set when a later wait runs out
            const int k = p.topk;
            const int n = seg_end - seg_begin;
            uint32_t gmax = 0u;
            for (int r = 0; r < kDecCl; ++r)
                if (win[r * kWinWords + 1] > 0u) gmax = max(gmax, win[r * kWinWords]);
            // thread t: bin gmax - 255 + t; its count in every CTA's window
            const int bt = static_cast<int>(gmax) - (kWinBins - 1) + tid;
            uint32_t cr[kDecCl];
            uint32_t hsum = 0u;
#pragma unroll
            for (int r = 0; r < kDecCl; ++r) {
                const uint32_t* w = win + r * kWinWords;
                const int i = bt - (static_cast<int>(w[0]) - (kWinBins - 1));
                cr[r] = (w[1] > 0u && i >= 0 && i < kWinBins) ? (w[kWinHead + (i >> 1)] >> ((i & 1) * 16)) & 0xFFFFu : 0u;
                hsum += cr[r];
            }
            uint32_t incl = hsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += y;
            }
            if (lane == 0) ks->sel.wcnt[warp] = incl;
            if (tid == 0) ks->sel.bnd.bin = -1;
            __syncthreads();
            uint32_t after = incl - hsum, wtotal = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t x = ks->sel.wcnt[q];
                after += q > warp ? x : 0u;
                wtotal += x;
            }
            const int nsel = min(k, n);   // the unit's winners
            const uint32_t kk = static_cast<uint32_t>(nsel);
            if (after < kk && kk <= after + hsum) ks->sel.bnd.bin = bt;
            __syncthreads();
            const int bstar = ks->sel.bnd.bin;
            if (tid == 0) DSAIDX_PHASE(it, 9);
            // every CTA's count of scores in bins at or above the boundary: the
            // sum over the bins from it up (a CTA with scores below its window
            // and the boundary below that window: not known, the slow path)
            {
                const bool up = bt >= bstar;
#pragma unroll
                for (int r = 0; r < kDecCl; ++r) {
                    uint32_t c = up ? cr[r] : 0u;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
                    if (lane == 0) ks->sel.scratch[warp * kDecCl + r] = c;
                }
            }
            __syncthreads();
            if (tid < kDecCl) {
                const uint32_t* w = win + tid * kWinWords;
                uint32_t c = 0u;
#pragma unroll
                for (int q = 0; q < 8; ++q) c += ks->sel.scratch[q * kDecCl + tid];
                bool known = true;
                if (w[1] > 0u && bstar >= 0 && bstar < static_cast<int>(w[0]) - (kWinBins - 1)) {
                    // boundary below this window: known only if the window holds all its scores
                    uint32_t inwin = 0u;
                    for (int i = 0; i < kWinBins / 2; ++i) {
                        const uint32_t x = w[kWinHead + i];
                        inwin += (x & 0xFFFFu) + (x >> 16);
                    }
                    known = inwin == w[1];
                }
                ks->cnt[tid] = known ? static_cast<int>(c) : -1;
            }
            __syncthreads();
            bool fast = wtotal >= kk && bstar >= 0;
            int ctot = 0;
#pragma unroll
            for (int r = 0; r < kDecCl; ++r) {
                const int c = ks->cnt[r];
                if (c < 0) fast = false;
                ctot += max(c, 0);
            }
            if (ctot > 2048 || ctot < nsel) fast = false;
            const int mycnt = max(ks->cnt[rank], 0);
            // the unit's output: the row itself (one segment) or the segment's run
            const bool single = nseg == 1;
            int32_t* oi = p.out_idx + static_cast<int64_t>(b) * k;
            float* os = p.out_score ? p.out_score + static_cast<int64_t>(b) * k : nullptr;
            int64_t* osl = p.out_slot ? p.out_slot + static_cast<int64_t>(b) * k : nullptr;
            const int32_t* btr = p.block_table + static_cast<int64_t>(b) * p.mbps;
            uint64_t* run_out = single ? nullptr : p.cand + static_cast<int64_t>(b) * p.cand_cap + static_cast<int64_t>(seg) * k;
            uint32_t* gh = single ? nullptr : p.ghist + static_cast<int64_t>(b) * kGHistWords;
            // (runs: the fast path adds the run's bin counts from its tables after
            // the ranks, one atomic per bin; the slow path one per winner)
            auto emit = [&](int r, uint64_t c) {
                if (single) {
                    oi[r] = comp_index(c);
                    if (os) os[r] = key_score(comp_key(c));
                    if (osl) osl[r] = slot_of(btr, p.mbps, kBs, comp_index(c));
                } else {
                    run_out[r] = c;
                    if (!fast) {
                        const uint32_t wb = win_bin(comp_key(c));
                        atomicAdd(gh + wb, 1u);
                        if (r == 0) atomicMax(gh + kGHistBins, wb + 1u);   // the sequence's largest bin (+1)
                    }
                }
            };
            if (flag) {
                // a block id failed its check or a wait gave up: no selection
            } else if (fast) {
                // ------------------------------------ 3. the pool: the candidates
                // (bins at or above the boundary) bin by bin from the top, within
                // a bin CTA by CTA, the same layout in every CTA; CTA r ranks the
                // places [r ctot / 8, (r + 1) ctot / 8) and reads only the bins
                // that reach them, so each CTA writes a candidate to the pools of
                // the CTAs whose places its bin reaches (mostly one), so no CTA
                // sorts anything
                const int wlo = static_cast<int>(gmax) - (kWinBins - 1);   // bin of thread 0
                uint32_t* bstart = reinterpret_cast<uint32_t*>(a_tiles);     // [kWinBins] first place of a bin
                uint32_t* blen = bstart + kWinBins;                          // [kWinBins] its entries
                uint32_t* bfill = blen + kWinBins;                           // [kWinBins] this CTA's next place
                // [kWinBins] CTAs whose places a bin reaches (bit mask), after the
                // ranking's scratch (sub-bin counts, cursors, a crowded bin, list)
                uint32_t* bdst = bfill + 4 * kWinBins + 2 * 2048 + kWinBins;
                {
                    uint32_t before = 0u, mine = 0u;
#pragma unroll
                    for (int r = 0; r < kDecCl; ++r) {
                        before += r < static_cast<int>(rank) ? cr[r] : 0u;
                        mine = r == static_cast<int>(rank) ? cr[r] : mine;
                    }
                    bstart[tid] = after;
                    blen[tid] = hsum;
                    bfill[tid] = after + before;
                    // owner of place x: the last r with r ctot / 8 <= x, (8 x + 7) / ctot
                    uint32_t dm = 0u, recv = 0u;
                    if (bt >= bstar && hsum > 0u) {
                        const uint32_t ct = static_cast<uint32_t>(ctot);
                        const uint32_t rf = (8u * after + 7u) / ct, rl = (8u * (after + hsum) - 1u) / ct;
                        dm = ((2u << rl) - 1u) & ~((1u << rf) - 1u);
                        if ((dm >> rank) & 1u) recv = hsum - mine;   // what the other CTAs send here
                    }
                    bdst[tid] = dm;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) recv += __shfl_xor_sync(0xffffffffu, recv, o);
                    if (lane == 0) ks->sel.scratch[warp] = recv;
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t e = 0u;
#pragma unroll
                    for (int q = 0; q < 8; ++q) e += ks->sel.scratch[q];
                    mbar_arrive_expect_tx(lbar, e * 8u);
                }
                {
                    // this CTA's candidates are first gathered into a list
                    // (count per thread, scan, write: no atomics), then placed
                    // one per thread, so that the atomic on a bin's next place
                    // is not a dependent step of every candidate in turn
                    const uint32_t kthr = static_cast<uint32_t>(bstar) << kWinShift;   // smallest key of the boundary bin
                    const float4* s4 = reinterpret_cast<const float4*>(csc);
                    const int nj = (nkeys + 3) >> 2;
                    auto is_cand = [&](float v, int i) { return i < nkeys && score_key(v) >= kthr; };
                    uint32_t mc = 0u;
                    for (int j = tid; j < nj; j += kThreads) {
                        const float4 x = s4[j];
                        mc += (is_cand(x.x, 4 * j) ? 1u : 0u) + (is_cand(x.y, 4 * j + 1) ? 1u : 0u) +
                              (is_cand(x.z, 4 * j + 2) ? 1u : 0u) + (is_cand(x.w, 4 * j + 3) ? 1u : 0u);
                    }
                    uint32_t incl = mc;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    if (lane == 31) ks->sel.scratch[8 + warp] = incl;
                    __syncthreads();
                    uint32_t at = incl - mc, nlist = 0u;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t x = ks->sel.scratch[8 + q];
                        at += q < warp ? x : 0u;
                        nlist += x;
                    }
                    // the list lives where the ranking's crowded-bin buffer goes later
                    uint64_t* lst = reinterpret_cast<uint64_t*>(bfill + 3 * kWinBins);
                    auto put = [&](float v, int i) {
                        if (is_cand(v, i)) lst[at++] = make_comp(score_key(v), key_begin + i);
                    };
                    for (int j = tid; j < nj; j += kThreads) {
                        const float4 x = s4[j];
                        put(x.x, 4 * j);
                        put(x.y, 4 * j + 1);
                        put(x.z, 4 * j + 2);
                        put(x.w, 4 * j + 3);
                    }
                    __syncthreads();
                    for (int q = tid; q < static_cast<int>(nlist); q += kThreads) {
                        const uint64_t c = lst[q];
                        const int t = static_cast<int>(win_bin(comp_key(c))) - wlo;
                        const uint32_t slot = atomicAdd(&bfill[t], 1u);
                        uint32_t dm = bdst[t];
                        if ((dm >> rank) & 1u) pool[slot] = c;
                        dm &= ~(1u << rank);
                        while (dm != 0u) {
                            const uint32_t dst = static_cast<uint32_t>(__ffs(dm) - 1);
                            dm &= dm - 1u;
                            dsmem_st_async_u64(dsmem_addr(pool + slot, dst), c, dsmem_addr(lbar, dst));
                        }
                    }
                }
                const bool lok = __syncthreads_and(mbar_wait_cluster(lbar, lcnt & 1u, status, 2 * kWaitLimitNs));
                if (tid == 0) DSAIDX_PHASE(it, 10);
                ++lcnt;
                if (lok) {
                    // ------------------------------------ 4. this CTA's eighth of the
                    // pool: rank = the entries of higher bins plus the larger entries
                    // of its own bin
                    const int lo = static_cast<int>(rank) * ctot / kDecCl;
                    const int hi = (static_cast<int>(rank) + 1) * ctot / kDecCl;
                    {
                        uint32_t* scnt = bfill + kWinBins;                             // [256] sub-bin counts
                        uint32_t* scur = scnt + 256;                                   // [256] sub-bin cursors
                        uint64_t* srt = reinterpret_cast<uint64_t*>(scur + 256);      // [2048] a crowded bin, by sub-bin
                        uint32_t* clist = reinterpret_cast<uint32_t*>(srt + 2048);     // [256] crowded bins
                        rank_pool(pool, lo, hi, nsel, bstar - wlo, wlo, bstart, blen, scnt, scur, clist, srt,
                                  &ks->nmine, ks->sel.wcnt, emit);
                    }
                    if (tid == 0) DSAIDX_PHASE(it, 11);
                    if (!single && rank == lead) {
                        // the run's entries per bin: every entry of a bin above the
                        // boundary, the boundary bin's first nsel - start
                        for (int t = bstar - wlo + tid; t < kWinBins; t += kThreads) {
                            const int start = static_cast<int>(bstart[t]);
                            const int c = t == bstar - wlo ? nsel - start : static_cast<int>(blen[t]);
                            if (c > 0) atomicAdd(gh + wlo + t, static_cast<uint32_t>(c));
                        }
                        if (tid == 0) atomicMax(gh + kGHistBins, static_cast<uint32_t>(gmax) + 1u);
                    }
                } else {
                    flag = 1;   // (a wait that ran out: the status word says so)
                }
            } else {
                // ------------------------------------ slow path: one CTA selects from
                // the chunks' scores in the cluster's global scratch
                float* gsc = p.scratch + static_cast<int64_t>(cl) * kDecCl * p.chunk;
                for (int i = tid; i < nkeys; i += kThreads) gsc[key_begin - seg_begin + i] = csc[i];
                __threadfence();
                __syncthreads();
                if (tid == 0) {
                    fence_acq_rel_cluster();
                    mbar_arrive_remote(dsmem_addr(rbar, lead));
                }
                if (rank == lead) {
                    const bool ok = __syncthreads_and(mbar_wait_cluster(rbar, rcnt & 1u, status, 2 * kWaitLimitNs));
                    ++rcnt;
                    __threadfence();
                    if (ok) {
                        const int nout = seg_select(GScoreSet{gsc, n, seg_begin}, k, shist, sbuf, &ks->sel);
                        for (int j = tid; j < nout; j += kThreads) emit(j, sbuf[j]);
                    } else {
                        flag = 1;
                    }
                }
            }
            // ------------------------------------ the unit's results are written
            if (single) {
                if (rank == lead) {
                    // -1 past the winners (a flagged row: all of it)
                    for (int j = (flag ? 0 : nsel) + tid; j < k; j += kThreads) {
                        oi[j] = -1;
                        if (os) os[j] = -INFINITY;
                        if (osl) osl[j] = -1;
                    }
                }
            } else {
                if (flag && tid == 0) atomicOr(p.seqflag + b, 1u);
                if (fast || wflag) {
                    // every CTA's part of the run is written before the ticket
                    __threadfence();
                    __syncthreads();
                    if (tid == 0) {
                        fence_acq_rel_cluster();
                        mbar_arrive_remote(dsmem_addr(rbar, lead));
                    }
                    if (rank == lead) {
                        mbar_wait_cluster(rbar, rcnt & 1u, status, 2 * kWaitLimitNs);
                        ++rcnt;
                    }
                }
                if (rank == lead) {
                    // zero-pad the run past its winners
                    if (!flag)
                        for (int j = nsel + tid; j < k; j += kThreads) run_out[j] = 0ull;
                    __threadfence();
                    __syncthreads();
                    if (tid == 0) ks->last = (atomicAdd(p.ctr + b, 1u) == static_cast<uint32_t>(nseg - 1)) ? 1u : 0u;
                    __syncthreads();
                    if (ks->last) {
                        // ------------------------------------ sequence merge
                        __threadfence();
                        // (-1: a segment failed a device check; merge_runs also
                        // leaves the histogram zeroed)
                        const int mout = merge_runs(p.cand + static_cast<int64_t>(b) * p.cand_cap, nseg, k, gh,
                                                    p.seqflag + b, shist, reinterpret_cast<uint32_t*>(pool), sbuf,
                                                    &ks->sel);
                        write_topk_row(sbuf, mout, k, oi, os, osl, btr, p.mbps, kBs);
                        // leave the rest of the sequence's workspace zeroed for the next call
                        if (tid == 0) {
                            p.ctr[b] = 0u;
                            p.seqflag[b] = 0u;
                        }
                    }
                }
            }
        } else if (rank == lead) {
            // an empty sequence, or one whose length is out of range: a -1 row
            if (!valid && tid == 0) set_status(status, IDX_ERR_DEVICE_CHECK);
            write_topk_row(sbuf, -1, p.topk, p.out_idx + static_cast<int64_t>(b) * p.topk,
                           p.out_score ? p.out_score + static_cast<int64_t>(b) * p.topk : nullptr,
                           p.out_slot ? p.out_slot + static_cast<int64_t>(b) * p.topk : nullptr);
        }
        // generic accesses of the stages come before the next unit's copies
        // into them; this CTA is done with its receive areas.  The arrive is
        // relaxed: the barrier only has to keep the peers' next writes into
        // the receive areas behind this CTA's reads of them, and every such
        // read has returned its value before the block barrier above (the
        // values were consumed: ranks, emitted outputs), so no memory ordering
        // is needed and the arrive need not wait for the outputs' global
        // stores to complete
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) DSAIDX_PHASE(it, 12);
        cluster_arrive_relaxed();
        // the next unit (drawn by rank 0 during this one); slot (it + 1) & 1 is
        // used every other unit, so this is its (it >> 1)-th use
        const bool uok =
            __syncthreads_and(mbar_wait_cluster(&ubar[(it + 1) & 1u], (it >> 1) & 1u, status, 2 * kWaitLimitNs));
        u = uok ? static_cast<int>(ks->unext[(it + 1) & 1u]) : total;
        __syncthreads();
    }

    if (tid == 0) DSAIDX_PHASE(0, 13);
    // no CTA leaves while another may still send it something
    cluster_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 2 * kN);
    if (tid == 32) DSAIDX_PHASE(0, 14);
}

}  // namespace dsaidx
