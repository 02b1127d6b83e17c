// cluster_select.cuh -- exact top-k of one decode segment, computed by the 8
// CTAs of a thread-block cluster together, with no leader CTA.
//
// The selection rule is the one of the indexer ("The Hypothesis That Refused
// to Die", section "The Context": the k best-scoring cached positions); ties
// go to the lower index.  Candidates are 64-bit composites
// (score_key << 32) | ~index, so "larger composite" is exactly that order.
//
// Every CTA holds the composites of its own chunk of keys and a 4096-bin
// histogram of their top 12 bits.  A remote shared-memory load costs a round
// trip of ~0.3 us on GB300 and a cluster barrier more, so data moves by
// one-way pushes (st.async, counted on the receiver's mbarrier):
//   1. every CTA sums one 512-bin slice of the histogram over the cluster --
//      with a receive area (small chunks), every CTA pushes each owner its
//      slice at the end of its key loop; otherwise after one cluster barrier
//      each CTA pulls its slice from every CTA (eight remote 8-byte loads per
//      thread) -- and pushes the sum, with its device-check flag, to every
//      CTA: each CTA then holds the cluster's histogram and finds the bin of
//      the k-th largest composite by itself;
//      when the bins at or above it hold more than kClCap composites (a wide
//      boundary bin, or ties), 256-bin histograms of the next 8 bits of the
//      boundary group, pushed the same way, refine the threshold a level at a
//      time;
//   2. every CTA collects its candidates (composites >= the threshold),
//      pushes their number to every CTA, sorts them, and pushes the sorted
//      list to every CTA;
//   3. every CTA ranks each of its candidates by binary searches in the other
//      CTAs' lists; rank r < k goes to output position r.
// Every push into a CTA is awaited by that CTA, and every remote load of a
// CTA's histogram happens before the loader's first push of the summed
// slice, so no CTA leaves while another still reads or writes its shared
// memory.  The pushes of step 1 land in areas a CTA does not use during its
// key loop (the receive area) or after every CTA has left it (the rest).
#pragma once

#include "common.cuh"
#include "topk.cuh"

namespace dsaidx {

constexpr int kCl = 8;                          // CTAs per cluster
constexpr int kClCap = 2048;                    // candidates one cluster ranks
constexpr int kClSliceBins = kHistBins / kCl;   // histogram bins each CTA sums
constexpr int kClLevels = 7;                    // refinement levels (8,8,8,8,8,8,4 bits)
constexpr int kClBarHist = 0;                   // every CTA's histogram is complete (kCl arrivals)
constexpr int kClBarFull = 1;                   // the summed histogram and the flags have arrived
constexpr int kClBarRefine0 = 2;                // level l's sub-histograms have arrived: 2 + l
constexpr int kClBarCount = kClBarRefine0 + kClLevels;   // every CTA's candidate count has arrived
constexpr int kClBarList = kClBarCount + 1;     // every CTA's sorted candidates have arrived
constexpr int kClBarRecv = kClBarList + 1;      // every CTA's slice of this CTA's bins has arrived
constexpr int kClBars = kClBarRecv + 1;
constexpr int kCountSortMax = 96;   // longest candidate list sorted by counting
constexpr uint32_t kClFullBytes = kHistBins * 4 + kCl * 4;
constexpr uint32_t kClSubBytes = kCl * 256 * 4;
constexpr uint32_t kClCountBytes = kCl * 4;
constexpr uint32_t kClRecvBytes = kCl * kClSliceBins * 4;
static_assert(kClCap >= IDX_MAX_TOPK, "a cluster must be able to rank k candidates");
static_assert(kClSliceBins == 2 * 256, "each of 256 threads sums two bins");

struct ClusterSmem {
    uint32_t flag[kCl];        // [r]: CTA r failed a device check or gave up a wait (pushed by r)
    uint32_t lcnt[kCl];        // [r]: number of CTA r's candidates (pushed by r)
    uint32_t wsum[8];          // block-reduction scratch
    Boundary bnd;              // result of block_suffix_find_reg
    uint32_t nloc;             // this CTA's candidates
    int dead;                  // a wait of the selection timed out
};

// Shared-memory buffers of the selection (the same offsets in every CTA).
// full/list and sub/gath may share memory: each pair's uses are ordered by the
// pushes (a CTA writes its list only after reading the full histogram, and
// receives lists only after it has pushed its count, i.e. after its last
// refinement level).
struct ClusterBufs {
    uint32_t* hist;   // [4096] histogram of this CTA's composites' top 12 bits
    uint32_t* mine;   // [256] this CTA's refinement histogram
    uint32_t* full;   // [4096] the cluster's histogram (received)
    uint32_t* sub;    // [2][kCl][256] refinement histograms (received)
    uint64_t* list;   // [kClCap] this CTA's candidates, sorted descending
    uint64_t* gath;   // [kClCap] every CTA's sorted list, in rank order (received)
    uint64_t* runs;   // [kClCap] sort scratch
    uint64_t* cbar;   // [kClBars] barriers of the selection
    uint32_t* recv;   // [kCl][512] every CTA's slice of this CTA's bins (received), or null
};

// Barrier set-up, by one thread before the cluster's first barrier: the
// histogram barrier takes one arrive per CTA; the others complete when their
// bytes have arrived (the list barrier's byte count is set once the counts
// are known).
__device__ __forceinline__ void cluster_select_init(uint64_t* cbar) {
    mbar_init(&cbar[kClBarHist], kCl);
    for (int i = kClBarFull; i < kClBars; ++i) mbar_init(&cbar[i], 1);
}
__device__ __forceinline__ void cluster_select_expect(uint64_t* cbar) {
    mbar_arrive_expect_tx(&cbar[kClBarFull], kClFullBytes);
    for (int l = 0; l < kClLevels; ++l) mbar_arrive_expect_tx(&cbar[kClBarRefine0 + l], kClSubBytes);
    mbar_arrive_expect_tx(&cbar[kClBarCount], kClCountBytes);
    mbar_arrive_expect_tx(&cbar[kClBarRecv], kClRecvBytes);
}

__device__ __forceinline__ bool cl_wait(uint64_t* bar, int32_t* status, ClusterSmem* cs) {
    if (*reinterpret_cast<volatile int*>(&cs->dead)) return false;
    const bool ok = mbar_wait_cluster(bar, 0, status);
    if (!ok) *reinterpret_cast<volatile int*>(&cs->dead) = 1;
    return ok;
}

// Thread t holds the counts of bins t*PER .. t*PER+PER-1 (higher bin = larger
// composites).  Finds the bin holding the need-th largest counted element:
// out->bin (-1 when fewer than need were counted), out->above (elements in
// higher bins; the total when bin = -1), out->at (the bin's count).  All 256
// threads; the result is valid for all of them after the call.
template <int PER>
__device__ __forceinline__ void block_suffix_find_reg(const uint32_t (&v)[PER], uint32_t need, uint32_t* wsum,
                                                      Boundary* out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t s = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) s += v[j];
    uint32_t incl = s;   // over this warp's lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
    }
    if (lane == 0) wsum[warp] = incl;
    __syncthreads();
    uint32_t total = 0, higher = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t x = wsum[q];
        total += x;
        if (q > warp) higher += x;
    }
    const uint32_t after = higher + incl - s;   // elements in bins above this thread's
    if (total < need) {
        if (tid == 0) {
            out->bin = -1;
            out->above = total;
            out->at = 0;
        }
    } else if (after < need && need <= after + s) {
        uint32_t acc = after;
#pragma unroll
        for (int j = PER - 1; j >= 0; --j) {
            if (acc + v[j] >= need) {
                out->bin = tid * PER + j;
                out->above = acc;
                out->at = v[j];
                break;
            }
            acc += v[j];
        }
    }
    __syncthreads();
}

// The cluster's exact top-k.  walk(f) calls f(composite, valid) over this
// CTA's composites (valid ones are never 0) with warp-uniform trip counts;
// collect0(kthr, dst, cap, seg, wsum) collects the composites whose score key
// is >= kthr into dst the way block_collect_warp does (seg: scratch) and
// returns their number -- a faster first pass than walk where the caller can
// test the 32-bit key alone;
// B.hist must hold their top-12-bit histogram.  emit(r, c) receives every
// candidate c of this CTA whose rank r among the cluster's composites is
// below k (each rank in [0, min(k, count)) exactly once over the cluster).
// Returns the number of ranked candidates (count >= k unless the cluster
// holds fewer than k composites), or -1 when a CTA of the cluster reported
// `flagged` (every CTA returns -1 then) or a wait timed out.  Called by all
// 256 threads of every CTA of the cluster.
template <class Walk, class Collect0, class Emit>
__device__ int cluster_select(Walk walk, Collect0 collect0, Emit emit, const ClusterBufs& B, int k, bool flagged,
                              ClusterSmem* cs, int32_t* status) {
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_rank();

    // (1) the cluster's histogram, summed slice by slice: CTA r sums bins
    //     [512 r, 512 r + 512) and pushes the sum, with its flag, to every CTA
    uint32_t a0 = 0, a1 = 0;
    const uint32_t soff = (static_cast<uint32_t>(kClSliceBins) * rank + 2u * static_cast<uint32_t>(tid)) * 4u;
    if (B.recv) {
        // one-way: every CTA pushes each owner its slice of that owner's bins
        // as soon as its own histogram is complete (the receive area is not
        // used before); the owner waits for all eight and adds them up
        __syncthreads();
        for (int c = tid; c < kCl * (kClSliceBins / 4); c += kTopkThreads) {
            const uint32_t q = static_cast<uint32_t>(c / (kClSliceBins / 4));
            const int j = c - static_cast<int>(q) * (kClSliceBins / 4);
            const uint4 v = reinterpret_cast<const uint4*>(B.hist + q * kClSliceBins)[j];
            dsmem_st_async_v4(dsmem_addr(B.recv + rank * kClSliceBins + 4 * j, q), v,
                              dsmem_addr(&B.cbar[kClBarRecv], q));
        }
        if (!cl_wait(&B.cbar[kClBarRecv], status, cs)) return -1;
#pragma unroll
        for (int q = 0; q < kCl; ++q) {
            const uint2 h = reinterpret_cast<const uint2*>(B.recv + q * kClSliceBins)[tid];
            a0 += h.x;
            a1 += h.y;
        }
    } else {
        // every CTA's histogram is complete (and its key stage buffers are
        // free): one barrier, then each CTA pulls its bins from every CTA
        __syncthreads();
        if (tid < kCl) {
            fence_acq_rel_cluster();
            mbar_arrive_remote(dsmem_addr(&B.cbar[kClBarHist], static_cast<uint32_t>(tid)));
        }
        if (!cl_wait(&B.cbar[kClBarHist], status, cs)) return -1;
        uint2 h[kCl];
#pragma unroll
        for (int q = 0; q < kCl; ++q) h[q] = dsmem_ld_v2(dsmem_addr(B.hist, q) + soff);
#pragma unroll
        for (int q = 0; q < kCl; ++q) {
            a0 += h[q].x;
            a1 += h[q].y;
        }
    }
#pragma unroll
    for (int q = 0; q < kCl; ++q)
        dsmem_st_async_v2(dsmem_addr(B.full, q) + soff, a0, a1, dsmem_addr(&B.cbar[kClBarFull], q));
    if (tid < kCl)
        dsmem_st_async_u32(dsmem_addr(&cs->flag[rank], static_cast<uint32_t>(tid)), flagged ? 1u : 0u,
                           dsmem_addr(&B.cbar[kClBarFull], static_cast<uint32_t>(tid)));
    if (!cl_wait(&B.cbar[kClBarFull], status, cs)) return -1;
    uint32_t anyflag = 0;
#pragma unroll
    for (int q = 0; q < kCl; ++q) anyflag |= cs->flag[q];
    if (anyflag) return -1;   // the same decision in every CTA

    // the bin of the k-th largest composite (16 bins per thread)
    uint32_t above, at;
    int bstar;
    {
        uint32_t v[16];
        const uint4* f4 = reinterpret_cast<const uint4*>(B.full) + 4 * tid;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = f4[j];
            v[4 * j] = x.x;
            v[4 * j + 1] = x.y;
            v[4 * j + 2] = x.z;
            v[4 * j + 3] = x.w;
        }
        block_suffix_find_reg<16>(v, static_cast<uint32_t>(k), cs->wsum, &cs->bnd);
        bstar = cs->bnd.bin;
        above = cs->bnd.above;   // the total when bstar = -1: every composite is a candidate
        at = cs->bnd.at;
    }
    // candidates: composites >= thr, `count` of them in the cluster
    uint64_t thr = bstar >= 0 ? (static_cast<uint64_t>(bstar) << 52) : 0ull;
    uint64_t mask = 0xFFFull << 52;
    uint32_t need = static_cast<uint32_t>(k) - min(above, static_cast<uint32_t>(k));
    uint32_t count = above + at;
    // this CTA's composites >= thr, collected once: when they fit, the
    // refinement levels and the final filter read this list instead of
    // walking every composite again
    // (thr has zero low 52 bits here: the key alone decides)
    const uint32_t n0 = collect0(bstar >= 0 ? static_cast<uint32_t>(bstar) << 20 : 0u, B.list,
                                 static_cast<uint32_t>(kClCap), B.runs, cs->wsum);
    const bool pre = n0 <= static_cast<uint32_t>(kClCap);
    auto cands = [&](auto f) {
        if (pre) walk_smem(B.list, n0, f);
        else walk(f);
    };
    const uint64_t thr0 = thr;
#pragma unroll 1
    for (int lvl = 0; count > static_cast<uint32_t>(kClCap) && lvl < kClLevels; ++lvl) {
        // refine: histogram of the next digit over the boundary group
        const int sh = lvl < 6 ? 44 - 8 * lvl : 0;
        const uint64_t dmask = lvl < 6 ? 0xFFull : 0xFull;
        B.mine[tid] = 0;
        __syncthreads();
        cands([&](uint64_t c, bool v) {
            hist_add_warp(B.mine, static_cast<uint32_t>((c >> sh) & dmask), v && (c & mask) == thr);
        });
        __syncthreads();
        const uint32_t val = B.mine[tid];
        uint32_t* slot = B.sub + ((lvl & 1) * kCl + static_cast<int>(rank)) * 256 + tid;
#pragma unroll
        for (int q = 0; q < kCl; ++q)
            dsmem_st_async_u32(dsmem_addr(slot, q), val, dsmem_addr(&B.cbar[kClBarRefine0 + lvl], q));
        if (!cl_wait(&B.cbar[kClBarRefine0 + lvl], status, cs)) return -1;
        uint32_t v[1] = {0};
#pragma unroll
        for (int q = 0; q < kCl; ++q) v[0] += B.sub[((lvl & 1) * kCl + q) * 256 + tid];
        block_suffix_find_reg<1>(v, need, cs->wsum, &cs->bnd);
        const int d = max(cs->bnd.bin, 0);   // >= 0: the group holds at least `need`
        above += cs->bnd.above;
        need -= min(need, cs->bnd.above);
        thr |= static_cast<uint64_t>(d) << sh;
        mask |= dmask << sh;
        count = above + cs->bnd.at;
    }

    // (2) this CTA's candidates: their number to every CTA, then sorted, then
    //     the list to every CTA
    uint64_t* mylist = B.list;   // sorted in place, then pushed and ranked
    uint64_t* scratch = B.runs;
    uint32_t nfound = n0;
    if (!(pre && thr == thr0)) {
        // refined (or the first collection overflowed): collect again
        mylist = pre ? B.runs : B.list;
        scratch = pre ? B.list : B.runs;
        // segment scratch: gath receives nothing before this CTA pushes its count
        nfound = block_collect_warp(cands, [&](uint64_t c) { return c >= thr; }, mylist, kClCap,
                                    pre ? B.gath : B.runs, cs->wsum);
    }
    const int nr = min(static_cast<int>(nfound), kClCap);
    if (tid < kCl)
        dsmem_st_async_u32(dsmem_addr(&cs->lcnt[rank], static_cast<uint32_t>(tid)), static_cast<uint32_t>(nr),
                           dsmem_addr(&B.cbar[kClBarCount], static_cast<uint32_t>(tid)));
    if (nr <= kCountSortMax) {
        // short list: sort by counting into the scratch buffer, which then
        // holds the list (its cost grows with the square of the length: the
        // warp-run sort is faster above about a hundred entries)
        block_count_sort(mylist, nr, scratch);
        uint64_t* t = mylist;
        mylist = scratch;
        scratch = t;
    } else {
        block_sort_any(mylist, nr, scratch);
    }
    if (!cl_wait(&B.cbar[kClBarCount], status, cs)) return -1;
    int off[kCl + 1];
    off[0] = 0;
#pragma unroll
    for (int q = 0; q < kCl; ++q) off[q + 1] = min(off[q] + min(static_cast<int>(cs->lcnt[q]), kClCap), kClCap);
    const int all = off[kCl];
    if (tid == 0) mbar_arrive_expect_tx(&B.cbar[kClBarList], static_cast<uint32_t>(all) * 8u);
    {
        int mine_off = 0, mine_n = 0;
#pragma unroll
        for (int q = 0; q < kCl; ++q) {
            if (q == static_cast<int>(rank)) {
                mine_off = off[q];
                mine_n = off[q + 1] - off[q];
            }
        }
#pragma unroll 1
        for (int j = tid; j < mine_n * kCl; j += kTopkThreads) {
            const int e = j / kCl;
            const uint32_t q = static_cast<uint32_t>(j % kCl);
            dsmem_st_async_u64(dsmem_addr(B.gath + mine_off + e, q), mylist[e], dsmem_addr(&B.cbar[kClBarList], q));
        }
    }
    if (!cl_wait(&B.cbar[kClBarList], status, cs)) return -1;

    // (3) rank = own position + larger members of the other lists
    int maxlen = 0;
#pragma unroll
    for (int q = 0; q < kCl; ++q) maxlen = max(maxlen, off[q + 1] - off[q]);
    const int iters = 32 - __clz(maxlen);   // binary-search steps for the longest list
#pragma unroll 1
    for (int i = tid; i < nr; i += kTopkThreads) {
        const uint64_t x = mylist[i];
        int lo[kCl], len[kCl];
#pragma unroll
        for (int q = 0; q < kCl; ++q) {
            lo[q] = off[q];
            len[q] = (q == static_cast<int>(rank)) ? 0 : off[q + 1] - off[q];
        }
#pragma unroll 1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int q = 0; q < kCl; ++q) {
                const int half = len[q] >> 1;
                const int idx = lo[q] + half;
                const uint64_t y = B.gath[min(idx, kClCap - 1)];   // unconditional: no branch
                const bool gt = (len[q] > 0) & (y > x);
                lo[q] = gt ? idx + 1 : lo[q];
                len[q] = gt ? len[q] - half - 1 : half;
            }
        }
        int r = i;   // larger members of this CTA's own list
#pragma unroll
        for (int q = 0; q < kCl; ++q)
            if (q != static_cast<int>(rank)) r += lo[q] - off[q];
        if (r < k) emit(r, x);
    }
    return static_cast<int>(count);
}

}  // namespace dsaidx
