// segsel.cuh -- exact top-k building blocks of the decode selection, by one
// 256-thread CTA, written for latency: every pass over scores reads four per
// 16-byte load with several loads in flight.
//
// The rule is the indexer's ("The Hypothesis That Refused to Die", section
// "The Context": the k best-scoring positions), ties to the lower index.
// Candidates are 64-bit composites (score key << 32) | ~index, so a larger
// composite is a better candidate (common.cuh, topk.cuh).
//
// seg_select (a segment's scores in global scratch, the crowded case):
//  1. key range: the smallest and largest score key of the segment;
//  2. histogram: 4096 bins of the keys mapped onto the full 32 bits by
//     (key - lo) << z (order-preserving; iid scores fill about one octave of
//     the float format, where the plain top 12 bits would give a few bins);
//  3. boundary: the bin holding the k-th largest mapped key;
//  4. collect: every composite in a bin at or above the boundary (k plus the
//     boundary bin's few extra entries) into a buffer, warp-aggregated;
//  5. when the collected set is much larger than k (many equal or near-equal
//     scores), refine the boundary bin by 8-bit digits of the composite;
//  6. sort the collected composites and map the winners' keys back.
// bin_order: a sorted order of at most 2048 composites by mapped bins and
// ranks inside a bin.  merge_runs: the top-k of a long sequence from its
// segments' sorted runs.
#pragma once

#include "common.cuh"
#include "topk.cuh"

namespace dsaidx {

struct SegSelSmem {
    uint32_t red[16];
    uint32_t wcnt[8];
    Boundary bnd;
    uint32_t scratch[256];
};

// Calls f(key, index, valid) for the n scores s[0, n) (16-byte aligned,
// readable up to n rounded up to 4), index = base + position, with four loads
// in flight per thread and warp-uniform trip counts.
template <class F>
__device__ __forceinline__ void seg_walk(const float* s, int n, int base, F f) {
    const float4* s4 = reinterpret_cast<const float4*>(s);
    const int nj = (n + 3) >> 2;
    constexpr int U = 4;
    for (int j0 = 0; j0 < nj; j0 += kTopkThreads * U) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * kTopkThreads + static_cast<int>(threadIdx.x);
            x[u] = j < nj ? s4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = 4 * (j0 + u * kTopkThreads + static_cast<int>(threadIdx.x));
            f(score_key(x[u].x), base + i, i < n);
            f(score_key(x[u].y), base + i + 1, i + 1 < n);
            f(score_key(x[u].z), base + i + 2, i + 2 < n);
            f(score_key(x[u].w), base + i + 3, i + 3 < n);
        }
    }
}

// Calls f(key, index, valid) for the n composites c[0, n) (16-byte aligned,
// readable up to n rounded up to 2), two per load, four loads in flight.
template <class F>
__device__ __forceinline__ void comp_walk(const uint64_t* c, int n, F f) {
    const uint4* c4 = reinterpret_cast<const uint4*>(c);
    const int nj = (n + 1) >> 1;
    constexpr int U = 4;
    for (int j0 = 0; j0 < nj; j0 += kTopkThreads * U) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * kTopkThreads + static_cast<int>(threadIdx.x);
            x[u] = j < nj ? c4[j] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = 2 * (j0 + u * kTopkThreads + static_cast<int>(threadIdx.x));
            f(x[u].y, static_cast<int32_t>(~x[u].x), i < n);
            f(x[u].w, static_cast<int32_t>(~x[u].z), i + 1 < n);
        }
    }
}

// A segment of n scores in shared memory (key indices base + position).
struct ScoreSet {
    const float* s;
    int n, base;
    template <class F>
    __device__ __forceinline__ void operator()(F f) const { seg_walk(s, n, base, f); }
};
// A segment of n scores in global memory written by other CTAs (read through
// L2, not L1).  Like every walk here, the trip count is the same in all lanes
// of a warp (callers may vote inside f).
struct GScoreSet {
    const float* s;
    int n, base;
    template <class F>
    __device__ __forceinline__ void operator()(F f) const {
        const float4* s4 = reinterpret_cast<const float4*>(s);
        const int nj = (n + 3) >> 2;
        for (int j0 = 0; j0 < nj; j0 += kTopkThreads) {
            const int j = j0 + static_cast<int>(threadIdx.x);
            const float4 x = j < nj ? __ldcg(s4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            const int i = 4 * j;
            f(score_key(x.x), base + i, i < n);
            f(score_key(x.y), base + i + 1, i + 1 < n);
            f(score_key(x.z), base + i + 2, i + 2 < n);
            f(score_key(x.w), base + i + 3, i + 3 < n);
        }
    }
};
// A set of n composites in global memory (read through L2).
struct GCompSet {
    const uint64_t* c;
    int n;
    template <class F>
    __device__ __forceinline__ void operator()(F f) const {
        const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(c);
        const int nj = (n + 1) >> 1;
        for (int j0 = 0; j0 < nj; j0 += kTopkThreads) {
            const int j = j0 + static_cast<int>(threadIdx.x);
            ulonglong2 x;
            x.x = 0ull;
            x.y = 0ull;
            if (j < nj) x = __ldcg(c2 + j);
            const int i = 2 * j;
            f(static_cast<uint32_t>(x.x >> 32), comp_index(x.x), i < n && x.x != 0ull);
            f(static_cast<uint32_t>(x.y >> 32), comp_index(x.y), i + 1 < n && x.y != 0ull);
        }
    }
};
// A set of n composites in shared memory.
struct CompSet {
    const uint64_t* c;
    int n;
    template <class F>
    __device__ __forceinline__ void operator()(F f) const { comp_walk(c, n, f); }
};

// The exact top-k of a set (ScoreSet or CompSet, `walk`) into buf[0, nout)
// sorted descending as composites of the ORIGINAL score keys; returns nout =
// min(k, set size).  hist: 4096 words; buf: >= 4096 composites (collection
// and sort scratch, disjoint from the set).  All 256 threads.
template <class Set>
__device__ __noinline__ int seg_select(const Set walk, int k, uint32_t* hist, uint64_t* buf, SegSelSmem* sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // 1. key range
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int i = tid; i < kHistBins; i += kTopkThreads) hist[i] = 0u;
    walk([&](uint32_t key, int, bool v) {
        lo = v ? min(lo, key) : lo;
        hi = v ? max(hi, key) : hi;
    });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        sm->red[warp] = lo;
        sm->red[8 + warp] = hi;
    }
    __syncthreads();
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        lo = min(lo, sm->red[w]);
        hi = max(hi, sm->red[8 + w]);
    }
    const int z = hi > lo ? __clz(hi - lo) : 0;
    // 2. histogram of the mapped keys' top 12 bits
    walk([&](uint32_t key, int, bool v) {
        if (v) atomicAdd(&hist[((key - lo) << z) >> kHistShift], 1u);
    });
    __syncthreads();
    // 3. boundary bin of the k-th largest
    block_find_suffix(hist, kHistBins, static_cast<uint32_t>(k), sm->scratch, &sm->bnd);
    const int bstar = sm->bnd.bin;   // -1: fewer than k scores, all are taken
    const uint32_t bthr = bstar >= 0 ? static_cast<uint32_t>(bstar) : 0u;
    // 4. collect the composites (mapped keys) in bins >= the boundary: each
    //    warp appends to its own segment of buf[2048, 4096) with ballots,
    //    then the segments are packed into buf[0, count)
    constexpr int kSeg = 2048 / 8;
    uint64_t* segs = buf + 2048;
    uint32_t cnt = 0;   // this warp's, the same in every lane
    walk([&](uint32_t key, int idx, bool v) {
        const uint32_t m = (key - lo) << z;
        const bool t = v && (m >> kHistShift) >= bthr;
        const unsigned b = __ballot_sync(0xffffffffu, t);
        if (t) {
            const uint32_t p = cnt + static_cast<uint32_t>(__popc(b & ((1u << lane) - 1u)));
            if (p < static_cast<uint32_t>(kSeg)) segs[warp * kSeg + p] = make_comp(m, idx);
        }
        cnt += static_cast<uint32_t>(__popc(b));
    });
    if (lane == 0) sm->wcnt[warp] = cnt;
    __syncthreads();
    uint32_t before = 0, count = 0;
    bool over = false;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t c = sm->wcnt[w];
        before += w < warp ? c : 0u;
        count += c;
        over |= c > static_cast<uint32_t>(kSeg);
    }
    int nsort;
    if (!over && count <= 2048u) {
        for (uint32_t i = lane; i < cnt; i += 32) buf[before + i] = segs[warp * kSeg + i];
        __syncthreads();
        nsort = static_cast<int>(count);
        if (bstar >= 0 && count > static_cast<uint32_t>(max(kTopkThreads, next_pow2(k)))) {
            // 5. a crowded boundary bin: keep its best (k - above) by radix
            //    passes over the collected list, then compact
            const uint32_t above = sm->bnd.above;
            const uint32_t m = static_cast<uint32_t>(k) - above;
            auto each = [&](auto f) { walk_smem(buf, count, f); };
            SelectSmem* ss = reinterpret_cast<SelectSmem*>(hist);   // the histogram is no longer needed
            const uint64_t thr = radix_refine(each, bstar, m, ss);
            nsort = static_cast<int>(block_collect(
                each, [&](uint64_t c) { return static_cast<int>(comp_key(c) >> kHistShift) > bstar || c >= thr; },
                segs, 2048u, sm->scratch));
            for (int i = tid; i < nsort; i += kTopkThreads) buf[i] = segs[i];
            __syncthreads();
        }
    } else {
        // many equal or near-equal scores in the boundary bin (more than the
        // buffer holds): refine the boundary bin over the whole segment, then
        // collect exactly k
        __syncthreads();
        const uint32_t above = sm->bnd.above;
        const uint32_t m = static_cast<uint32_t>(k) - above;
        auto each_all = [&](auto f) {
            walk([&](uint32_t key, int idx, bool v) { f(make_comp((key - lo) << z, idx), v); });
        };
        SelectSmem* ss = reinterpret_cast<SelectSmem*>(hist);
        const uint64_t thr = radix_refine(each_all, bstar, m, ss);
        nsort = static_cast<int>(block_collect(
            each_all, [&](uint64_t c) { return static_cast<int>(comp_key(c) >> kHistShift) > bstar || c >= thr; },
            buf, static_cast<uint32_t>(k), sm->scratch));
        nsort = min(nsort, k);
    }
    // 6. sort, then map the keys back
    block_sort_any(buf, nsort, buf + 2048);
    const int nout = min(k, nsort);
    for (int j = tid; j < nout; j += kTopkThreads) {
        const uint64_t c = buf[j];
        buf[j] = make_comp((comp_key(c) >> z) + lo, comp_index(c));
    }
    __syncthreads();
    return nout;
}


// ---------------------------------------------------------------------------
// Ordering a small candidate set without a comparison sort
// ---------------------------------------------------------------------------

// Sorts the n composites of a[0, n) descending, n <= 2048, leaving them in
// a[0, n); every key is at least lo.  The keys in [lo, hi] are mapped onto 32
// bits over that range, keys above hi go to the top bin (so a few outlying
// large scores need not stretch the range that the rest share), and a
// 4096-bin histogram gives each bin its first output place (thread t holds
// bins 16 t .. 16 t + 15 in registers); every element is scattered to its
// bin's next place in tmp and then placed by its rank inside its bin (bins
// hold a few elements for spread keys).  A bin of more than 64 elements (many
// equal or very close keys) sends the set to the block sort.  Bin b lives at
// word b ^ ((b >> 3) & 12) of hist and cur, so that the 16-byte slots of
// eight consecutive threads' bins fall on distinct banks.  hist, cur: 4096
// words each; tmp: n composites (disjoint from a).  All 256 threads.
__device__ __noinline__ void bin_order(uint64_t* a, int n, uint64_t* tmp, uint32_t lo, uint32_t hi, uint32_t* hist,
                                       uint32_t* cur, SegSelSmem* sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int z = hi > lo ? __clz(hi - lo) : 0;
    auto word_of = [&](uint64_t c) {
        const uint32_t key = comp_key(c);
        const uint32_t b = key > hi ? static_cast<uint32_t>(kHistBins - 1) : ((key - lo) << z) >> kHistShift;
        return b ^ ((b >> 3) & 12u);
    };
    auto slot_of = [](uint32_t s) { return s ^ ((s >> 3) & 3u); };   // 16-byte slot s = 4 t + j
    {
        uint4* h4 = reinterpret_cast<uint4*>(hist);
        for (int i = tid; i < kHistBins / 4; i += kTopkThreads) h4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) atomicAdd(&hist[word_of(a[i])], 1u);
    __syncthreads();
    // counts of this thread's 16 bins, their first places, the largest count
    uint32_t v[16];
    {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = h4[slot_of(static_cast<uint32_t>(4 * tid + j))];
            v[4 * j] = x.x;
            v[4 * j + 1] = x.y;
            v[4 * j + 2] = x.z;
            v[4 * j + 3] = x.w;
        }
    }
    uint32_t sum = 0, mx = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        sum += v[j];
        mx = max(mx, v[j]);
    }
    uint32_t incl = sum;   // over this warp's lanes >= lane (higher bins)
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) {
        sm->scratch[warp] = incl;
        sm->scratch[8 + warp] = mx;
    }
    __syncthreads();
    uint32_t after = incl - sum;
    mx = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        after += q > warp ? sm->scratch[q] : 0u;
        mx = max(mx, sm->scratch[8 + q]);
    }
    if (mx > 64u) {
        block_sort_any(a, n, tmp);
        return;
    }
    {
        uint32_t st[16];
        uint32_t acc = after;
#pragma unroll
        for (int j = 15; j >= 0; --j) {
            st[j] = acc;
            acc += v[j];
        }
        uint4* o4 = reinterpret_cast<uint4*>(hist);
        uint4* c4 = reinterpret_cast<uint4*>(cur);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = make_uint4(st[4 * j], st[4 * j + 1], st[4 * j + 2], st[4 * j + 3]);
            const uint32_t sl = slot_of(static_cast<uint32_t>(4 * tid + j));
            o4[sl] = x;
            c4[sl] = x;
        }
    }
    __syncthreads();
    // scatter every element to its bin's next place
    for (int i = tid; i < n; i += kTopkThreads) {
        const uint64_t c = a[i];
        tmp[atomicAdd(&cur[word_of(c)], 1u)] = c;
    }
    __syncthreads();
    // place every element by its rank inside its bin [hist[w], cur[w]): the
    // same trip counts in a warp (the rank loop runs to the warp's largest
    // bin), bin mates read four at a time (a composite is never zero, so a
    // zero in a lane past its bin's end counts nothing)
    for (int i0 = 0; i0 < n; i0 += kTopkThreads) {
        const int i = i0 + tid;
        const bool ok = i < n;
        const uint64_t c = ok ? tmp[i] : 0ull;
        const uint32_t w = word_of(c);
        const uint32_t s0 = ok ? hist[w] : 0u;
        const uint32_t cnt = ok ? cur[w] - s0 : 0u;
        const uint32_t m = __reduce_max_sync(0xffffffffu, cnt);
        uint32_t r = s0;
        for (uint32_t j = 0; j < m; j += 4) {
            const uint64_t t0 = j < cnt ? tmp[s0 + j] : 0ull;
            const uint64_t t1 = j + 1 < cnt ? tmp[s0 + j + 1] : 0ull;
            const uint64_t t2 = j + 2 < cnt ? tmp[s0 + j + 2] : 0ull;
            const uint64_t t3 = j + 3 < cnt ? tmp[s0 + j + 3] : 0ull;
            r += (t0 > c ? 1u : 0u) + (t1 > c ? 1u : 0u) + (t2 > c ? 1u : 0u) + (t3 > c ? 1u : 0u);
        }
        if (ok) a[r] = c;
    }
    __syncthreads();
}

// Histogram windows of the decode selection: bins of the score key at
// 1/16 octave (key >> 19: sign, exponent and 4 mantissa bits; 8192 bins over
// all keys); a CTA's window is the 256 bins below its largest score.
constexpr int kWinShift = 19;
constexpr int kWinBins = 256;                        // bins of a window, ending at the chunk's largest
constexpr int kWinHead = 4;                          // anchor bin, count, largest key, device-check flag
constexpr int kWinWords = kWinHead + kWinBins / 2;   // then 16-bit counts in pairs (528 bytes)
constexpr int kCountSortMax = 96;                    // longest candidate list sorted by counting

__device__ __forceinline__ uint32_t win_bin(uint32_t key) { return key >> kWinShift; }


// Ranks of the candidates of a bin-major pool, for the rank positions
// [lo, hi) of one CTA: pool[0, ctot) holds the bins from the top down (bin
// index t = (key >> kWinShift) - wlo; bin t's entries, in any order, at
// [bstart[t], bstart[t] + blen[t])), tb is the lowest bin index with
// candidates.  emit(r, c) is called once for each rank r < nsel in [lo, hi):
// an entry of a bin of at most kRankCrowd entries by the CTA whose [lo, hi)
// holds its pool slot (rank = bstart plus the larger entries of the bin); a
// crowded bin is sorted by counting on the next 8 key bits (256 sub-bins of a
// few entries, ranks inside a sub-bin by comparison) by every CTA whose
// [lo, hi) it reaches, each emitting the ranks in its range.  Scratch: scnt,
// scur, clist 256 words each, srt 2048 composites, counter one word, wcnt 8
// words.  All 256 threads.
constexpr int kRankCrowd = 128;
template <class Emit>
__device__ __forceinline__ void rank_pool(const uint64_t* pool, int lo, int hi, int nsel, int tb, int wlo,
                                          const uint32_t* bstart, const uint32_t* blen, uint32_t* scnt,
                                          uint32_t* scur, uint32_t* clist, uint64_t* srt, uint32_t* counter,
                                          uint32_t* wcnt, Emit emit) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = lo + tid; i < hi; i += kTopkThreads) {
        const uint64_t x = pool[i];
        const int t = static_cast<int>(win_bin(comp_key(x))) - wlo;
        const int s0 = static_cast<int>(bstart[t]), e0 = s0 + static_cast<int>(blen[t]);
        if (e0 - s0 > kRankCrowd) continue;
        int rk = s0;
        for (int j = s0; j < e0; ++j) rk += pool[j] > x ? 1 : 0;
        if (rk < nsel) emit(rk, x);
    }
    auto sub = [](uint64_t c) { return (comp_key(c) >> (kWinShift - 8)) & 0xFFu; };
    if (tid == 0) *counter = 0u;
    __syncthreads();
    {
        const int t = tid;
        const int s0 = static_cast<int>(bstart[t]), len = static_cast<int>(blen[t]);
        if (t >= tb && len > kRankCrowd && s0 < hi && s0 + len > lo) clist[atomicAdd(counter, 1u)] = static_cast<uint32_t>(t);
    }
    __syncthreads();
    const int ncrowd = static_cast<int>(*counter);
    for (int ci = 0; ci < ncrowd; ++ci) {
        const int t = static_cast<int>(clist[ci]);
        const int s0 = static_cast<int>(bstart[t]), len = static_cast<int>(blen[t]);
        scnt[tid] = 0u;
        __syncthreads();
        for (int j = tid; j < len; j += kTopkThreads) atomicAdd(&scnt[sub(pool[s0 + j])], 1u);
        __syncthreads();
        // sub-bin tid starts after every entry of the higher sub-bins
        const uint32_t v = scnt[tid];
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32) incl += y;
        }
        if (lane == 0) wcnt[warp] = incl;
        __syncthreads();
        uint32_t start = incl - v;
#pragma unroll
        for (int q = 0; q < 8; ++q) start += q > warp ? wcnt[q] : 0u;
        scur[tid] = start;
        __syncthreads();
        for (int j = tid; j < len; j += kTopkThreads) {
            const uint64_t y = pool[s0 + j];
            srt[atomicAdd(&scur[sub(y)], 1u)] = y;
        }
        __syncthreads();
        // ranks inside a sub-bin: the same trip counts in a warp (to the
        // warp's largest sub-bin), sub-bin mates read four at a time (a
        // composite is never zero, so a zero past a sub-bin's end counts
        // nothing)
        for (int q0 = 0; q0 < len; q0 += kTopkThreads) {
            const int q = q0 + tid;
            const uint64_t y = q < len ? srt[q] : 0ull;
            const uint32_t u = sub(y);
            const int en = static_cast<int>(scur[u]);
            const int c = q < len ? static_cast<int>(scnt[u]) : 0;
            const int st = en - c;
            const int m = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(c));
            int fp = st;
            for (int z = 0; z < m; z += 4) {
                const uint64_t t0 = z < c ? srt[st + z] : 0ull;
                const uint64_t t1 = z + 1 < c ? srt[st + z + 1] : 0ull;
                const uint64_t t2 = z + 2 < c ? srt[st + z + 2] : 0ull;
                const uint64_t t3 = z + 3 < c ? srt[st + z + 3] : 0ull;
                fp += (t0 > y ? 1 : 0) + (t1 > y ? 1 : 0) + (t2 > y ? 1 : 0) + (t3 > y ? 1 : 0);
            }
            const int rk = s0 + fp;
            if (q < len && rk >= lo && rk < hi && rk < nsel) emit(rk, y);
        }
        __syncthreads();
    }
}

// Exact sorted top-k over the nseg sorted runs of k composites (zero-padded)
// of one sequence, runs[j * k + e] in global memory, given the histogram gh
// (kGHistWords words: kGHistBins bins of key >> 19 over every run entry, then
// the largest bin + 1) and the sequence's device-check flag, read together
// with the largest bin.  The boundary bin of the k-th largest entry comes
// from the 256 bins below the largest (all 8192 bins when those hold fewer
// than k), and so does the bin where the count from the top reaches
// min(16, k); gh is then zeroed for the next call (every segment added its
// counts before taking its ticket), the stores draining while the candidates
// are read.  The candidates are each run's prefix at or above the boundary
// (runs are sorted): with two runs, the two prefixes merged; else read in
// rounds -- every open run's next R entries, R sized so that a round is about
// 2048 loads over the block, a run staying open while its last read entry is
// a candidate -- and put in order by bin_order over the key range from the
// boundary bin to the top of the min(16, k) bin (the few entries above, such
// as one planted far larger score, share the top bin).  With more than 2048
// candidates, selects over all run entries (seg_select).
// buf: >= 4096 composites; hist, cur: 4096 words.  Returns nout, buf[0, nout)
// sorted descending, or -1 when the flag is set.  All 256 threads.
__device__ __noinline__ int merge_runs(const uint64_t* runs, int nseg, int k, uint32_t* gh, const uint32_t* seqflag,
                                       uint32_t* hist, uint32_t* cur, uint64_t* buf, SegSelSmem* sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t bad = __ldcg(seqflag);
    const int gm = static_cast<int>(__ldcg(gh + kGHistBins)) - 1;   // largest bin of any entry
    if (tid == 0) {
        sm->bnd.bin = -1;
        sm->bnd.above = 0u;
        sm->red[1] = static_cast<uint32_t>(gm);   // top of bin_order's range (all bins when not found below)
    }
    if (bad == 0u && gm >= 0) {   // (the same in every thread)
        // the 256 bins below the largest: thread t holds bin gm - 255 + t
        {
            const int bt = gm - (kWinBins - 1) + tid;
            const uint32_t v = bt >= 0 ? __ldcg(gh + bt) : 0u;
            uint32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += y;
            }
            if (lane == 0) sm->wcnt[warp] = incl;
            __syncthreads();
            uint32_t after = incl - v;
#pragma unroll
            for (int q = 0; q < 8; ++q) after += q > warp ? sm->wcnt[q] : 0u;
            const uint32_t kk = static_cast<uint32_t>(k);
            if (after < kk && kk <= after + v) {
                sm->bnd.bin = bt;
                sm->bnd.above = after + v;   // entries at or above the bin
            }
            // the bin where the count from the top reaches min(16, k) (at or
            // above the boundary bin, since that count is at most k)
            const uint32_t kt = min(kk, 16u);
            if (after < kt && kt <= after + v) sm->red[1] = static_cast<uint32_t>(bt);
            __syncthreads();
        }
        if (sm->bnd.bin < 0) {
            // fewer than k entries in those bins: the suffix over all 8192 bins
            // (thread t holds bins 32 t .. 32 t + 31)
            uint32_t v[32];
            {
                const uint4* g4 = reinterpret_cast<const uint4*>(gh) + 8 * tid;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 x = __ldcg(g4 + j);
                    v[4 * j] = x.x;
                    v[4 * j + 1] = x.y;
                    v[4 * j + 2] = x.z;
                    v[4 * j + 3] = x.w;
                }
            }
            uint32_t sum = 0;
#pragma unroll
            for (int j = 0; j < 32; ++j) sum += v[j];
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_down_sync(0xffffffffu, incl, o);
                if (lane + o < 32) incl += y;
            }
            __syncthreads();
            if (lane == 0) sm->wcnt[warp] = incl;
            __syncthreads();
            uint32_t after = incl - sum, total = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t x = sm->wcnt[q];
                after += q > warp ? x : 0u;
                total += x;
            }
            const uint32_t kk = min(static_cast<uint32_t>(k), total);
            if (kk > 0u && after < kk && kk <= after + sum) {
                uint32_t acc = after;
#pragma unroll
                for (int j = 31; j >= 0; --j) {
                    if (acc < kk && kk <= acc + v[j]) {
                        sm->bnd.bin = 32 * tid + j;
                        sm->bnd.above = acc + v[j];
                    }
                    acc += v[j];
                }
            }
        }
    }
    // every read of gh is done: zero it (16-byte stores, nothing waits on them)
    __syncthreads();
    {
        uint4* g4 = reinterpret_cast<uint4*>(gh);
        for (int i = tid; i < kGHistWords / 4; i += kTopkThreads) g4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (bad != 0u) return -1;
    if (sm->bnd.bin < 0) return 0;
    const int gtop = static_cast<int>(sm->red[1]);
    const int bstar = sm->bnd.bin;
    const uint32_t ncand = sm->bnd.above;
    if (ncand <= 2048u && nseg == 2) {
        uint64_t* cand = buf + 2048;
        // Two runs (a sequence of two segments): each run is sorted, so its
        // candidates (entries of bins >= bstar) are a prefix.  Find the two
        // prefix lengths, copy the prefixes next to each other and merge them
        // by merge path (a co-rank search per thread, then its share of the
        // outputs in order).  Measured 3.5 against 7 us for the pooled order
        // below; with 16 runs the four pairwise levels this would take cost
        // more than the pooled order (13 against 7 us), so more runs use it.
        const uint64_t thr = static_cast<uint64_t>(static_cast<uint32_t>(bstar) << kWinShift) << 32;
        auto qual = [&](unsigned long long c) { return c != 0ull && c >= thr; };
        const unsigned long long* rr = reinterpret_cast<const unsigned long long*>(runs);
        uint32_t* rlen = sm->scratch;        // [2] prefix lengths
        if (warp < 2) {
            // warp r probes run r: chunks whose last entry qualifies are full
            // (and come first), then the entries of the first chunk that is not
            const unsigned long long* R = rr + static_cast<int64_t>(warp) * k;
            const int chunk = (k + 31) >> 5;   // lane l's chunk: [l chunk, (l + 1) chunk)
            const int jl = min(k, (lane + 1) * chunk) - 1;
            const bool full = jl >= lane * chunk && qual(__ldcg(R + jl));
            const int base = __popc(__ballot_sync(0xffffffffu, full)) * chunk;
            int len = min(base, k);
            for (int q0 = 0; q0 < chunk && base < k; q0 += 32) {
                const int j = base + q0 + lane;
                len += __popc(__ballot_sync(0xffffffffu, q0 + lane < chunk && j < k && qual(__ldcg(R + j))));
            }
            if (lane == 0) rlen[warp] = static_cast<uint32_t>(len);
        }
        __syncthreads();
        const int la = static_cast<int>(rlen[0]), lb = static_cast<int>(rlen[1]);
        const int total = la + lb;
        if (total <= 2048) {
            // run 0's prefix at cand[0, la), run 1's at cand[la, total); all
            // of a thread's loads in flight at once
            {
                unsigned long long v[2048 / kTopkThreads];
#pragma unroll
                for (int q = 0; q < 2048 / kTopkThreads; ++q) {
                    const int f = tid + q * kTopkThreads;
                    v[q] = f < total ? __ldcg(f < la ? rr + f : rr + k + (f - la)) : 0ull;
                }
#pragma unroll
                for (int q = 0; q < 2048 / kTopkThreads; ++q) {
                    const int f = tid + q * kTopkThreads;
                    if (f < total) cand[f] = static_cast<uint64_t>(v[q]);
                }
            }
            __syncthreads();
            const int nout = min(k, total);
            const int per = (nout + kTopkThreads - 1) / kTopkThreads;
            const int d = tid * per;   // this thread's first output
            if (d < nout) {
                const uint64_t* A = cand;
                const uint64_t* B = cand + la;
                int lo = max(0, d - lb), hi = min(d, la);
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (A[mid] > B[d - 1 - mid]) lo = mid + 1;
                    else hi = mid;
                }
                int i = lo, j = d - lo;
                for (int g = d; g < min(nout, d + per); ++g) {
                    const bool ta = j >= lb || (i < la && A[i] > B[j]);
                    buf[g] = ta ? A[i++] : B[j++];
                }
            }
            __syncthreads();
            return nout;
        }
        __syncthreads();
    }
    if (ncand <= 2048u) {
        uint64_t* cand = buf;   // put in order in place, buf[2048, 4096) the scratch
        uint32_t* cnt = &sm->red[0];
        // open runs of a round: two lists of 128 in sm->scratch, used in turn
        if (tid == 0) {
            *cnt = 0u;
            sm->red[2] = 0u;
            sm->red[3] = 0u;
        }
        __syncthreads();
        const unsigned long long* rr = reinterpret_cast<const unsigned long long*>(runs);
        constexpr int U = 8;   // loads in flight per thread
        // a round's length R = 2^lg: the largest power of two at most
        // U * 256 / open, and at least 32 (entry f of a round is entry
        // f & (R - 1) of open run f >> lg, no division)
        auto round_lg = [&](int open) {
            const int r = U * kTopkThreads / open;
            return r < 32 ? 5 : 31 - __clz(static_cast<uint32_t>(r));
        };
        // every run is open at first; a run stays open only when all of the
        // R >= 32 entries it gave are candidates, so at most 64 stay open
        int m = 0, nopen = nseg, li = 0;
        bool all = true;
        int lg = round_lg(nseg);
        while (true) {
            const int R = 1 << lg;
            const int rlen = min(R, k - m);   // entries read of each open run
            const int nflat = nopen * R;
            const uint32_t* cur_list = sm->scratch + 128 * li;
            uint32_t* next_list = sm->scratch + 128 * (li ^ 1);
            uint32_t* next_n = &sm->red[2 + (li ^ 1)];
            for (int f0 = 0; f0 < nflat; f0 += U * kTopkThreads) {
                uint64_t c[U];
                int jr[U], e[U];
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const int f = f0 + q * kTopkThreads + tid;
                    const int jj = f >> lg;
                    e[q] = f & (R - 1);
                    const bool in = f < nflat && e[q] < rlen;
                    jr[q] = in ? (all ? jj : static_cast<int>(cur_list[jj])) : 0;
                    c[q] = in ? static_cast<uint64_t>(__ldcg(rr + static_cast<int64_t>(jr[q]) * k + m + e[q])) : 0ull;
                }
                uint32_t mask = 0u;
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const bool t = c[q] != 0ull && static_cast<int>(win_bin(comp_key(c[q]))) >= bstar;
                    mask |= t ? (1u << q) : 0u;
                    if (t && e[q] == rlen - 1 && m + rlen < k)
                        next_list[atomicAdd(next_n, 1u) & 127u] = static_cast<uint32_t>(jr[q]);
                }
                // the candidates appended with one shared atomic per warp
                const uint32_t mine = static_cast<uint32_t>(__popc(mask));
                uint32_t incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t base = 0u;
                if (lane == 31 && incl != 0u) base = atomicAdd(cnt, incl);
                uint32_t pos = __shfl_sync(0xffffffffu, base, 31) + incl - mine;
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    if ((mask >> q) & 1u) {
                        if (pos < 2048u) cand[pos] = c[q];
                        ++pos;
                    }
                }
            }
            __syncthreads();
            nopen = static_cast<int>(min(*next_n, 128u));
            if (nopen == 0) break;
            if (tid == 0) sm->red[2 + li] = 0u;   // the list read this round is written next
            m += rlen;
            li ^= 1;
            all = false;
            lg = round_lg(nopen);
            __syncthreads();
        }
        const int got = static_cast<int>(min(*cnt, 2048u));
        // keys from the boundary bin's floor; the range mapped runs to the top
        // of gtop (at most 15 entries lie above it)
        const uint32_t lo = static_cast<uint32_t>(bstar) << kWinShift;
        const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(gtop + 1) << kWinShift) - 1u);
        bin_order(cand, got, buf + 2048, lo, hi, hist, cur, sm);
        return min(k, got);
    }
    return seg_select(GCompSet{runs, nseg * k}, k, hist, buf, sm);
}

}  // namespace dsaidx
