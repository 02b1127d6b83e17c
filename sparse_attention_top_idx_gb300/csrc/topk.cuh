// topk.cuh -- block-level exact top-k machinery (256 threads per block).
//
// Every candidate is a 64-bit composite (score_key << 32) | ~index: the order
// of composites is "higher score first, then lower index", the tie rule of the
// library, and composites are unique within one query row.  Selection works on
// a 4096-bin histogram of the top 12 bits of score_key followed by exact radix
// refinement of the boundary bin, and finishes with a sort of the k winners.
#pragma once

#include "common.cuh"

namespace dsaidx {

constexpr int kTopkThreads = 256;

__device__ __forceinline__ uint64_t make_comp(uint32_t key, int32_t idx) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(idx));
}
__device__ __forceinline__ int32_t comp_index(uint64_t c) {
    return static_cast<int32_t>(~static_cast<uint32_t>(c & 0xFFFFFFFFull));
}
__device__ __forceinline__ uint32_t comp_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ uint32_t key_bin(uint32_t key) { return key >> kHistShift; }

// Shared-memory histogram increment for the lanes with `valid`.  A plain
// atomic per lane: on sm_103a this measured about three times faster than
// first aggregating equal bins with a warp match, even when most lanes of a
// warp share a few bins.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool valid) {
    if (valid) atomicAdd(&hist[bin], 1u);
}

struct Boundary {
    int bin;          // largest bin whose suffix count reaches `need` (-1: total < need)
    uint32_t above;   // candidates in bins strictly above `bin` (the total when bin = -1)
    uint32_t at;      // candidates inside `bin` (0 when bin = -1)
};

// Find the bin holding the need-th largest candidate of a histogram of nbins
// (a multiple of 256) bins.  Called by all 256 threads; scratch holds >= 256
// words.  Result in *out (shared), valid after the call for every thread.
// Thread t sums bins per t .. per t + per - 1; with 4096 bins (16 a thread,
// hist 16-byte aligned) it reads them as four 16-byte slots, each thread
// starting at slot (t >> 1) & 3, so that eight consecutive threads hit
// distinct banks (word-by-word, a warp's 32 threads hit two banks).
__device__ __forceinline__ void block_find_suffix(const uint32_t* hist, int nbins, uint32_t need,
                                  uint32_t* scratch, Boundary* out) {
    const int tid = threadIdx.x;
    const int per = nbins / kTopkThreads;
    uint32_t s = 0;
    if (per == 16) {
        const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 4 * tid;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = h4[(j + (tid >> 1)) & 3];
            s += x.x + x.y + x.z + x.w;
        }
    } else {
        for (int i = 0; i < per; ++i) s += hist[tid * per + i];
    }
    scratch[tid] = s;
    __syncthreads();
    if (tid < 32) {
        // lane l owns partials [8l, 8l + 8)
        uint32_t ls = 0;
        for (int i = 0; i < 8; ++i) ls += scratch[tid * 8 + i];
        uint32_t incl = ls;  // sum over lanes >= l
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
            if (tid + o < 32) incl += v;
        }
        uint32_t after = incl - ls;  // sum over lanes > l
        uint32_t total = __shfl_sync(0xffffffffu, incl, 0);
        if (total < need) {
            if (tid == 0) {
                out->bin = -1;
                out->above = total;
                out->at = 0;
            }
        } else if (after < need && need <= incl) {
            uint32_t acc = after;
            int p = tid * 8;
            for (int j = 7; j >= 0; --j) {
                uint32_t v = scratch[tid * 8 + j];
                if (acc + v >= need) {
                    p = tid * 8 + j;
                    break;
                }
                acc += v;
            }
            for (int j = per - 1; j >= 0; --j) {
                uint32_t v = hist[p * per + j];
                if (acc + v >= need) {
                    out->bin = p * per + j;
                    out->above = acc;
                    out->at = v;
                    break;
                }
                acc += v;
            }
        }
    }
    __syncthreads();
}

// Shared scratch of the selection routines.
struct SelectSmem {
    uint32_t hist256[256];
    uint32_t scratch[256];
    Boundary bnd;
    uint32_t nsel;       // entries in sel
    uint32_t nbnd;       // entries seen in the boundary bin
    uint64_t thr;        // composite threshold of the boundary refinement
};

// Block-wide stream compaction without atomics: every composite c of the walk
// with valid && take(c) goes to dst (the first `cap` of them), thread t's in
// walk order after those of threads < t.  Two passes over the walk (count,
// then write at the scanned offset): on sm_103a this measured several times
// faster than a warp-aggregated atomic append, whose returned offset puts a
// shared atomic's latency in every iteration.  Returns the number taken
// (which may exceed cap); wsum: 8 words of scratch.  All 256 threads.
template <class Walk, class Take>
__device__ __forceinline__ uint32_t block_collect(Walk walk, Take take, uint64_t* dst, uint32_t cap,
                                                  uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t mine = 0;
    walk([&](uint64_t c, bool v) { mine += (v && take(c)) ? 1u : 0u; });
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t pos = incl - mine, total = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const uint32_t t = wsum[w];
        pos += (w < warp) ? t : 0u;
        total += t;
    }
    walk([&](uint64_t c, bool v) {
        if (v && take(c)) {
            if (pos < cap) dst[pos] = c;
            ++pos;
        }
    });
    __syncthreads();
    return total;
}

// The same compaction in one pass, for a walk with warp-uniform trip counts:
// each warp appends its taken composites (ballot + popc, a running count in a
// register) to its own segment of `seg` (cap / 8 entries per warp), then the
// segments are copied to dst in warp order.  When a warp's segment overflows,
// falls back to block_collect.  seg: cap composites of scratch, disjoint
// from dst.  Returns the number taken.  All 256 threads.
template <class Walk, class Take>
__device__ __forceinline__ uint32_t block_collect_warp(Walk walk, Take take, uint64_t* dst, uint32_t cap,
                                                       uint64_t* seg, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t segcap = cap / (kTopkThreads / 32);
    uint64_t* mine = seg + warp * segcap;
    uint32_t cnt = 0;   // the same in every lane
    walk([&](uint64_t c, bool v) {
        const bool t = v && take(c);
        const unsigned m = __ballot_sync(0xffffffffu, t);
        if (t) {
            const uint32_t p = cnt + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
            if (p < segcap) mine[p] = c;
        }
        cnt += static_cast<uint32_t>(__popc(m));
    });
    if (lane == 0) wsum[warp] = cnt;
    __syncthreads();
    uint32_t before = 0, total = 0;
    bool over = false;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const uint32_t t = wsum[w];
        before += (w < warp) ? t : 0u;
        total += t;
        over |= t > segcap;
    }
    if (!over) {
        for (uint32_t i = lane; i < cnt; i += 32) dst[before + i] = mine[i];
    }
    __syncthreads();
    if (over) return block_collect(walk, take, dst, cap, wsum);
    return total;
}

// block_collect_warp for a walk over 32-bit score keys: walkk(f) calls
// f(key, index, valid) with warp-uniform trip counts, and the composites of
// keys >= kthr are collected (the composite is built only for those).  On
// overflow of a warp's segment, two passes (count, then write at the scanned
// offset).  Returns the number taken.  All 256 threads.
template <class WalkK>
__device__ __forceinline__ uint32_t block_collect_keys(WalkK walkk, uint32_t kthr, uint64_t* dst, uint32_t cap,
                                                       uint64_t* seg, uint32_t* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t segcap = cap / (kTopkThreads / 32);
    uint64_t* mine = seg + warp * segcap;
    uint32_t cnt = 0, own = 0;   // cnt: the warp's (same in every lane); own: this lane's
    walkk([&](uint32_t key, int idx, bool v) {
        const bool t = v && key >= kthr;
        const unsigned m = __ballot_sync(0xffffffffu, t);
        if (t) {
            const uint32_t p = cnt + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
            if (p < segcap) mine[p] = make_comp(key, idx);
        }
        cnt += static_cast<uint32_t>(__popc(m));
        own += t ? 1u : 0u;
    });
    if (lane == 0) wsum[warp] = cnt;
    __syncthreads();
    uint32_t before = 0, total = 0;
    bool over = false;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const uint32_t t = wsum[w];
        before += (w < warp) ? t : 0u;
        total += t;
        over |= t > segcap;
    }
    if (!over) {
        for (uint32_t i = lane; i < cnt; i += 32) dst[before + i] = mine[i];
        __syncthreads();
        return total;
    }
    // a warp overflowed its segment: thread-ordered write at scanned offsets
    __syncthreads();
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    uint32_t pos = incl - own;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) pos += (w < warp) ? wsum[w] : 0u;
    walkk([&](uint32_t key, int idx, bool v) {
        if (v && key >= kthr) {
            if (pos < cap) dst[pos] = make_comp(key, idx);
            ++pos;
        }
    });
    __syncthreads();
    return total;
}

// Candidate walks.  A walk `each(f)` calls f(comp, valid) for every candidate,
// strided over the block's 256 threads, with the same number of calls in every
// lane of a warp (lanes past the end get valid = false), so f may use warp
// collectives.

// A shared-memory array of n composites.
template <class F>
__device__ __forceinline__ void walk_smem(const uint64_t* a, uint32_t n, F f) {
    for (uint32_t b0 = 0; b0 < n; b0 += kTopkThreads) {
        const uint32_t i = b0 + threadIdx.x;
        const bool v = i < n;
        f(v ? a[i] : 0ull, v);
    }
}

// A global row of n fp32 scores (16-byte aligned, readable up to n rounded up
// to 4): candidate i is (score_key(row[i]), i).  Four float4 loads in flight
// (measured best: eight or sixteen made the select slower, two no faster).
template <class F>
__device__ __forceinline__ void walk_row(const float* row, int n, F f) {
    constexpr int U = 4;
    const float4* r4 = reinterpret_cast<const float4*>(row);
    for (int b0 = 0; b0 < n; b0 += kTopkThreads * 4 * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b0 + (u * kTopkThreads + static_cast<int>(threadIdx.x)) * 4;
            v[u] = (i < n) ? __ldcg(r4 + (i >> 2)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b0 + (u * kTopkThreads + static_cast<int>(threadIdx.x)) * 4;
            f(make_comp(score_key(v[u].x), i), i < n);
            f(make_comp(score_key(v[u].y), i + 1), i + 1 < n);
            f(make_comp(score_key(v[u].z), i + 2), i + 2 < n);
            f(make_comp(score_key(v[u].w), i + 3), i + 3 < n);
        }
    }
}

// A compact walk over the same row, one load per iteration: for the rare
// paths that walk the candidates again (small code, slow).
template <class F>
__device__ __forceinline__ void walk_row_slow(const float* row, int n, F f) {
#pragma unroll 1
    for (int b0 = 0; b0 < n; b0 += kTopkThreads) {
        const int i = b0 + static_cast<int>(threadIdx.x);
        f(make_comp(score_key(i < n ? __ldcg(row + i) : 0.0f), i), i < n);
    }
}

// Exact refinement inside one bin: among the candidate set X (all composites
// whose top 12 bits equal `bin`), find the composite threshold thr such that
// exactly m members of X are >= thr.  `each` walks a superset of X (members
// outside X are filtered here).  Called by all 256 threads.
template <class Each>
__device__ uint64_t radix_refine(Each each, int bin, uint32_t m, SelectSmem* ss) {
    uint64_t prefix = static_cast<uint64_t>(bin) << 52;
    uint64_t mask = 0xFFFull << 52;
    uint32_t need = m;
#pragma unroll 1
    for (int pass = 0; pass < 7; ++pass) {
        const int sh = pass < 6 ? 44 - 8 * pass : 0;   // 8-bit digits, then the last 4 bits
        const uint64_t dmask = (pass == 6) ? 0xFull : 0xFFull;
        ss->hist256[threadIdx.x] = 0;
        __syncthreads();
        each([&](uint64_t c, bool v) {
            hist_add_warp(ss->hist256, static_cast<uint32_t>((c >> sh) & dmask), v && (c & mask) == prefix);
        });
        __syncthreads();
        block_find_suffix(ss->hist256, 256, need, ss->scratch, &ss->bnd);
        const int d = ss->bnd.bin;   // never -1: X holds at least `need` members
        const uint32_t above = ss->bnd.above;
        const uint32_t at = ss->bnd.at;
        __syncthreads();
        need -= above;
        prefix |= static_cast<uint64_t>(d) << sh;
        mask |= dmask << sh;
        if (at == need) break;  // every member with this prefix is selected
    }
    return prefix;
}

// ---------------------------------------------------------------------------
// Merge sort, descending, of up to 256 * E composites (all 256 threads).
// Each warp sorts a run of 32 * E composites in registers (bitonic network,
// E per lane, lane l holding run positions l*E .. l*E+E-1: compare-exchanges
// between a lane's registers, then across lanes by shuffles, no block
// barriers).  Three merge-path levels then merge the eight runs pairwise
// (8 -> 4 -> 2 -> 1): each thread finds, by a binary search on its output
// diagonal, how many of its first output's predecessors come from each run
// of its pair and merges its E outputs sequentially.  Zero is the padding
// value: positions at or beyond n hold zeros at every level (the zeros sort
// last), so they are neither read nor written.  This code runs once per
// block from a cold instruction cache, so its loops stay rolled: the code is
// small and each instruction is fetched once, then re-issued from the cache.
// ---------------------------------------------------------------------------

template <int E>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&v)[E], int lane) {
#pragma unroll 1
    for (int size = 2; size <= 32 * E; size <<= 1) {
        // strides >= E: the partner is register e of lane ^ stride/E; the
        // direction depends on the lane only
#pragma unroll 1
        for (int stride = size >> 1; stride >= E; stride >>= 1) {
            const bool lower = (lane & (stride / E)) == 0;
            const bool desc = (lane & (size / E)) == 0;
            const bool keep_max = (lower == desc);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint64_t p =
                    __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v[e]), stride / E);
                v[e] = ((v[e] > p) == keep_max) ? v[e] : p;
            }
        }
        // strides < E: both partners in this lane's registers
#pragma unroll
        for (int stride = E / 2; stride >= 1; stride >>= 1) {
            if (2 * stride <= size) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if ((e & stride) == 0) {
                        const bool desc = ((lane * E + e) & size) == 0;
                        const uint64_t x = v[e], y = v[e + stride];
                        if ((x < y) == desc) {
                            v[e] = y;
                            v[e + stride] = x;
                        }
                    }
                }
            }
        }
    }
}

// Sorts a[0 .. n) descending, n <= 256 * E; `runs` is scratch for n
// composites that must not overlap a.
template <int E>
__device__ __forceinline__ void block_merge_sort(uint64_t* a, int n, uint64_t* runs) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, tid = threadIdx.x;
    constexpr int R = 32 * E;
    {
        uint64_t v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = w * R + e * 32 + lane;   // any assignment will do: read conflict-free
            v[e] = i < n ? a[i] : 0ull;
        }
        warp_sort_desc<E>(v, lane);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int j = w * R + lane * E + e;
            if (j < n) runs[j] = v[e];
        }
    }
    // runs -> a -> runs -> a; a pair of runs of length L starts at 2 L p
    uint64_t* src = runs;
    uint64_t* dst = a;
#pragma unroll 1
    for (int L = R; L < 8 * R; L <<= 1) {
        __syncthreads();
        const int g0 = tid * E;                  // this thread's first output
        if (g0 < n) {
            const int base = g0 & ~(2 * L - 1);
            const int d = g0 - base;
            const uint64_t* A = src + base;
            const uint64_t* B = A + L;
            const int na = max(0, min(L, n - base)), nb = max(0, min(L, n - base - L));
            auto av = [&](int i) { return i < na ? A[i] : 0ull; };
            auto bv = [&](int j) { return j < nb ? B[j] : 0ull; };
            // i = outputs of [base, g0) that come from A (ties go to B first)
            int lo = max(0, d - L), hi = min(d, L);
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (av(mid) > bv(d - 1 - mid)) lo = mid + 1;
                else hi = mid;
            }
            int i = lo, j = d - lo;
            uint64_t x = av(i), y = bv(j);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (g0 + e >= n) break;
                const bool ta = j >= L || (i < L && x > y);
                dst[g0 + e] = ta ? x : y;
                if (ta) x = av(++i);
                else y = bv(++j);
            }
        }
        uint64_t* t = src;
        src = dst;
        dst = t;
    }
    __syncthreads();
}

// Sorts a[0 .. n) descending for n <= 256 * kMaxE (zero entries are padding
// and must not occur among the n); `runs`: scratch for n composites,
// disjoint from a.
template <int kMaxE>
__device__ __forceinline__ void block_sort_desc_r(uint64_t* a, int n, uint64_t* runs) {
    if (n <= 256) block_merge_sort<1>(a, n, runs);
    else if (n <= 512 || kMaxE < 4) block_merge_sort<(kMaxE < 2 ? kMaxE : 2)>(a, n, runs);
    else if (n <= 1024 || kMaxE < 8) block_merge_sort<(kMaxE < 4 ? kMaxE : 4)>(a, n, runs);
    else block_merge_sort<kMaxE>(a, n, runs);
}

// Sort by counting, for short lists: the position of a[i] is the number of
// larger entries (composites are unique).  P = 1, 2, 4 or 8 consecutive
// threads share an entry (the most that fit in the block): each compares it
// with its contiguous part of the list, two entries per 16-byte shared-memory
// load and eight per step into independent counts, and the P counts are added
// with shuffles.  Warps that hold no entry skip the comparisons.  n <= 256,
// all 256 threads; a 16-byte aligned with room for n + 1 entries; out must
// not overlap a.
__device__ __forceinline__ void block_count_sort(const uint64_t* a, int n, uint64_t* out) {
    const int t = threadIdx.x;
    {
        int lp = 0;   // log2 of the threads per entry
        while (lp < 3 && (n << (lp + 1)) <= kTopkThreads) ++lp;
        const int e = t >> lp, part = t & ((1 << lp) - 1);
        if (((t & ~31) >> lp) < n) {
            const uint64_t x = e < n ? a[e] : 0ull;
            const int len = (((n + (1 << lp) - 1) >> lp) + 1) & ~1;   // even: aligned pairs
            const int j1 = min(n, part * len + len);
            const uint4* a4 = reinterpret_cast<const uint4*>(a);
            int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
#pragma unroll 1
            for (int j = part * len; j < j1; j += 8) {
                uint64_t y[8];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int jj = j + 2 * u;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (jj < j1) v = a4[jj >> 1];
                    y[2 * u] = (static_cast<uint64_t>(v.y) << 32) | v.x;
                    y[2 * u + 1] = jj + 1 < j1 ? ((static_cast<uint64_t>(v.w) << 32) | v.z) : 0ull;
                }
                c0 += (y[0] > x) + (y[4] > x);
                c1 += (y[1] > x) + (y[5] > x);
                c2 += (y[2] > x) + (y[6] > x);
                c3 += (y[3] > x) + (y[7] > x);
            }
            int c = c0 + c1 + c2 + c3;
            for (int o = 1; o < (1 << lp); o <<= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (part == 0 && e < n) out[c] = x;
        }
    }
    __syncthreads();
}

// One out-of-line copy per kernel: the kernels sort from several places, each
// once per block and from a cold instruction cache, so sharing one copy keeps
// their code (and the instruction fetches) small.
static __device__ __noinline__ void block_sort_any(uint64_t* a, int n, uint64_t* runs) {
    block_sort_desc_r<8>(a, n, runs);
}

__device__ __forceinline__ int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Exact top-k of one candidate set whose 4096-bin histogram `hist` (shared)
// is exact for every candidate in the bins at and above the boundary.
// each(f) walks every candidate once (the fast walk, called at one place);
// each_slow(f) walks them again with compact code, only when the boundary bin
// overflows shared memory.  buf: shared buffer of cap >= 4096 composites:
// [0, 2048) collects the selection, the rest first the boundary bin, then the
// sort's scratch.  On return buf[0, nout) holds the winners in descending
// order (nout = min(k, candidates)).  All 256 threads.
template <class Each, class EachSlow>
__device__ int block_topk_sorted(Each each, EachSlow each_slow, const uint32_t* hist, int k, uint64_t* buf, int cap,
                                 SelectSmem* ss) {
    const int tid = threadIdx.x;
    block_find_suffix(hist, kHistBins, static_cast<uint32_t>(k), ss->scratch, &ss->bnd);
    const int bstar = ss->bnd.bin;
    const uint32_t above = ss->bnd.above;              // the total when bstar = -1
    const uint32_t count_ge = above + ss->bnd.at;      // candidates in bins >= bstar
    if (tid == 0) {
        ss->nsel = 0;
        ss->nbnd = 0;
    }
    __syncthreads();
    // bins above the boundary to buf, the boundary bin to bndbuf: two passes
    // without atomics (count per thread, scan, write at the scanned offsets).
    // A warp-aggregated atomic append measured ~2x slower here (its returned
    // offset puts a contended shared atomic in every iteration), and a
    // one-pass ballot append into per-warp segments no faster.
    uint64_t* bndbuf = buf + IDX_MAX_TOPK;
    const uint32_t bcap = static_cast<uint32_t>(cap - IDX_MAX_TOPK);
    {
        const int lane = tid & 31, warp = tid >> 5;
        uint32_t ca = 0, cb = 0;
        each([&](uint64_t c, bool v) {
            const int b = static_cast<int>(comp_key(c) >> kHistShift);
            ca += (v && b > bstar) ? 1u : 0u;
            cb += (v && b == bstar) ? 1u : 0u;
        });
        uint32_t ia = ca, ib = cb;   // inclusive scans over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t ya = __shfl_up_sync(0xffffffffu, ia, o), yb = __shfl_up_sync(0xffffffffu, ib, o);
            if (lane >= o) {
                ia += ya;
                ib += yb;
            }
        }
        if (lane == 31) {
            ss->scratch[warp] = ia;
            ss->scratch[8 + warp] = ib;
        }
        __syncthreads();
        uint32_t pa = ia - ca, pb = ib - cb;
#pragma unroll
        for (int w = 0; w < kTopkThreads / 32; ++w) {
            if (w < warp) {
                pa += ss->scratch[w];
                pb += ss->scratch[8 + w];
            }
        }
        each([&](uint64_t c, bool v) {
            const int b = static_cast<int>(comp_key(c) >> kHistShift);
            if (v && b > bstar) {
                if (pa < static_cast<uint32_t>(k)) buf[pa] = c;
                ++pa;
            } else if (v && b == bstar) {
                if (pb < bcap) bndbuf[pb] = c;
                ++pb;
            }
        });
        __syncthreads();
    }
    int nsort = static_cast<int>(above);   // composites to sort (the first k are output)
    if (bstar >= 0) {
        const uint32_t m = static_cast<uint32_t>(k) - above;   // needed from the boundary bin
        const uint32_t nb = ss->bnd.at;
        const uint32_t direct = static_cast<uint32_t>(max(kTopkThreads, next_pow2(k)));
        if (nb <= bcap && (nb == m || count_ge <= direct)) {
            // the whole boundary bin joins the sort
            for (uint32_t i = tid; i < nb; i += kTopkThreads) buf[above + i] = bndbuf[i];
            nsort = static_cast<int>(count_ge);
        } else {
            // refine the boundary bin to its m best by radix passes
            auto each_bnd = [&](auto f) { walk_smem(bndbuf, nb, f); };
            uint64_t thr;
            if (nb <= bcap) {
                thr = radix_refine(each_bnd, bstar, m, ss);
            } else {
                thr = radix_refine(each_slow, bstar, m, ss);
            }
            // the boundary bin's m best join the selection (two passes, no atomics)
            auto in = [&](uint64_t c) {
                return static_cast<int>(comp_key(c) >> kHistShift) == bstar && c >= thr;
            };
            const uint32_t room = static_cast<uint32_t>(k) - above;
            if (nb <= bcap) {
                block_collect(each_bnd, in, buf + above, room, ss->scratch);
            } else {
                block_collect(each_slow, in, buf + above, room, ss->scratch);
            }
            nsort = k;
        }
        __syncthreads();
    }
    block_sort_any(buf, nsort, bndbuf);
    return min(k, nsort);
}

// Physical pool slot of logical key s of a sequence (its block-table row
// bt_row of mbps entries, bs tokens per block): bt_row[s / bs] * bs + s % bs,
// the logical-to-physical translate (csa_translate_pack) of "DeepSeek-V4
// index_topk=1024 sparse indexer can't recall verbatim lines", section "How
// it was isolated".  -1 for s < 0 or a block past the row.
__device__ __forceinline__ int64_t slot_of(const int32_t* bt_row, int mbps, int bs, int32_t s) {
    if (s < 0) return -1;
    const int bi = s / bs;
    if (bi >= mbps) return -1;
    return static_cast<int64_t>(__ldg(bt_row + bi)) * bs + (s - bi * bs);
}

// Write a top-k row: buf[0, nout) as indices (and scores, and slots through
// the block-table row bt_row when out_slot is set), the rest of the k outputs
// as -1 (and -inf, -1).  nout < 0 writes a whole -1 row.  All threads.
__device__ __forceinline__ void write_topk_row(const uint64_t* buf, int nout, int k, int32_t* out_idx,
                                               float* out_score, int64_t* out_slot = nullptr,
                                               const int32_t* bt_row = nullptr, int mbps = 0, int bs = 1) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        if (j < nout) {
            const uint64_t c = buf[j];
            out_idx[j] = comp_index(c);
            if (out_score) out_score[j] = key_score(comp_key(c));
            if (out_slot) out_slot[j] = slot_of(bt_row, mbps, bs, comp_index(c));
        } else {
            out_idx[j] = -1;
            if (out_score) out_score[j] = -INFINITY;
            if (out_slot) out_slot[j] = -1;
        }
    }
}

}  // namespace dsaidx
