// topk.cuh -- block-level exact top-k machinery (256 threads per block).
//
// Every candidate is a 64-bit composite (score_key << 32) | ~index: the order
// of composites is "higher score first, then lower index", the tie rule of the
// library, and composites are unique within one query row.  Selection works on
// a 4096-bin histogram of the top 12 bits of score_key followed by exact radix
// refinement of the boundary bin, and finishes with a bitonic sort of the k
// winners.
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

// Warp-aggregated shared-memory histogram increment (one atomic per distinct
// bin in the warp).  Every lane of the warp must call it; `valid` masks lanes.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool valid) {
    unsigned active = __ballot_sync(0xffffffffu, valid);
    if (valid) {
        unsigned peers = __match_any_sync(active, bin);
        if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1))
            atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
    }
}

struct Boundary {
    int bin;          // largest bin whose suffix count reaches `need` (-1: total < need)
    uint32_t above;   // candidates in bins strictly above `bin` (the total when bin = -1)
    uint32_t at;      // candidates inside `bin` (0 when bin = -1)
};

// Find the bin holding the need-th largest candidate of a histogram of nbins
// (a multiple of 256) bins.  Called by all 256 threads; scratch holds >= 256
// words.  Result in *out (shared), valid after the call for every thread.
__device__ __forceinline__ void block_find_suffix(const uint32_t* hist, int nbins, uint32_t need,
                                  uint32_t* scratch, Boundary* out) {
    const int tid = threadIdx.x;
    const int per = nbins / kTopkThreads;
    uint32_t s = 0;
    for (int i = 0; i < per; ++i) s += hist[tid * per + i];
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

// Append c to buf (shared counter *cnt, capacity cap) for the lanes with
// `take`; one shared atomic per warp.  Every lane of the warp must call it.
// The counter still advances past cap, so callers can detect overflow.
__device__ __forceinline__ void warp_append(uint64_t* buf, uint32_t* cnt, uint32_t cap, uint64_t c,
                                            bool take) {
    const unsigned m = __ballot_sync(0xffffffffu, take);
    if (m == 0u) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(cnt, static_cast<uint32_t>(__popc(m)));
    base = __shfl_sync(0xffffffffu, base, leader);
    const uint32_t pos = base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
    if (take && pos < cap) buf[pos] = c;
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

// A global array of n composites, eight independent loads in flight per thread.
template <class F>
__device__ __forceinline__ void walk_global(const uint64_t* a, uint32_t n, F f) {
    constexpr uint32_t U = 8;
    const unsigned long long* p = reinterpret_cast<const unsigned long long*>(a);
    for (uint32_t b0 = 0; b0 < n; b0 += kTopkThreads * U) {
        unsigned long long v[U];
#pragma unroll
        for (uint32_t u = 0; u < U; ++u) {
            const uint32_t i = b0 + u * kTopkThreads + threadIdx.x;
            v[u] = (i < n) ? __ldcg(p + i) : 0ull;
        }
#pragma unroll
        for (uint32_t u = 0; u < U; ++u) {
            const uint32_t i = b0 + u * kTopkThreads + threadIdx.x;
            f(static_cast<uint64_t>(v[u]), i < n);
        }
    }
}

// A global row of n fp32 scores (16-byte aligned, readable up to n rounded up
// to 4): candidate i is (score_key(row[i]), i).  Eight float4 loads in flight.
template <class F>
__device__ __forceinline__ void walk_row(const float* row, int n, F f) {
    constexpr int U = 8;
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

// Exact refinement inside one bin: among the candidate set X (all composites
// whose top 12 bits equal `bin`), find the composite threshold thr such that
// exactly m members of X are >= thr.  `each` walks a superset of X (members
// outside X are filtered here).  Called by all 256 threads.
template <class Each>
__device__ uint64_t radix_refine(Each each, int bin, uint32_t m, SelectSmem* ss) {
    uint64_t prefix = static_cast<uint64_t>(bin) << 52;
    uint64_t mask = 0xFFFull << 52;
    uint32_t need = m;
    const int shifts[7] = {44, 36, 28, 20, 12, 4, 0};
    for (int pass = 0; pass < 7; ++pass) {
        const int sh = shifts[pass];
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

// In-place bitonic sort, descending, of n (power of two, <= 4096) composites.
__device__ __forceinline__ void bitonic_sort_desc(uint64_t* a, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n / 2; i += kTopkThreads) {
                int lo = 2 * i - (i & (stride - 1));
                int hi = lo + stride;
                bool desc = ((lo & size) == 0);
                uint64_t x = a[lo], y = a[hi];
                if ((x < y) == desc) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// Block sort, descending, of 256 * E composites held E per thread (thread t
// owns positions t*E .. t*E+E-1).  Bitonic network: compare-exchanges between
// a thread's own registers, then across lanes with warp shuffles, and through
// shared memory (two block barriers a stage) only for strides that cross
// warps: for 4096 keys, 6 of the 78 stages.
// ---------------------------------------------------------------------------
template <int E, int SIZE, int STRIDE>
__device__ __forceinline__ void bsort_stage(uint64_t (&v)[E], uint64_t* a) {
    const int t = threadIdx.x;
    if constexpr (STRIDE >= 32 * E) {
#pragma unroll
        for (int e = 0; e < E; ++e) a[t * E + e] = v[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = t * E + e;
            const uint64_t p = a[i ^ STRIDE];
            const bool keep_max = ((i & STRIDE) == 0) == ((i & SIZE) == 0);
            v[e] = keep_max ? (v[e] > p ? v[e] : p) : (v[e] < p ? v[e] : p);
        }
        __syncthreads();
    } else if constexpr (STRIDE >= E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = t * E + e;
            const uint64_t p = __shfl_xor_sync(0xffffffffu, static_cast<unsigned long long>(v[e]), STRIDE / E);
            const bool keep_max = ((i & STRIDE) == 0) == ((i & SIZE) == 0);
            v[e] = keep_max ? (v[e] > p ? v[e] : p) : (v[e] < p ? v[e] : p);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if ((e & STRIDE) == 0) {
                const bool desc = ((t * E + e) & SIZE) == 0;
                const uint64_t x = v[e], y = v[e + STRIDE];
                if ((x < y) == desc) {
                    v[e] = y;
                    v[e + STRIDE] = x;
                }
            }
        }
    }
}
template <int E, int SIZE, int STRIDE>
__device__ __forceinline__ void bsort_strides(uint64_t (&v)[E], uint64_t* a) {
    bsort_stage<E, SIZE, STRIDE>(v, a);
    if constexpr (STRIDE > 1) bsort_strides<E, SIZE, STRIDE / 2>(v, a);
}
template <int E, int SIZE>
__device__ __forceinline__ void bsort_sizes(uint64_t (&v)[E], uint64_t* a) {
    bsort_strides<E, SIZE, SIZE / 2>(v, a);
    if constexpr (SIZE < kTopkThreads * E) bsort_sizes<E, SIZE * 2>(v, a);
}
// Sorts a[0 .. 256*E) in place (shared memory), descending.  All 256 threads.
template <int E>
__device__ __forceinline__ void block_sort_desc(uint64_t* a) {
    uint64_t v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = a[threadIdx.x * E + e];
    bsort_sizes<E, 2>(v, a);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) a[threadIdx.x * E + e] = v[e];
    __syncthreads();
}
// Sorts a[0 .. n) descending for n <= 256 * kMaxE; entries up to the next
// size step (256, 512, ...) are overwritten with zero padding.
template <int kMaxE>
__device__ __forceinline__ void block_sort_desc_n(uint64_t* a, int n) {
    int n2 = kTopkThreads;
    while (n2 < n) n2 <<= 1;
    for (int i = n + static_cast<int>(threadIdx.x); i < n2; i += kTopkThreads) a[i] = 0ull;
    __syncthreads();
    if (n2 <= 256) block_sort_desc<1>(a);
    else if (n2 <= 512) block_sort_desc<2>(a);
    else if (n2 <= 1024) block_sort_desc<4>(a);
    else if (kMaxE <= 8 || n2 <= 2048) block_sort_desc<(kMaxE < 8 ? kMaxE : 8)>(a);
    else block_sort_desc<kMaxE>(a);
}

__device__ __forceinline__ int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Final selection of one query row from a candidate set whose 4096-bin
// histogram `hist` (shared) is exact.  `each` walks every candidate.  buf:
// shared buffer of cap >= 2048 + (boundary room) composites; up to 256 * kMaxE
// candidates at or above the boundary bin are selected by one sort.  Writes the k outputs (descending,
// -1 / -inf padded).  Called by all 256 threads.
template <int kMaxE, class Each>
__device__ void select_topk_from_hist(Each each, const uint32_t* hist, int k, uint64_t* buf, int cap,
                                      SelectSmem* ss, int32_t* out_idx, float* out_score) {
    const int tid = threadIdx.x;
    block_find_suffix(hist, kHistBins, static_cast<uint32_t>(k), ss->scratch, &ss->bnd);
    const int bstar = ss->bnd.bin;
    const uint32_t above = ss->bnd.above;
    const uint32_t count_ge = above + ss->bnd.at;     // candidates in bins >= bstar
    if (tid == 0) {
        ss->nsel = 0;
        ss->nbnd = 0;
    }
    __syncthreads();
    const uint32_t sortcap = static_cast<uint32_t>(min(cap, kTopkThreads * kMaxE));
    // sort everything at or above the boundary bin when that is no bigger a
    // sort than the k winners need; otherwise refine the boundary bin first
    const uint32_t direct = static_cast<uint32_t>(max(kTopkThreads, next_pow2(k)));
    if (count_ge <= sortcap && count_ge <= direct) {
        // common case: everything at or above the boundary bin fits; one sort
        each([&](uint64_t c, bool v) {
            warp_append(buf, &ss->nsel, sortcap, c, v && static_cast<int>(comp_key(c) >> kHistShift) >= bstar);
        });
        __syncthreads();
        block_sort_desc_n<kMaxE>(buf, static_cast<int>(count_ge));
        const int nsel = min(k, static_cast<int>(count_ge));
        for (int j = tid; j < k; j += kTopkThreads) {
            if (j < nsel) {
                const uint64_t c = buf[j];
                out_idx[j] = comp_index(c);
                if (out_score) out_score[j] = key_score(comp_key(c));
            } else {
                out_idx[j] = -1;
                if (out_score) out_score[j] = -INFINITY;
            }
        }
        return;
    }
    // many candidates share the boundary bin: refine it by radix passes
    uint64_t* sel = buf;
    uint64_t* bndbuf = buf + IDX_MAX_TOPK;
    const int bcap = cap - IDX_MAX_TOPK;
    // gather: bins above the boundary go straight to sel, the boundary bin to bndbuf
    each([&](uint64_t c, bool v) {
        const int b = static_cast<int>(comp_key(c) >> kHistShift);
        warp_append(sel, &ss->nsel, static_cast<uint32_t>(k), c, v && b > bstar);
        warp_append(bndbuf, &ss->nbnd, static_cast<uint32_t>(bcap), c, v && b == bstar);
    });
    __syncthreads();
    if (bstar >= 0) {
        const uint32_t m = static_cast<uint32_t>(k) - above;
        const uint32_t nb = ss->nbnd;
        const bool fits = nb <= static_cast<uint32_t>(bcap);
        if (fits && nb == m) {
            for (uint32_t i = tid; i < nb; i += kTopkThreads) sel[above + i] = bndbuf[i];
        } else {
            auto each_bnd = [&](auto f) { walk_smem(bndbuf, nb, f); };
            const uint64_t thr = fits ? radix_refine(each_bnd, bstar, m, ss) : radix_refine(each, bstar, m, ss);
            if (tid == 0) ss->nsel = above;
            __syncthreads();
            auto take = [&](uint64_t c, bool v) {
                const bool in = v && static_cast<int>(comp_key(c) >> kHistShift) == bstar && c >= thr;
                warp_append(sel, &ss->nsel, static_cast<uint32_t>(k), c, in);
            };
            if (fits) each_bnd(take);
            else each(take);
        }
        __syncthreads();
    }
    const int nsel = (bstar >= 0) ? k : static_cast<int>(above);
    block_sort_desc_n<8>(sel, nsel);
    for (int j = tid; j < k; j += kTopkThreads) {
        if (j < nsel) {
            uint64_t c = sel[j];
            out_idx[j] = comp_index(c);
            if (out_score) out_score[j] = key_score(comp_key(c));
        } else {
            out_idx[j] = -1;
            if (out_score) out_score[j] = -INFINITY;
        }
    }
}

}  // namespace dsaidx
