// prefill.cu -- causal-chunk scoring (tcgen05 kernel with 4 queries per CTA,
// scores to the workspace) followed by the per-row exact top-k select.
#include "prefill_kernel.cuh"

namespace dsaidx {

namespace {

constexpr int kSelBcap = 4096;

struct SelectPlan {
    int hist_off, sel_off, bnd_off, ss_off, total;
};
__host__ __device__ inline SelectPlan select_plan() {
    SelectPlan s{};
    s.hist_off = 0;
    s.sel_off = s.hist_off + kHistBins * 4;
    s.bnd_off = s.sel_off + IDX_MAX_TOPK * 8;
    s.ss_off = s.bnd_off + kSelBcap * 8;
    s.total = s.ss_off + static_cast<int>(align_up(sizeof(SelectSmem), 16)) + 64;
    return s;
}

// One CTA per query row: histogram of the row's visible scores, then the exact
// selection (the per-row top-k of ROCm/ATOM issue #1507, section "How it was
// isolated", applied to the causal rows of _score_topk_prefill).
__global__ void __launch_bounds__(kTopkThreads, 3) prefill_select_kernel(const ScoreParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const SelectPlan sp = select_plan();
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + sp.hist_off);
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem + sp.sel_off);
    SelectSmem* ss = reinterpret_cast<SelectSmem*>(smem + sp.ss_off);
    __shared__ int s_nvis, s_bad, s_b;
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    if (tid == 0) {
        int lo = 0, hi = p.batch - 1;   // largest b with cu_q[b] <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu_q[mid] <= r) lo = mid;
            else hi = mid - 1;
        }
        const int b = lo;
        const int S = p.seq_lens[b];
        const int nq = p.cu_q[b + 1] - p.cu_q[b];
        const int pos = S - nq + (r - p.cu_q[b]);
        const bool flagged = p.rowflag[r] != 0;
        const bool invalid = S > p.max_seq_len || nq > S || r >= p.cu_q[b + 1] || pos < 0;
        if (invalid) set_status(p.status, IDX_ERR_DEVICE_CHECK);
        if (flagged) p.rowflag[r] = 0;
        s_bad = flagged || invalid;
        s_nvis = pos + 1;
        s_b = b;
    }
    for (int i = tid; i < kHistBins; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    int32_t* oi = p.out_idx + static_cast<int64_t>(r) * p.topk;
    float* os = p.out_score ? p.out_score + static_cast<int64_t>(r) * p.topk : nullptr;
    int64_t* osl = p.out_slot ? p.out_slot + static_cast<int64_t>(r) * p.topk : nullptr;
    if (s_bad) {
        for (int j = tid; j < p.topk; j += kTopkThreads) {
            oi[j] = -1;
            if (os) os[j] = -INFINITY;
            if (osl) osl[j] = -1;
        }
        return;
    }
    const int nvis = s_nvis;
    const float* row = p.scores + static_cast<int64_t>(r) * p.score_stride;
    auto each = [&](auto f) { walk_row(row, nvis, f); };
    each([&](uint64_t c, bool v) { hist_add_warp(hist, key_bin(comp_key(c)), v); });
    __syncthreads();
    auto each_slow = [&](auto f) { walk_row_slow(row, nvis, f); };
    const int nout = block_topk_sorted(each, each_slow, hist, p.topk, sel, IDX_MAX_TOPK + kSelBcap, ss);
    write_topk_row(sel, nout, p.topk, oi, os, osl, p.block_table + static_cast<int64_t>(s_b) * p.mbps, p.mbps,
                   p.block_size);
}

template <bool kFp8, int kBs>
cudaError_t launch_prefill_t(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_done{0};
    static std::atomic<unsigned long long> sel_attr_done{0};
    const SmemPlan plan = make_plan(kFp8, kPrefillQT, 0);
    auto kern = prefill_score_kernel<kFp8, kBs>;
    cudaError_t e = set_smem_once(kern, plan.total, attr_done);
    if (e != cudaSuccess) return e;
    if (p.num_groups > 0) {
        kt_mark(st);
        kern<<<p.num_groups, kPrefillThreads, plan.total, st>>>(c->tmap, p);
        kt_mark(st);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const SelectPlan sp = select_plan();
    e = set_smem_once(prefill_select_kernel, sp.total, sel_attr_done);
    if (e != cudaSuccess) return e;
    kt_mark(st);
    prefill_select_kernel<<<p.total_q, kTopkThreads, sp.total, st>>>(p);
    kt_mark(st);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const idx_cache* c, const ScoreParams& p, cudaStream_t st) {
    const bool fp8 = c->key_dtype == IDX_KEY_FP8_E4M3;
    if (fp8 && c->block_size == 64) return launch_prefill_t<true, 64>(c, p, st);
    if (fp8 && c->block_size == 32) return launch_prefill_t<true, 32>(c, p, st);
    if (!fp8 && c->block_size == 64) return launch_prefill_t<false, 64>(c, p, st);
    return launch_prefill_t<false, 32>(c, p, st);
}

}  // namespace dsaidx
