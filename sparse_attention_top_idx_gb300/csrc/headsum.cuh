// headsum.cuh -- the weighted ReLU head sum of the indexer score,
// sum_h w[t, h] * ReLU(q[t, h] . k[s]) ("The Hypothesis That Refused to Die",
// section "The Context"), over the 64 per-head dot products that the tensor
// cores left in TMEM for one query and the 32 keys of a warp's TMEM lane
// quadrant.  The decode and prefill kernels both call it, so a query scored
// alone (decode) and as a row of a causal chunk (prefill) gets bit-identical
// scores.
#pragma once

#include "common.cuh"

namespace dsaidx {

// The head weights a lane needs: with the .16x256b load shape lane t of a warp
// sees heads 8 i + 2 (t % 4) + {0, 1}, i = 0..7, of every row it holds.
__device__ __forceinline__ void load_head_weights(const float* w64, int lane, unsigned long long (&wr)[8]) {
    const float* w = w64 + 2 * (lane & 3);
#pragma unroll
    for (int i = 0; i < 8; ++i) wr[i] = *reinterpret_cast<const unsigned long long*>(w + 8 * i);
}

// The quadrant row whose sum head_sum_rows returns in lane t.
__device__ __forceinline__ int head_sum_row(int lane) { return 8 * (lane & 3) + (lane >> 2); }

// 2 * sum_h w'[h] * max(D[h], 0) for quadrant row head_sum_row(lane), where
// taddr addresses the quadrant's first lane and the query's first of 64 fp32
// columns.  The quadrant is read as two 16-lane slabs in four .16x256b.x4
// loads, each overlapping the arithmetic on the one before; lane t sums its
// 16 heads of rows r4 + {0, 8, 16, 24} (r4 = t / 4) in four independent
// packed accumulators (even and odd heads in the two halves), the max taken
// as D + |D| = 2 max(D, 0) exactly (an add with an absolute-value operand on
// the FMA pipe), then a two-step shuffle over the four lanes of a row group
// leaves each lane with one row's whole sum.  release() runs once every TMEM
// read has completed, before the last of the arithmetic.  Every lane of the
// warp must call it (aligned TMEM loads and full-warp shuffles).
template <class Release>
__device__ __forceinline__ float head_sum_rows(uint32_t taddr, const unsigned long long (&wr)[8], int lane,
                                               Release release) {
    auto accumulate = [&](const uint32_t (&v)[16], int wbase, unsigned long long& ra, unsigned long long& rb) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a0 = __uint_as_float(v[4 * i]), a1 = __uint_as_float(v[4 * i + 1]);
            const float b0 = __uint_as_float(v[4 * i + 2]), b1 = __uint_as_float(v[4 * i + 3]);
            ra = f2_fma(wr[wbase + i], f2_pack(a0 + fabsf(a0), a1 + fabsf(a1)), ra);
            rb = f2_fma(wr[wbase + i], f2_pack(b0 + fabsf(b0), b1 + fabsf(b1)), rb);
        }
    };
    constexpr uint32_t kSlab1 = 16u << 16;   // lane field + 16
    uint32_t v0[16], v1[16];
    unsigned long long r0 = 0ull, r1 = 0ull, r2 = 0ull, r3 = 0ull;   // rows r4, 8 + r4, 16 + r4, 24 + r4
    tmem_ld_16x256b_x4(taddr, v0);
    tmem_wait_ld16(v0);
    tmem_ld_16x256b_x4(taddr + 32, v1);
    accumulate(v0, 0, r0, r1);
    tmem_wait_ld16(v1);
    tmem_ld_16x256b_x4(taddr + kSlab1, v0);
    accumulate(v1, 4, r0, r1);
    tmem_wait_ld16(v0);
    tmem_ld_16x256b_x4(taddr + kSlab1 + 32, v1);
    accumulate(v0, 0, r2, r3);
    tmem_wait_ld16(v1);
    release();
    accumulate(v1, 4, r2, r3);
    const float2 p0 = f2_unpack(r0), p1 = f2_unpack(r1), p2 = f2_unpack(r2), p3 = f2_unpack(r3);
    const float s0 = p0.x + p0.y, s1 = p1.x + p1.y, s2 = p2.x + p2.y, s3 = p3.x + p3.y;
    // reduce-scatter over the four lanes (t % 4 = 0..3) of the row group
    const bool hi2 = (lane & 2) != 0;
    float k0 = hi2 ? s2 : s0, k1 = hi2 ? s3 : s1;
    k0 += __shfl_xor_sync(0xffffffffu, hi2 ? s0 : s2, 2);
    k1 += __shfl_xor_sync(0xffffffffu, hi2 ? s1 : s3, 2);
    const bool hi1 = (lane & 1) != 0;
    float k = hi1 ? k1 : k0;
    k += __shfl_xor_sync(0xffffffffu, hi1 ? k0 : k1, 1);
    return k;
}

}  // namespace dsaidx
