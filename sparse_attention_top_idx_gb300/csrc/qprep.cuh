// qprep.cuh -- query preparation for the scoring kernels: the bf16 query rows
// of a work unit, staged in shared memory, become the B operand of the
// tcgen05 contraction (K-major, 128-byte swizzle) and the head weights w'.
//
// fp8 keys: every (query, head) row is quantised like a key -- scale
// sq = amax / 448 (IEEE division), codes e4m3(q / sq) rounded to nearest even
// with saturation -- and its scale is folded into the head weight,
// w' = w * sq, so that sum_h w' * ReLU(qcode . kcode) * kscale is the score of
// "The Hypothesis That Refused to Die" (section "The Context") on the
// quantised operands.  bf16 keys: the query bytes are used as they are.
#pragma once

#include "common.cuh"

namespace dsaidx {

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

// Half h (0 or 1: elements 64 h .. 64 h + 63) of query row r (bf16, staged in
// shared memory) turned into its B-tile bytes in qtile (a tile of `rows`
// rows), by two adjacent lanes (lane ^ 1 holds the other half; mask pm has
// both).  fp8: the row's amax is reduced over the pair, sq = amax / 448 (IEEE),
// codes e4m3(q / sq) correctly rounded (chunks 4 h .. 4 h + 3 of the swizzled
// row), w' = w * sq; amax = 0 gives zero codes.  bf16: the 128 bytes go to
// K-half h of the tile, w' = w.  Returns w'.
//
// The lanes of a warp hold half rows 128 bytes apart, so reading their
// 16-byte chunks in the same order would put all 32 lanes on the same four
// banks; each lane starts at a different chunk (`rot`) instead.  The half row
// is read twice (amax, then 16 elements at a time) so that few values are
// live at once.
template <bool kFp8>
__device__ __forceinline__ float quant_row_half(const uint8_t* raw_row, int h, float wv, unsigned pm,
                                                uint8_t* qtile, int r, int rows) {
    const uint4* src = reinterpret_cast<const uint4*>(raw_row + h * 128);
    const int rot = static_cast<int>(threadIdx.x);
    if constexpr (!kFp8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = (i + rot) & 7;
            *reinterpret_cast<uint4*>(qtile + h * (rows * 128) + sw128_off(r, c)) = src[c];
        }
        return wv;
    } else {
        // bf16 magnitude bits compare like the values: the largest |x| is the
        // largest (bits & 0x7FFF), converted once
        uint32_t mbits = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 v = src[(i + rot) & 7];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) mbits = max(mbits, max(w4[e] & 0x7FFFu, (w4[e] >> 16) & 0x7FFFu));
        }
        mbits = max(mbits, __shfl_xor_sync(pm, mbits, 1));
        const float amax = __uint_as_float(mbits << 16);
        const float sq = __fdiv_rn(amax, 448.0f);
        const DivBy div(sq);
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
            const int c = (i + (rot >> 1)) & 3;   // output chunk: input chunks 2 c and 2 c + 1
            // the two lanes of a row take the chunk pair in opposite orders
            const int first = 2 * c + (rot & 1);
            const uint4 va = src[first], vb = src[first ^ 1];
            const uint4 v0 = (rot & 1) ? vb : va, v1 = (rot & 1) ? va : vb;
            const uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (amax != 0.0f) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t wlo = w8[2 * j], whi = w8[2 * j + 1];
                    const float x0 = __uint_as_float(wlo << 16), x1 = __uint_as_float(wlo & 0xFFFF0000u);
                    const float x2 = __uint_as_float(whi << 16), x3 = __uint_as_float(whi & 0xFFFF0000u);
                    o[j] = cvt_e4m3x2_pair(div(x0), div(x1)) | (cvt_e4m3x2_pair(div(x2), div(x3)) << 16);
                }
            }
            *reinterpret_cast<uint4*>(qtile + sw128_off(r, 4 * h + c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
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

}  // namespace dsaidx
