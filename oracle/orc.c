/*
 * orc.c -- CPU oracle for the DSA lightning-indexer path (key store, score,
 * causal mask, top-k).  TEST INFRASTRUCTURE ONLY: nothing on the product path
 * may link, load or call this file.  It shares no code, header, table or
 * constant generator with the CUDA library; the two meet only in the tests.
 *
 * Plain, slow and written to be read against its sources:
 *
 *  - "DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
 *    (ROCm/ATOM issue #1507), section "How it was isolated": the index keys
 *    are quantised to fp8 with a per-token scale and scattered into a paged
 *    cache (indexer_k_quant_and_cache), the paged logits are computed per
 *    query over the cache (fp8 paged MQA logits) and the best index_topk
 *    positions are kept per row (top_k_per_row_decode); the block sizes are
 *    32 and 64.
 *  - "The Pivot: A Single Edit That Finally Fixed DeepSeek V4's Long-Context
 *    Recall Failure", section "Assumptions and Input Knowledge": an index-key
 *    record is 132 bytes per token in fp8 (128 one-byte codes plus a 4-byte
 *    fp32 scale) and 256 bytes per token in bf16.
 *  - "The Hypothesis That Refused to Die", section "The Context": the indexer
 *    scores every cached position with a compressed query-key dot product and
 *    keeps the top K (512 there).  The score used here is
 *        score[t,s] = sum_h w[t,h] * ReLU(q[t,h] . k[s])   (fp32 accumulation)
 *    with the per-head weights w given as an input (the weights projection
 *    and softmax scaling the same page lists under "The Bash Command" are the
 *    caller's business and arrive folded into w).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes): per-token key scale = fl32(amax / 448); codes = e4m3 round-to-
 * nearest-even with saturation of fl32(x / scale); amax == 0 gives scale 0 and
 * all-zero codes; the query is quantised the same way per (t, h) row and its
 * scale sq is folded into the head weight, w' = fl32(w * sq); a query at
 * position pos sees keys s <= pos; ties in score go to the lower index; the
 * top-k is listed in descending score order and padded with -1.  The fp4
 * round trip (below) keeps fl32(amax / 6) per block of 32 as the scale, rounds
 * fl32(x / scale) to the nearest e2m1 value (ties to the even code,
 * saturating at 6) and hands on fl32(code * scale) in fp32.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared [-fopenmp] orc.c -o liborc.so
 * (-ffp-contract=off keeps every multiply and add separately rounded, so x86
 * and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_E4M3_MAX 448.0

/* ------------------------------------------------------------------------ */
/* bf16 and fp32 bit helpers                                                 */
/* ------------------------------------------------------------------------ */

/* A bf16 value is the top half of an fp32 bit pattern. */
/* Largest row length the per-row helpers take (the index keys have d = 128). */
#define ORC_MAX_D 1024

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ------------------------------------------------------------------------ */
/* fp8 e4m3 ("e4m3fn" in the OCP 8-bit floating point specification):       */
/* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,  */
/* S.1111.111 is NaN, largest finite magnitude 448, subnormal step 2^-9.     */
/* ------------------------------------------------------------------------ */

/* Value of an e4m3 code, from the format definition. */
float orc_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* m/8 * 2^(1-7) */
    else
        v = ldexp(8.0 + (double)m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
    return (float)(sign ? -v : v);
}

/* Round-half-even of a non-negative double that holds an exact dyadic value. */
static double orc_round_half_even(double n)
{
    double f = floor(n);
    double r = n - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/*
 * Encode an fp32 value to e4m3, round to nearest with ties to even, finite
 * values beyond the largest magnitude saturating to +-448 (the "satfinite"
 * conversion), NaN to 0x7F.  The sign is kept, so -0 and negative values that
 * round to zero give 0x80.
 */
uint8_t orc_e4m3_encode(float x)
{
    uint32_t bits;
    uint8_t sign;
    double a, q, n, v;
    int e;
    memcpy(&bits, &x, 4);
    sign = (bits >> 31) ? 0x80 : 0x00;
    if (isnan(x))
        return 0x7F;
    a = fabs((double)x);
    if (a >= ORC_E4M3_MAX)
        return (uint8_t)(sign | 0x7E);
    /* Spacing of the e4m3 grid around a: 2^-9 below 2^-6 (subnormals),
       otherwise 2^(floor(log2 a) - 3).  Both scalings below are exact. */
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1) */
        q = ldexp(1.0, (e - 1) - 3);
    }
    n = orc_round_half_even(a / q);
    v = n * q;
    if (v > ORC_E4M3_MAX)
        v = ORC_E4M3_MAX;
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, -9))); /* subnormal */
    (void)frexp(v, &e);
    {
        int ef = (e - 1) + 7;                                      /* biased */
        int m = (int)(ldexp(v, -(e - 1)) * 8.0) - 8;               /* 0..7 */
        return (uint8_t)(sign | (ef << 3) | m);
    }
}

/* Encode n floats (used by the tests to pin the encoder). */
void orc_e4m3_encode_n(const float* x, uint8_t* out, int64_t n)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_n(const uint8_t* c, float* out, int64_t n)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = orc_e4m3_decode(c[i]);
}

/*
 * Per-row fp8 quantisation of d float values: amax over the row, scale =
 * fl32(amax / 448), code_i = e4m3(fl32(x_i / scale)).  A zero row gets scale
 * 0 and zero codes.
 */
void orc_quant_row_f32(const float* x, int d, uint8_t* codes, float* scale_out)
{
    float amax = 0.0f, scale;
    int i;
    for (i = 0; i < d; i++) {
        float v = fabsf(x[i]);
        if (v > amax)
            amax = v;
    }
    scale = amax / 448.0f;
    *scale_out = scale;
    for (i = 0; i < d; i++) {
        if (amax == 0.0f) {
            codes[i] = 0x00;
        } else {
            float y = x[i] / scale;
            codes[i] = orc_e4m3_encode(y);
        }
    }
}

/* The same for a row of bf16 values (each exactly a float). */
void orc_quant_row(const uint16_t* x_bf16, int d, uint8_t* codes, float* scale_out)
{
    float x[ORC_MAX_D];
    int i;
    for (i = 0; i < d && i < ORC_MAX_D; i++)
        x[i] = orc_bf16_to_f32(x_bf16[i]);
    orc_quant_row_f32(x, d < ORC_MAX_D ? d : ORC_MAX_D, codes, scale_out);
}

void orc_quant_rows_f32(const float* x, int64_t rows, int d, uint8_t* codes, float* scales)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; r++)
        orc_quant_row_f32(x + r * d, d, codes + r * d, scales + r);
}

/* float -> bf16 bits, round to nearest even (finite inputs). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u = u + 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

void orc_f32_to_bf16_n(const float* x, uint16_t* out, int64_t n)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = orc_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard rotation of an index key                                   */
/* ------------------------------------------------------------------------ */

/* 1 when v has an odd number of set bits. */
static int orc_odd_parity(unsigned v)
{
    int p = 0;
    while (v) {
        p ^= (int)(v & 1u);
        v >>= 1;
    }
    return p;
}

/*
 * y = H x for one row of d bf16 values (d a power of two), H the orthonormal
 * Walsh-Hadamard matrix in Sylvester order, H[i][j] = (-1)^popcount(i & j) /
 * sqrt(d): the rotation that "DeepSeek-V4 index_topk=1024 sparse indexer
 * can't recall verbatim lines" (ROCm/ATOM issue #1507), section "Root cause",
 * says the index query gets and the index key must get too (its fix (B) puts
 * it on the key store path); H is orthogonal, so (Hq).(Hk) = q.k.  The +-1
 * sum is taken in double (exact for a row whose exponents span at most 38
 * binades), multiplied by the double nearest 1/sqrt(d) and rounded once to
 * float.
 */
void orc_wht_row(const uint16_t* x_bf16, int d, float* y)
{
    const double c = 1.0 / sqrt((double)d);
    int i, j;
    for (i = 0; i < d; i++) {
        double s = 0.0;
        for (j = 0; j < d; j++) {
            double v = (double)orc_bf16_to_f32(x_bf16[j]);
            s += orc_odd_parity((unsigned)(i & j)) ? -v : v;
        }
        y[i] = (float)(s * c);
    }
}

void orc_wht_rows(const uint16_t* x_bf16, int64_t rows, int d, float* y)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; r++)
        orc_wht_row(x_bf16 + r * d, d, y + r * d);
}

void orc_quant_rows(const uint16_t* x_bf16, int64_t rows, int d, uint8_t* codes, float* scales)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; r++)
        orc_quant_row(x_bf16 + r * d, d, codes + r * d, scales + r);
}

/* ------------------------------------------------------------------------ */
/* fp4 (e2m1) round trip of an index key in blocks of 32                     */
/* ------------------------------------------------------------------------ */

/*
 * The 4-bit float e2m1 (1 sign, 2 exponent and 1 mantissa bit, no infinities
 * or NaN): code c = 0..7 has magnitude orc_e2m1_mag[c] (0 and 0.5 are the
 * zero and the subnormal, then 1, 1.5, 2, 3, 4, 6), bit 3 is the sign.
 */
static const double orc_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/*
 * Encode a finite fp32 value to e2m1: the code whose magnitude is nearest to
 * |x| (found by trying all eight), a tie between two neighbours going to the
 * even code (low bit 0); magnitudes from 6 up saturate to 6 (taken before the
 * search: far above 6 the double distances to 4 and 6 round to one value).
 * The sign bit is kept, so -0 and negative values that round to zero give 0x8.
 */
uint8_t orc_e2m1_encode(float x)
{
    double a = fabs((double)x);
    int c, best = 0;
    double bd = a;
    if (a >= orc_e2m1_mag[7])
        return (uint8_t)((signbit(x) ? 8 : 0) | 7);
    for (c = 1; c < 8; c++) {
        double dist = fabs(a - orc_e2m1_mag[c]);
        if (dist < bd || (dist == bd && (c & 1) == 0)) {
            best = c;
            bd = dist;
        }
    }
    return (uint8_t)((signbit(x) ? 8 : 0) | best);
}

double orc_e2m1_decode(uint8_t c)
{
    double m = orc_e2m1_mag[c & 7];
    return (c & 8) ? -m : m;
}

void orc_e2m1_encode_n(const float* x, uint8_t* out, int64_t n)
{
    int64_t i;
    for (i = 0; i < n; i++)
        out[i] = orc_e2m1_encode(x[i]);
}

/*
 * The fp4 round trip that "DeepSeek-V4 index_topk=1024 sparse indexer can't
 * recall verbatim lines" (ROCm/ATOM issue #1507), section "Where (main
 * 0c7d50f9)", lists on the indexer's key path after the rotation
 * (fp4_act_quant_inplace(kv, 32), the fp4 quantisation-aware round trip):
 * every block of ORC_FP4_BLOCK = 32 consecutive values gets its own scale
 * s = fl32(amax / 6) (6 is the largest e2m1 magnitude),
 * each value x becomes the e2m1 code of fl32(x / s) and is replaced by
 * fl32(code * s), the decoded value.  A block whose values are all zero keeps
 * them.  d must be a multiple of 32; the output stays in fp32.
 */
#define ORC_FP4_BLOCK 32

void orc_fp4_roundtrip_row(const float* x, int d, float* y)
{
    int b, j;
    for (b = 0; b < d; b += ORC_FP4_BLOCK) {
        float amax = 0.0f, s;
        for (j = 0; j < ORC_FP4_BLOCK; j++) {
            float a = fabsf(x[b + j]);
            if (a > amax)
                amax = a;
        }
        if (amax == 0.0f) {
            for (j = 0; j < ORC_FP4_BLOCK; j++)
                y[b + j] = x[b + j];
            continue;
        }
        s = amax / 6.0f;
        for (j = 0; j < ORC_FP4_BLOCK; j++) {
            float v = x[b + j] / s;
            y[b + j] = (float)(orc_e2m1_decode(orc_e2m1_encode(v)) * (double)s);
        }
    }
}

void orc_fp4_roundtrip_rows(const float* x, int64_t rows, int d, float* y)
{
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; r++)
        orc_fp4_roundtrip_row(x + r * d, d, y + r * d);
}

/* ------------------------------------------------------------------------ */
/* Paged index-key cache                                                     */
/* ------------------------------------------------------------------------ */

/* Key dtypes: 0 = fp8 e4m3 + fp32 scale (132 B/token at d=128), 1 = bf16. */
#define ORC_FP8 0
#define ORC_BF16 1

/*
 * One block of bs tokens.  fp8: bs rows of d one-byte codes, then bs fp32
 * scales.  bf16: bs rows of d bf16 values.
 */
int64_t orc_block_bytes(int dtype, int bs, int d)
{
    if (dtype == ORC_FP8)
        return (int64_t)bs * d + (int64_t)bs * 4;
    return (int64_t)bs * d * 2;
}

/*
 * Write n keys into the pool: token i goes to slot slot_mapping[i] =
 * block * bs + offset; a negative slot is skipped.  mode bit 0 (rotate): each
 * key is first Walsh-Hadamard rotated (orc_wht_row); mode bit 1 (fp4): the
 * float row then takes the fp4 round trip (orc_fp4_roundtrip_row).  With
 * either, the float result is what is quantised (fp8) or rounded to bf16.
 * Returns the number of tokens written, or -1 if a slot is out of range (-2
 * for d > ORC_MAX_D or, with fp4, d not a multiple of 32).
 */
int64_t orc_store_keys_any(uint8_t* pool, int64_t num_blocks, int bs, int d, int dtype,
                           const uint16_t* k_bf16, const int64_t* slot_mapping, int64_t n, int mode)
{
    int64_t i, written = 0;
    int64_t bb = orc_block_bytes(dtype, bs, d);
    float y[ORC_MAX_D], t[ORC_MAX_D];
    int j;
    const int rotate = mode & 1, fp4 = (mode >> 1) & 1, fl = rotate || fp4;
    if (d > ORC_MAX_D || (fp4 && d % ORC_FP4_BLOCK != 0))
        return -2;
    for (i = 0; i < n; i++) {
        int64_t slot = slot_mapping[i];
        int64_t blk, off;
        uint8_t* base;
        if (slot < 0)
            continue;
        blk = slot / bs;
        off = slot % bs;
        if (blk >= num_blocks)
            return -1;
        base = pool + blk * bb;
        if (rotate)
            orc_wht_row(k_bf16 + i * d, d, y);
        else if (fp4)
            for (j = 0; j < d; j++)
                y[j] = orc_bf16_to_f32(k_bf16[i * d + j]);
        if (fp4) {
            orc_fp4_roundtrip_row(y, d, t);
            memcpy(y, t, (size_t)d * sizeof(float));
        }
        if (dtype == ORC_FP8) {
            float sc;
            if (fl)
                orc_quant_row_f32(y, d, base + off * d, &sc);
            else
                orc_quant_row(k_bf16 + i * d, d, base + off * d, &sc);
            memcpy(base + (int64_t)bs * d + off * 4, &sc, 4);
        } else if (fl) {
            for (j = 0; j < d; j++) {
                uint16_t b = orc_f32_to_bf16(y[j]);
                memcpy(base + off * d * 2 + (int64_t)j * 2, &b, 2);
            }
        } else {
            memcpy(base + off * d * 2, k_bf16 + i * d, (size_t)d * 2);
        }
        written++;
    }
    return written;
}

int64_t orc_store_keys(uint8_t* pool, int64_t num_blocks, int bs, int d, int dtype,
                       const uint16_t* k_bf16, const int64_t* slot_mapping, int64_t n)
{
    return orc_store_keys_any(pool, num_blocks, bs, d, dtype, k_bf16, slot_mapping, n, 0);
}

/*
 * Logical-to-physical translate of selected key indices (csa_translate_pack
 * in "DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim
 * lines", ROCm/ATOM issue #1507, section "How it was isolated"): index s of a
 * sequence whose block-table row has mbps entries becomes the pool slot
 * table_row[s / bs] * bs + s % bs; a negative index or a block past the row
 * becomes -1.
 */
void orc_translate_slots(const int32_t* table_row, int64_t mbps, int bs, const int32_t* idx, int64_t n,
                         int64_t* out)
{
    int64_t i;
    for (i = 0; i < n; i++) {
        int64_t s = idx[i];
        if (s < 0 || s / bs >= mbps)
            out[i] = -1;
        else
            out[i] = (int64_t)table_row[s / bs] * bs + s % bs;
    }
}

/*
 * Read logical key s of a sequence back out of the pool through its block
 * table row (block = table[s / bs], offset = s % bs).  fp8: codes + scale.
 * bf16: the d raw values.
 */
void orc_gather_keys(const uint8_t* pool, int bs, int d, int dtype, const int32_t* table_row,
                     int64_t S, uint8_t* codes_out, float* scales_out, uint16_t* bf16_out)
{
    int64_t s, bb = orc_block_bytes(dtype, bs, d);
    for (s = 0; s < S; s++) {
        const uint8_t* base = pool + (int64_t)table_row[s / bs] * bb;
        int64_t off = s % bs;
        if (dtype == ORC_FP8) {
            memcpy(codes_out + s * d, base + off * d, (size_t)d);
            memcpy(scales_out + s, base + (int64_t)bs * d + off * 4, 4);
        } else {
            memcpy(bf16_out + s * d, base + off * d * 2, (size_t)d * 2);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Scores                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * Scores of one query row against keys 0..nvis-1 of its sequence.
 *
 * fp8 keys: the query row of each head is quantised like a key (codes qc,
 * scale sq), w'[h] = fl32(w[h] * sq[h]), dot = sum_d qc*kc in fp32 with d
 * ascending, score = fl32(ks[s] * sum_h fl32(w'[h] * max(dot, 0))), h ascending.
 * bf16 keys: dot = sum_d q*k in fp32 over the bf16 values, score =
 * sum_h fl32(w[h] * max(dot, 0)).
 *
 * q: [H, d] bf16 bits.  w: [H].  kc/ks (fp8) or kb (bf16) are the logical keys.
 * exact_out (optional): the same quantity with every dot product and the head
 * sum evaluated in fp64 (exact for the fp8 code products), used to bound the
 * rounding of the fp32 loop.
 */
void orc_scores_row(int dtype, int d, int H, const uint16_t* q, const float* w, int64_t nvis,
                    const uint8_t* kc, const float* ks, const uint16_t* kb,
                    float* out, double* exact_out)
{
    int64_t s;
    int h, i;
    float* qf = (float*)malloc(sizeof(float) * (size_t)H * d);
    float* wq = (float*)malloc(sizeof(float) * (size_t)H);
    float* kf = (float*)malloc(sizeof(float) * (size_t)d);
    if (dtype == ORC_FP8) {
        uint8_t* qc = (uint8_t*)malloc((size_t)d);
        for (h = 0; h < H; h++) {
            float sq;
            orc_quant_row(q + (int64_t)h * d, d, qc, &sq);
            for (i = 0; i < d; i++)
                qf[h * d + i] = orc_e4m3_decode(qc[i]);
            wq[h] = w[h] * sq;
        }
        free(qc);
    } else {
        for (h = 0; h < H; h++) {
            for (i = 0; i < d; i++)
                qf[h * d + i] = orc_bf16_to_f32(q[(int64_t)h * d + i]);
            wq[h] = w[h];
        }
    }
    for (s = 0; s < nvis; s++) {
        float acc = 0.0f;
        double acc_x = 0.0;
        for (i = 0; i < d; i++)
            kf[i] = (dtype == ORC_FP8) ? orc_e4m3_decode(kc[s * d + i])
                                       : orc_bf16_to_f32(kb[s * d + i]);
        for (h = 0; h < H; h++) {
            float dot = 0.0f;
            double dot_x = 0.0;
            for (i = 0; i < d; i++) {
                float p = qf[h * d + i] * kf[i];
                dot = dot + p;
                dot_x += (double)qf[h * d + i] * (double)kf[i];
            }
            {
                float r = dot > 0.0f ? dot : 0.0f;
                float t = wq[h] * r;
                acc = acc + t;
            }
            acc_x += (double)wq[h] * (dot_x > 0.0 ? dot_x : 0.0);
        }
        if (dtype == ORC_FP8) {
            acc = ks[s] * acc;
            acc_x = (double)ks[s] * acc_x;
        }
        out[s] = acc;
        if (exact_out)
            exact_out[s] = acc_x;
    }
    free(qf);
    free(wq);
    free(kf);
}

/* ------------------------------------------------------------------------ */
/* Top-k                                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
    float score;
    int32_t idx;
} orc_pair;

/* Higher score first; equal scores by lower index.  A total order. */
static int orc_cmp_pair(const void* a, const void* b)
{
    const orc_pair* x = (const orc_pair*)a;
    const orc_pair* y = (const orc_pair*)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/*
 * Top-k of one row of nvis scores by a full sort: the first min(k, nvis)
 * (score desc, index asc) entries; the rest of the k slots get index -1 and
 * score -inf.
 */
void orc_topk_row(const float* scores, int64_t nvis, int k, int32_t* out_idx, float* out_score)
{
    int64_t s;
    int j;
    orc_pair* p = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(nvis > 0 ? nvis : 1));
    for (s = 0; s < nvis; s++) {
        p[s].score = scores[s];
        p[s].idx = (int32_t)s;
    }
    qsort(p, (size_t)nvis, sizeof(orc_pair), orc_cmp_pair);
    for (j = 0; j < k; j++) {
        if (j < nvis) {
            out_idx[j] = p[j].idx;
            if (out_score)
                out_score[j] = p[j].score;
        } else {
            out_idx[j] = -1;
            if (out_score)
                out_score[j] = -INFINITY;
        }
    }
    free(p);
}

/*
 * The whole path for a batch of query rows.
 *
 *  keys: one flat logical array per sequence, concatenated: sequence b owns
 *        rows key_off[b] .. key_off[b] + seq_lens[b] - 1 of kc/ks (fp8) or kb
 *        (bf16).
 *  rows: query row r belongs to sequence row_seq[r] and sits at position
 *        row_pos[r]; it sees keys 0..row_pos[r] (causal).
 *  q: [R, H, d] bf16 bits, w: [R, H].
 *  out_idx/out_score: [R, k].  scores_full (optional): [R, max_s] with the
 *  score of every visible key (the rest untouched); exact_full likewise.
 */
void orc_score_topk(int dtype, int d, int H, int k, int64_t R,
                    const uint16_t* q, const float* w,
                    const int32_t* row_seq, const int64_t* row_pos,
                    const int64_t* key_off,
                    const uint8_t* kc, const float* ks, const uint16_t* kb,
                    int32_t* out_idx, float* out_score,
                    int64_t max_s, float* scores_full, double* exact_full)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < R; r++) {
        int64_t nvis = row_pos[r] + 1 > 0 ? row_pos[r] + 1 : 0;
        int64_t off = key_off[row_seq[r]];
        float* sc = (float*)malloc(sizeof(float) * (size_t)(nvis > 0 ? nvis : 1));
        double* ex = exact_full ? exact_full + r * max_s : NULL;
        orc_scores_row(dtype, d, H, q + r * H * d, w + r * H, nvis,
                       kc ? kc + off * d : NULL, ks ? ks + off : NULL,
                       kb ? kb + off * d : NULL, sc, ex);
        orc_topk_row(sc, nvis, k, out_idx + r * k, out_score ? out_score + r * k : NULL);
        if (scores_full)
            memcpy(scores_full + r * max_s, sc, sizeof(float) * (size_t)nvis);
        free(sc);
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
