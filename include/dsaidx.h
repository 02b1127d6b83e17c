/*
 * dsaidx.h -- C ABI of the DSA lightning-indexer library for GB300 (sm_103a).
 *
 * The library implements the indexer hot path of DeepSeek sparse attention:
 * store per-token 128-dim index keys in a paged cache, score every causally
 * visible key against each query and return the index_topk best positions.
 *
 * What the operations follow:
 *  - "DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
 *    (ROCm/ATOM issue #1507), section "How it was isolated": index keys are
 *    quantised to fp8 with a per-token scale and scattered into a paged cache
 *    (indexer_k_quant_and_cache), scored per query straight from the paged
 *    blocks at block size 32 or 64 (paged MQA logits), and reduced to the
 *    index_topk best positions per row (top_k_per_row_decode); prefill scores
 *    causal query chunks the same way (_score_topk_prefill).  Section
 *    "Environment": index_topk 1024 (512 in the repro), contexts up to
 *    1,048,576 tokens.
 *  - "The Pivot: A Single Edit That Finally Fixed DeepSeek V4's Long-Context
 *    Recall Failure", section "Assumptions and Input Knowledge": an fp8 index
 *    key takes 132 bytes per token (128 e4m3 codes + one fp32 scale), a bf16
 *    key 256 bytes.
 *  - "The Hypothesis That Refused to Die", section "The Context": the indexer
 *    ranks every cached position by a compressed query-key dot product and
 *    keeps the top K.  The score computed here is
 *        score[t, s] = sum_h w[t, h] * ReLU(q[t, h] . k[s])
 *    accumulated in fp32, with the per-head weights w supplied by the caller
 *    (any softmax or head-count scaling is folded into w).
 *
 * Conventions shared by every call:
 *  - head_dim is 128.  heads is 64 (other head counts return
 *    IDX_ERR_UNSUPPORTED).  topk is 1..2048.
 *  - Every pointer named *_dev is a device pointer into memory the caller owns
 *    (the library never allocates or frees device memory and never
 *    synchronises a stream, except idx_read_device_status).  `stream` is a
 *    cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - Results are valid in stream order after the call's kernels complete.
 *  - Host-side argument errors return at once, before any launch, and leave
 *    every buffer untouched.  Problems only the device can see (a block id
 *    outside the pool, seq_len > max_seq_len, a slot outside the pool, a
 *    pipeline wait that ran out) set a status word in the workspace (or in
 *    status_dev for idx_store_keys), skip the offending work and write -1 rows
 *    for the affected queries; no kernel traps or faults on them.
 *  - Query positions: the nq_b queries of sequence b are its LAST nq_b
 *    positions, pos = seq_len_b - nq_b + i, and a query sees keys s <= pos.
 *    Decode is the case nq_b = 1 (every key of the sequence is visible).
 *  - Top-k output: indices in descending score order, equal scores ordered by
 *    ascending index; when fewer than topk keys are visible the row is padded
 *    with index -1 (and score -inf).
 */
#ifndef DSAIDX_H
#define DSAIDX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_HEAD_DIM 128
#define IDX_MAX_TOPK 2048

typedef enum idx_status {
    IDX_OK = 0,
    IDX_ERR_INVALID_ARG = 1,        /* null pointer, bad size or out-of-range argument */
    IDX_ERR_UNSUPPORTED = 2,        /* valid but not built: heads != 64, head_dim != 128 */
    IDX_ERR_CUDA = 3,               /* a CUDA runtime call or launch failed */
    IDX_ERR_WORKSPACE_TOO_SMALL = 4,
    IDX_ERR_DEVICE_CHECK = 5,       /* device-side check failed (see idx_read_device_status) */
    IDX_ERR_TIMEOUT = 6             /* a bounded device wait ran out */
} idx_status;

/* Index-key storage formats of the paged cache. */
typedef enum idx_key_dtype {
    IDX_KEY_FP8_E4M3 = 0,   /* 128 e4m3 codes + fp32 scale per token (132 B) */
    IDX_KEY_BF16 = 1        /* 128 bf16 values per token (256 B) */
} idx_key_dtype;

/* Opaque host handle bound to one pool on the current device.  It holds the
 * pool geometry and the TMA descriptors of the pool; it owns no device
 * memory.  Not thread-safe to destroy while calls using it are being issued. */
typedef struct idx_cache idx_cache;

/*
 * Bytes of one paged block.  Layout of an fp8 block of bs tokens: bs rows of
 * 128 one-byte e4m3 codes (row i at byte 128*i), then bs fp32 scales (scale i
 * at byte 128*bs + 4*i): 8448 bytes at bs = 64.  A bf16 block is bs rows of
 * 128 bf16 values (row i at byte 256*i).  Returns 0 for unsupported arguments.
 * Follows the 132 / 256 bytes-per-token records of "The Pivot: A Single Edit
 * That Finally Fixed DeepSeek V4's Long-Context Recall Failure", section
 * "Assumptions and Input Knowledge"; the in-block order of codes and scales is
 * this library's choice (it keeps every 128-byte code row 16-byte aligned for
 * TMA).
 */
size_t idx_block_bytes(int key_dtype, int block_size, int head_dim);

/*
 * Bind a caller-owned pool of num_blocks blocks to a new handle.
 *  pool_dev: device pointer, 256-byte aligned, num_blocks * idx_block_bytes()
 *            bytes.  block_size: 32 or 64 (ROCm/ATOM issue #1507, section
 *            "How it was isolated", checks both).  head_dim: 128.
 * Errors: IDX_ERR_INVALID_ARG (null, misaligned, num_blocks < 1 or >= 2^31,
 * bad block size), IDX_ERR_UNSUPPORTED (head_dim), IDX_ERR_CUDA (no device or
 * the TMA descriptor could not be built).  *out is set only on IDX_OK.
 */
idx_status idx_cache_create(idx_cache** out, void* pool_dev, int64_t num_blocks,
                            int block_size, int head_dim, int key_dtype);

/* Release a handle (host memory only; the pool is untouched).  NULL is a
 * no-op.  (Library utility; no passage.) */
void idx_cache_destroy(idx_cache* cache);

/*
 * Quantise n keys and scatter them into the pool (the quant-and-cache write of
 * ROCm/ATOM issue #1507, section "How it was isolated").
 *  k_bf16_dev:       [n, 128] bf16, row-major, 16-byte aligned.
 *  slot_mapping_dev: [n] int64; token i goes to slot = block * block_size +
 *                    offset.  A negative slot skips the token; a slot beyond
 *                    the pool skips it too and sets status_dev.
 *  status_dev:       nullable device int32; set to IDX_ERR_DEVICE_CHECK when a
 *                    slot was out of range (never cleared by the library).
 * fp8 pools: per token amax over the 128 values, scale = amax / 448 (IEEE
 * division), code_i = e4m3(x_i / scale) rounded to nearest even with
 * saturation to +-448; amax = 0 gives scale 0 and zero codes.  bf16 pools:
 * the 256 bytes are copied.
 */
idx_status idx_store_keys(const idx_cache* cache, const void* k_bf16_dev,
                          const int64_t* slot_mapping_dev, int64_t n,
                          int32_t* status_dev, void* stream);

/*
 * idx_store_keys with each key first Walsh-Hadamard rotated: the fix (B) of
 * "DeepSeek-V4 index_topk=1024 sparse indexer can't recall verbatim lines"
 * (ROCm/ATOM issue #1507, section "Root cause"), which rotates the index key
 * on the store path to match the rotated index query, so that scores use
 * (Hq).(Hk) = q.k.  H is the orthonormal 128-point Walsh-Hadamard matrix in
 * Sylvester order, H[i][j] = (-1)^popcount(i & j) / sqrt(128).  The +-1 sums
 * of the bf16 inputs are formed exactly in double (exact for rows whose
 * exponents span at most 38 binades), multiplied by the double nearest
 * 1/sqrt(128) and rounded once to float; that float row is quantised as
 * above (fp8) or rounded to bf16, nearest even (bf16 pools).  Same
 * arguments, layout, ownership and errors as idx_store_keys.  The caller
 * supplies queries already rotated (the score calls do not rotate).
 */
idx_status idx_store_keys_rotated(const idx_cache* cache, const void* k_bf16_dev,
                                  const int64_t* slot_mapping_dev, int64_t n,
                                  int32_t* status_dev, void* stream);

/* Options of idx_store_keys_ex. */
#define IDX_STORE_ROTATE 1u          /* the Walsh-Hadamard rotation of idx_store_keys_rotated */
#define IDX_STORE_FP4_ROUNDTRIP 2u   /* the fp4 round trip below, after the rotation if any */

/*
 * idx_store_keys with options (flags: IDX_STORE_* bits; 0 is idx_store_keys,
 * IDX_STORE_ROTATE is idx_store_keys_rotated).  IDX_STORE_FP4_ROUNDTRIP puts
 * the key through the quantisation-aware fp4 round trip that "DeepSeek-V4
 * index_topk=1024 sparse indexer can't recall verbatim lines" (ROCm/ATOM
 * issue #1507, section "Where (main 0c7d50f9)") lists on the indexer's key
 * path after the rotation, fp4_act_quant_inplace(kv, 32): every block of 32
 * consecutive values of the (rotated or bf16-widened) float row gets the
 * scale s = fl32(amax / 6); each value x is replaced by fl32(c * s), c the
 * e2m1 value (0, 0.5, 1, 1.5, 2, 3, 4, 6 with sign) nearest to fl32(x / s),
 * a tie going to the even code and magnitudes beyond 6 to 6; a block of
 * zeros is kept.  The resulting float row is then quantised (fp8) or rounded
 * to bf16, nearest even, as for the rotated store.  Finite keys; same
 * arguments, layout, ownership and errors as idx_store_keys, plus
 * IDX_ERR_INVALID_ARG for unknown flag bits.
 */
idx_status idx_store_keys_ex(const idx_cache* cache, const void* k_bf16_dev,
                             const int64_t* slot_mapping_dev, int64_t n, unsigned flags,
                             int32_t* status_dev, void* stream);

/*
 * Gather read of the cache (cp_gather_indexer_k_quant_cache in "DeepSeek-V4
 * index_topk=1024 sparse indexer can't recall verbatim lines", ROCm/ATOM issue
 * #1507, section "How it was isolated", where a gathered copy cross-checks
 * the paged read): copies, byte for byte, every block that holds keys of a
 * sequence into a caller-owned dense grid of blocks -- block j of sequence b
 * (j < ceil(seq_lens[b] / block_size)) from block_table[b][j] to
 * dst_pool_dev + (b * max_blocks_per_seq + j) * idx_block_bytes().
 *  dst_pool_dev: batch * max_blocks_per_seq blocks, 16-byte aligned; blocks
 *                past a sequence's end are not written.  The grid is itself a
 *                pool: bound to a handle with the identity block table
 *                (row b: b * max_blocks_per_seq + j) the score calls read
 *                the same keys contiguously.
 *  status_dev:   nullable device int32, set to IDX_ERR_DEVICE_CHECK when a
 *                block id lies outside the pool (that block is skipped).
 * Errors: IDX_ERR_INVALID_ARG (null or misaligned pointers, other device),
 * IDX_ERR_CUDA (launch).
 */
idx_status idx_gather_blocks(const idx_cache* cache, const int32_t* block_table_dev,
                             int max_blocks_per_seq, const int32_t* seq_lens_dev, int batch,
                             void* dst_pool_dev, int32_t* status_dev, void* stream);

/*
 * Workspace bytes a decode call needs for this batch shape (depends on the
 * handle's device and key format).  0 on invalid arguments.  (Library
 * utility; no passage: the pages' kernels allocate their own scratch.)
 */
size_t idx_workspace_bytes_decode(const idx_cache* cache, int batch, int max_seq_len,
                                  int heads, int topk);

/*
 * Zero a newly allocated workspace (required once before its first use, and
 * again after any call that reported a device error).  The score calls leave
 * the workspace ready for the next call.  (Library utility; no passage.)
 */
idx_status idx_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * Decode: one query per sequence, every key of the sequence visible
 * (deepgemm_fp8_paged_mqa_logits + top_k_per_row_decode in ROCm/ATOM issue
 * #1507, section "How it was isolated", fused into one kernel: the scores stay
 * in shared memory).
 *  q_bf16_dev:      [batch, heads, 128] bf16.  fp8 pools: each (b, h) row is
 *                   quantised like a key (scale sq = amax / 448) and the scale
 *                   folded into the head weight, w' = w * sq.
 *  w_dev:           [batch, heads] fp32 head weights.
 *  block_table_dev: [batch, max_blocks_per_seq] int32 physical block ids;
 *                   logical key s of sequence b lives in block
 *                   block_table[b][s / block_size], row s % block_size.
 *  seq_lens_dev:    [batch] int32 keys per sequence (0 allowed).
 *  max_seq_len:     host upper bound on seq_lens (sizes the grid).
 *  out_idx_dev:     [batch, topk] int32.  out_score_dev: nullable
 *                   [batch, topk] fp32 scores of the selected keys.
 *  workspace_dev:   ws_bytes >= idx_workspace_bytes_decode(...), zeroed once
 *                   by idx_workspace_init; 256-byte aligned.
 * Concurrent calls must not share a workspace.
 */
idx_status idx_score_topk_decode(const idx_cache* cache, const void* q_bf16_dev,
                                 const float* w_dev, const int32_t* block_table_dev,
                                 int max_blocks_per_seq, const int32_t* seq_lens_dev,
                                 int batch, int max_seq_len, int heads, int topk,
                                 int32_t* out_idx_dev, float* out_score_dev,
                                 void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * idx_score_topk_decode that also writes each selected key's physical pool
 * slot: out_slot_dev (nullable, [batch, topk] int64, 8-byte aligned) gets
 * block_table[b][s / block_size] * block_size + s % block_size for selected
 * logical index s and -1 where out_idx is -1 -- the logical-to-physical
 * translate (csa_translate_pack) that "DeepSeek-V4 index_topk=1024 sparse
 * indexer can't recall verbatim lines" (ROCm/ATOM issue #1507, section "How it
 * was isolated") runs on the selected indices before sparse attention.  An
 * index whose block lies past max_blocks_per_seq gets -1.  Otherwise the same
 * arguments, results and errors as idx_score_topk_decode.
 */
idx_status idx_score_topk_decode_slots(const idx_cache* cache, const void* q_bf16_dev,
                                       const float* w_dev, const int32_t* block_table_dev,
                                       int max_blocks_per_seq, const int32_t* seq_lens_dev,
                                       int batch, int max_seq_len, int heads, int topk,
                                       int32_t* out_idx_dev, float* out_score_dev,
                                       int64_t* out_slot_dev, void* workspace_dev, size_t ws_bytes,
                                       void* stream);

/*
 * Decode without a workspace argument, for callers that cannot allocate
 * device memory: for example a plug-in that runs inside another framework's
 * process, where device memory belongs to that framework's allocator, or a
 * caller on a path where cudaMalloc / cudaFree are not allowed because they
 * may synchronise the device.  (The pages have no counterpart: this is a
 * convenience of this library.)
 *
 * Same arguments, results and errors as idx_score_topk_decode, without
 * workspace_dev / ws_bytes.  The scratch lives in a fixed 32 MiB area of
 * library-owned device memory that every GPU loading the library holds until
 * the process exits; a shape whose idx_workspace_bytes_decode() exceeds
 * 32 MiB is rejected with IDX_ERR_WORKSPACE_TOO_SMALL before anything runs.
 * (About 4 bytes per key of the longest sequence per cluster launched, at
 * most 10 MiB, plus, when sequences span several 65,536-key segments,
 * batch * (32 KiB + 8 * topk * ceil(max_seq_len / 65536)) bytes.)  The call allocates
 * nothing; it clears the part of the area it uses (an asynchronous memset on
 * `stream`) and launches the decode kernel.
 *  - The first call on each device looks up the area's device address (with
 *    that device current); make that first call before any stream capture.
 *  - All calls share the area: calls that may overlap on the GPU (different
 *    streams without ordering, or several host threads) race and corrupt each
 *    other's results; issue them in one stream or order them explicitly.
 *  - Device-side checks still produce -1 rows, but their status word is not
 *    readable by the caller (use idx_score_topk_decode to read it).
 */
idx_status idx_score_topk_decode_static(const idx_cache* cache, const void* q_bf16_dev,
                                        const float* w_dev, const int32_t* block_table_dev,
                                        int max_blocks_per_seq, const int32_t* seq_lens_dev,
                                        int batch, int max_seq_len, int heads, int topk,
                                        int32_t* out_idx_dev, float* out_score_dev, void* stream);

/* Workspace bytes a prefill call needs.  0 on invalid arguments.  (Library
 * utility; no passage.) */
size_t idx_workspace_bytes_prefill(const idx_cache* cache, int batch, int total_q,
                                   int max_seq_len, int heads, int topk);

/*
 * Prefill: causal query chunks (_score_topk_prefill in ROCm/ATOM issue #1507,
 * section "Root cause found", reading the paged cache directly instead of a
 * gathered copy).
 *  q_bf16_dev:       [total_q, heads, 128] bf16; w_dev: [total_q, heads] fp32.
 *  cu_seqlens_q_dev: [batch + 1] int32, cu[0] = 0, rows cu[b]..cu[b+1]-1 are
 *                    the queries of sequence b (at its last positions).
 *  seq_lens_dev:     [batch] int32 keys of each sequence, this chunk included.
 *  out_idx_dev:      [total_q, topk]; out_score_dev nullable [total_q, topk].
 * Other arguments as for decode.  batch <= 4096.
 */
idx_status idx_score_topk_prefill(const idx_cache* cache, const void* q_bf16_dev,
                                  const float* w_dev, const int32_t* cu_seqlens_q_dev,
                                  const int32_t* seq_lens_dev, const int32_t* block_table_dev,
                                  int max_blocks_per_seq, int batch, int total_q,
                                  int max_seq_len, int heads, int topk,
                                  int32_t* out_idx_dev, float* out_score_dev,
                                  void* workspace_dev, size_t ws_bytes, void* stream);

/*
 * idx_score_topk_prefill that also writes each selected key's physical pool
 * slot to out_slot_dev (nullable, [total_q, topk] int64, 8-byte aligned; -1
 * where out_idx is -1), the translate described at
 * idx_score_topk_decode_slots.  Otherwise the same as idx_score_topk_prefill.
 */
idx_status idx_score_topk_prefill_slots(const idx_cache* cache, const void* q_bf16_dev,
                                        const float* w_dev, const int32_t* cu_seqlens_q_dev,
                                        const int32_t* seq_lens_dev, const int32_t* block_table_dev,
                                        int max_blocks_per_seq, int batch, int total_q, int max_seq_len,
                                        int heads, int topk, int32_t* out_idx_dev, float* out_score_dev,
                                        int64_t* out_slot_dev, void* workspace_dev, size_t ws_bytes,
                                        void* stream);

/*
 * Synchronise `stream` and read the device status word of a workspace into
 * *code_out (IDX_OK, IDX_ERR_DEVICE_CHECK or IDX_ERR_TIMEOUT).  For tests and
 * debugging; the status stays set until idx_workspace_init.  (Library
 * utility; no passage.)
 */
idx_status idx_read_device_status(const void* workspace_dev, void* stream, int32_t* code_out);

/* Static description of a status code.  (Library utility; no passage.) */
const char* idx_status_str(idx_status status);

/*
 * Test hook for the failure path (library utility; no passage).  Shortens the
 * limit of the decode kernel's pipeline waits to limit_ns nanoseconds and
 * makes its MMA issuer withhold the completion signal of the first
 * accumulator of every CTA, so that a bounded wait runs out: the call then
 * records IDX_ERR_TIMEOUT in the workspace status, writes -1 rows for the
 * affected sequences, drains its own copies and MMAs, frees TMEM and returns
 * (no GPU fault, trap or hang).  0 (or any value >= 2 s) restores the normal
 * 2 s limit and the normal signalling.  Process-wide; affects calls issued
 * after it returns.
 */
idx_status idx_test_set_wait_limit(unsigned long long limit_ns);

/*
 * Per-kernel timing of the score calls (library utility; no passage).
 * idx_kernel_timing(capacity), capacity > 0: every later score call records
 * a CUDA event before and after each kernel it launches, on the call's
 * stream, for up to `capacity` kernels (decode: one kernel per call; prefill:
 * the scoring kernel, then the row selection); capacity 0 stops and frees
 * the events.  Returns the capacity set, 0 when stopped, -1 on a CUDA error.
 * idx_kernel_times(out_ms, max) waits for the recorded events, writes the
 * durations in milliseconds of up to `max` recorded kernels in launch order
 * to host array out_ms (nullable: only counts), starts a new record and
 * returns how many it wrote (-1 on a CUDA error).  Not for calls issued
 * during stream capture.
 */
int idx_kernel_timing(int capacity);
int idx_kernel_times(float* out_ms, int max);

/*
 * (Library utility; no passage.)  Copies `bytes` from src to dst with a
 * kernel on `stream`, for staging a step's inputs and results: each pointer is
 * device memory, pinned host memory (used through its device alias), or, on a
 * device that reads host page tables, any host memory; both 16-byte aligned
 * and bytes a multiple of 16.  Launched like the score calls' kernels
 * (programmatic serialization: it may be scheduled while the previous kernel
 * in the stream finishes, and waits for it before touching memory).  Errors:
 * IDX_ERR_INVALID_ARG (null, misaligned or unreachable pointers), IDX_ERR_CUDA.
 */
idx_status idx_copy(void* dst, const void* src, size_t bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSAIDX_H */
