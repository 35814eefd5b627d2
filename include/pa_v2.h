/*
 * pa_v2.h -- C ABI of a GB300 (sm_103a) library for PagedAttention V2 single-query decode
 * attention over a block-paged KV cache, plus the slot-mapping cache writer.
 *
 * Every entry point takes plain pointers, sizes and a CUDA stream; nothing here depends on
 * any framework's tensor types.  Pointers named "device" must point to device memory (or
 * memory the device can address).  All buffers are owned by the caller: these calls
 * allocate nothing, never synchronise the stream, and return as soon as the work is
 * enqueued.  Results are valid in stream order.
 *
 * Every call may be captured into a CUDA graph (stream capture).  What the decode, append,
 * cache-writer, copy_blocks and prefix calls choose on the host (grid, kernel form,
 * partitions per CTA, cluster split, context split plan) follows from the sizes, dtypes and
 * pointer alignments passed, never from the contents of device buffers, so a replay is
 * correct for whatever the captured buffers hold then (lengths up to the captured
 * max_seq_len or table width).  pa_swap_blocks reads its mapping on the host: a replay
 * repeats the captured pairs.  Make one uncaptured call of each configuration first, which
 * sets the kernels' shared-memory attributes; the PA_CHECK=1 host check synchronises the
 * stream and cannot be captured.
 *
 * Layouts are row-major C arrays:
 *   query        [num_seqs][num_heads][head_size]                      q dtype
 *   output       [num_seqs][num_heads][head_size]                      q dtype
 *   key_cache    [num_blocks][num_kv_heads][head_size / x][block_size][x]
 *   value_cache  [num_blocks][num_kv_heads][head_size][block_size]
 *                x = 16 / (bytes per cache element): 8 for fp16/bf16, 16 for fp8 e4m3.
 *   block_tables [num_seqs][max_blocks_per_seq]   int32, logical block -> physical block
 *   seq_lens     [num_seqs]                       int32, tokens per sequence
 *   exp_sums     [num_seqs][num_heads][max_num_partitions]             float32
 *   max_logits   [num_seqs][num_heads][max_num_partitions]             float32
 *   tmp_output   [num_seqs][num_heads][max_num_partitions][head_size]  float32 or q dtype
 * These are the argument layouts of "paged_attention_v2_pytorch.py" (paged_attention_v2_pytorch)
 * and the cache views of "paged_attn.py" (split_kv_cache).
 */
#ifndef PA_V2_H_
#define PA_V2_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_DT_F16 = 0,
    PA_DT_BF16 = 1,
    PA_DT_F32 = 2,
    PA_DT_FP8_E4M3 = 3
} pa_dtype;

/* "auto": the cache holds the query dtype; "fp8_e4m3": the cache holds OCP e4m3fn codes. */
typedef enum {
    PA_KV_AUTO = 0,
    PA_KV_FP8_E4M3 = 1
} pa_kv_cache_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* a pointer, size, ratio or scale breaks the contract below */
    PA_ERR_UNSUPPORTED = 2, /* a valid combination this build does not implement          */
    PA_ERR_CUDA = 3,        /* the CUDA runtime reported an error while enqueueing          */
    PA_ERR_SCRATCH_TOO_SMALL = 4 /* pa_v2_decode_noalloc: the step needs more than its fixed
                                    device scratch (PA_NOALLOC_SCRATCH_BYTES)                 */
} pa_status;

/* Size of the fixed device scratch behind pa_v2_decode_noalloc (32 MiB per device). */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pa_v2_decode -- one decode step of paged attention, two phases.
 *
 * Defines: "paged_attention_v2_pytorch.py", paged_attention_v2_pytorch (phase 1: per
 * sequence s, query head h and 512-token partition p, the scores
 *   s_t = scale * <q, k_t * k_scale> + (alibi ? alibi_slopes[h] * t : 0),  t = 0 .. L-1,
 * the partition max m_p, exp-sum l_p = sum exp(s_t - m_p) and weighted V; phase 2: the
 * log-sum-exp combine), and "paged_attention_v2_triton.py", _paged_attn_v2_reduce_kernel
 * (out = sum_p exp(m_p - g) l_p tmp_p / sum_p exp(m_p - g) l_p, g = max_p m_p).
 * Query head h reads kv head h / (num_heads / num_kv_heads) (the GQA view of the query).
 *
 * Writes, for every sequence with L = seq_lens[s] tokens and P = ceil(L / 512) partitions:
 *   max_logits[s][h][p], exp_sums[s][h][p]  for p < P (m_p in natural-log units, absolute
 *       ALiBi positions); max_logits = -inf and exp_sums = 0 for P <= p < max_num_partitions;
 *   tmp_output[s][h][p][:] = sum_t exp(s_t - m_p) v_t / l_p  (partition-normalised) for
 *       p < P when P > 1; left untouched otherwise;
 *   output[s][h][:] = softmax(s) V in the query dtype; all zeros when L == 0.
 * Sequences with P == 1 take a single pass: output is written directly, and the p = 0
 * statistics are still written.
 *
 * Arguments:
 *   output, exp_sums, max_logits, tmp_output   device, caller-owned, layouts above.
 *   query, key_cache, value_cache               device; key_cache, value_cache and query
 *                                               16-byte aligned.
 *   num_seqs (0 .. 65535), num_heads, num_kv_heads (num_heads % num_kv_heads == 0),
 *   head_size in {64, 80, 96, 112, 120, 128, 192, 256} (the supported sizes listed in
 *       "paged_attn.py", get_supported_head_sizes); head_size % x == 0.
 *   scale                 softmax scale (e.g. 1/sqrt(head_size)).
 *   block_tables          device int32 [num_seqs][max_blocks_per_seq].
 *   max_blocks_per_seq    >= ceil(max_seq_len / block_size).
 *   num_blocks            physical blocks in each cache (ids must lie in [0, num_blocks)).
 *   seq_lens              device int32 [num_seqs]; every entry in [0, max_seq_len].
 *   block_size            8, 16 or 32 (512 % block_size == 0, "paged_attn.py" forward_decode).
 *   max_seq_len           upper bound on every seq_lens entry.
 *   max_num_partitions    >= ceil(max_seq_len / 512) and >= 1; the third extent of the
 *                         workspace arrays.
 *   alibi_slopes          device float32 [num_heads], or NULL for no ALiBi bias.
 *   q_dtype               PA_DT_F16 or PA_DT_BF16 (query and output).
 *   kv_cache_dtype        PA_KV_AUTO (cache in q_dtype) or PA_KV_FP8_E4M3.
 *   tmp_dtype             element type of tmp_output: PA_DT_F32, or q_dtype (as the pages'
 *                         "paged_attn.py" forward_decode allocates it: half the workspace
 *                         traffic, at the cost of one more rounding of each partition's
 *                         output to the output dtype).
 *   k_scale, v_scale      > 0, finite; multiply the decoded key and value elements.
 *   stream                the CUDA stream the kernels are enqueued on.
 *
 * Errors: PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED are returned before anything is
 * enqueued.  Table contents are not read on the host: a block id outside [0, num_blocks),
 * a sequence longer than its table row or than max_num_partitions * 512, or a negative
 * length is skipped on the device (those tokens are masked out) and recorded in the flags
 * pa_get_device_errors returns; with the environment variable PA_CHECK=1 the tables are
 * instead copied to the host and checked first (this synchronises the stream) and a bad
 * entry returns PA_ERR_INVALID_ARG.  PA_ERR_CUDA reports a launch error.
 */
PA_API pa_status pa_v2_decode(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                       const void* query, const void* key_cache, const void* value_cache,
                       int num_seqs, int num_heads, int num_kv_heads, int head_size,
                       float scale, const int32_t* block_tables, int max_blocks_per_seq,
                       int num_blocks, const int32_t* seq_lens, int block_size,
                       int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                       pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype,
                       float k_scale, float v_scale, cudaStream_t stream);

/*
 * pa_v2_decode_fused -- pa_v2_decode with the partition combine done inside phase 1.
 *
 * Defines: the same step as pa_v2_decode ("paged_attention_v2_pytorch.py",
 * paged_attention_v2_pytorch; "paged_attention_v2_triton.py", _paged_attn_v2_reduce_kernel),
 * with the V1/V2 dispatch of "paged_attn.py" (forward_decode) re-decided for this GPU: the
 * pages choose per call between a single pass (V1) and partitions plus a reduce kernel (V2);
 * here every sequence is partitioned, and the last CTA of each (sequence, head group) to
 * finish runs the reduce (an arrival counter, no waiting), so no second kernel waits for the
 * whole grid.  A sequence that one CTA covers entirely (one partition) is a single pass.
 *
 * Arguments and results: as pa_v2_decode (output, max_logits and exp_sums identical in
 * meaning), except
 *   tmp_output   scratch: its contents after the call are unspecified (with an fp32
 *                tmp_output each CTA merges the partitions it streams into one row).
 *   counters     device uint32 [num_counters], num_counters >=
 *                pa_v2_decode_num_counters(num_seqs, num_heads, num_kv_heads); 4-byte aligned.
 *                Every entry must be zero before the first call that uses the array (clear
 *                it once when it is allocated); every call leaves it all zero again.  Like
 *                the workspace, it must not be used by calls that can overlap on the GPU.
 *                NULL: exactly pa_v2_decode.
 * When the combine would read more than 64 KiB of rows per (sequence, head group) (a 16-bit
 * tmp_output over many partitions), the call falls back to pa_v2_decode's two kernels and the
 * counters are not touched.
 * Errors: as pa_v2_decode; PA_ERR_INVALID_ARG also for a misaligned or too short counters array.
 */
PA_API pa_status pa_v2_decode_fused(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                    const void* query, const void* key_cache, const void* value_cache,
                                    int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                    float scale, const int32_t* block_tables, int max_blocks_per_seq,
                                    int num_blocks, const int32_t* seq_lens, int block_size,
                                    int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                                    pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype,
                                    float k_scale, float v_scale, uint32_t* counters, int64_t num_counters,
                                    cudaStream_t stream);

/*
 * pa_v2_decode_append -- one decode step that also appends each sequence's newest token to
 * the cache: pa_reshape_and_cache of that token followed by pa_v2_decode, in one kernel.
 *
 * Defines: "paged_attn.py", forward_decode after write_to_paged_cache (the decode writes the
 * new key/value into the paged cache, then attends over it), with the slot of sequence s's
 * new token taken from its block table: position t = seq_lens[s] - 1, slot
 * block_tables[s][t / block_size] * block_size + t % block_size (what slot_mapping holds in a
 * decode step).  The token is encoded exactly as pa_reshape_and_cache encodes it (bitwise
 * copy, or e4m3fn of x / k_scale resp. x / v_scale in IEEE fp32), and attention uses the
 * encoded value.  The CTA that streams the token's page writes it into the caches and into
 * its shared-memory copy of that page, so the step has no separate writer kernel.
 *
 * Arguments: as pa_v2_decode, except that tmp_output is scratch (its contents after the call
 * are unspecified: a CTA that streams several partitions of a long sequence folds them into
 * one fp32 row, and phase 2 merges those rows); output, max_logits and exp_sums are as there.
 * In addition:
 *   key, value          device [num_seqs][num_kv_heads][head_size] rows in q_dtype (the
 *                       newest token of each sequence); consecutive sequences' rows are
 *                       key_stride_s / value_stride_s ELEMENTS apart (>= num_kv_heads *
 *                       head_size, multiples of 8); 16-byte aligned.
 *   key_cache, value_cache  written (the new token's slot) as well as read.
 *   order               device int32 [num_seqs] scratch (4-byte aligned), or NULL.  Where
 *                       the step's CTAs stride over several partitions each (wide ragged
 *                       batches), the call first writes the pa_v2_decode_order permutation
 *                       into it and serves the sequences in that order, so the CTAs with the
 *                       most partitions start first instead of forming the grid's tail.  The
 *                       results do not depend on it.
 * Sequences with seq_lens[s] == 0 append nothing.  Every other sequence must have its newest
 * token at position seq_lens[s] - 1 of its table row; a page id outside the cache there
 * masks the token (and is flagged) as in pa_v2_decode.
 * Errors: as pa_v2_decode; PA_ERR_INVALID_ARG also for a null, misaligned or short row or a
 * misaligned order buffer.
 */
PA_API pa_status pa_v2_decode_append(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                     const void* query, const void* key, const void* value,
                                     int64_t key_stride_s, int64_t value_stride_s, void* key_cache,
                                     void* value_cache, int num_seqs, int num_heads, int num_kv_heads,
                                     int head_size, float scale, const int32_t* block_tables,
                                     int max_blocks_per_seq, int num_blocks, const int32_t* seq_lens,
                                     int block_size, int max_seq_len, int max_num_partitions,
                                     const float* alibi_slopes, pa_dtype q_dtype,
                                     pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype, float k_scale,
                                     float v_scale, int32_t* order, cudaStream_t stream);

/*
 * pa_v2_decode_order -- the order in which the decode grid serves the sequences: order[0 ..
 * num_seqs) becomes a permutation of 0 .. num_seqs - 1 by decreasing partition count
 * ceil(seq_lens[s] / 512) (counts above 1022 share one class; the order inside a class is
 * unspecified).  A scheduling aid, not part of the pages' method (their grid is
 * (sequences, heads, partitions) in index order): with partitions dealt to CTAs in strides,
 * a CTA's work grows with its sequence's length, and starting the longest first shortens the
 * grid's tail (longest-job-first).  pa_v2_decode_append calls it itself when given an order
 * buffer.
 * Arguments: seq_lens device int32 [num_seqs]; num_seqs 0 .. 65535; order device int32
 * [num_seqs]; both 4-byte aligned.  Reads seq_lens after the previous kernel in the stream.
 * Errors: PA_ERR_INVALID_ARG before anything is enqueued; PA_ERR_CUDA on a launch failure.
 */
PA_API pa_status pa_v2_decode_order(const int32_t* seq_lens, int num_seqs, int32_t* order, cudaStream_t stream);

/*
 * pa_v2_decode_head_scales, pa_v2_decode_append_head_scales -- pa_v2_decode and
 * pa_v2_decode_append with one k_scale and one v_scale per kv head.
 *
 * Defines: the step of pa_v2_decode (resp. pa_v2_decode_append) with the dequantisation of
 * "paged_attention_v2_pytorch.py" (paged_attention_v2_pytorch: cache values times k_scale /
 * v_scale) taken per kv head, the per-head scale variant of that step: keys and values of
 * kv head j are multiplied by k_scales[j] and v_scales[j], and the appended rows of head j
 * are encoded as e4m3fn((float)x / k_scales[j]) (resp. v_scales[j]) for an fp8 cache.  The
 * pages pass one float each; these entry points are this library's extension.
 *
 * Arguments: as pa_v2_decode (resp. pa_v2_decode_append), with k_scale / v_scale replaced by
 *   k_scales, v_scales  device float [num_kv_heads], 4-byte aligned, read after the previous
 *                       kernel in the stream has completed (so a kernel that writes them
 *                       right before the call is seen).  Each must be finite and > 0: a
 *                       value that is not is used as given and recorded in the device error
 *                       flags (bit 8).
 * With every entry equal to one value v the results are bit-identical to the per-tensor
 * entry point called with k_scale = v (resp. v_scale = v): the score multiplier is rounded
 * as scale * k_scale, then times log2(e), in binary32 on both paths.
 * Errors: as the per-tensor entry points; PA_ERR_INVALID_ARG also for a null or misaligned
 * scale array.
 */
PA_API pa_status pa_v2_decode_head_scales(void* output, float* exp_sums, float* max_logits, void* tmp_output,
                                          const void* query, const void* key_cache, const void* value_cache,
                                          int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                          float scale, const int32_t* block_tables, int max_blocks_per_seq,
                                          int num_blocks, const int32_t* seq_lens, int block_size,
                                          int max_seq_len, int max_num_partitions, const float* alibi_slopes,
                                          pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype, pa_dtype tmp_dtype,
                                          const float* k_scales, const float* v_scales, cudaStream_t stream);

PA_API pa_status pa_v2_decode_append_head_scales(
    void* output, float* exp_sums, float* max_logits, void* tmp_output, const void* query, const void* key,
    const void* value, int64_t key_stride_s, int64_t value_stride_s, void* key_cache, void* value_cache,
    int num_seqs, int num_heads, int num_kv_heads, int head_size, float scale, const int32_t* block_tables,
    int max_blocks_per_seq, int num_blocks, const int32_t* seq_lens, int block_size, int max_seq_len,
    int max_num_partitions, const float* alibi_slopes, pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
    pa_dtype tmp_dtype, const float* k_scales, const float* v_scales, int32_t* order, cudaStream_t stream);

/* Arrival counters pa_v2_decode_fused needs: num_seqs * num_kv_heads *
 * ceil((num_heads / num_kv_heads) / 8) (one per sequence and group of up to 8 query heads of a
 * kv head); 0 for invalid sizes. */
PA_API int64_t pa_v2_decode_num_counters(int num_seqs, int num_heads, int num_kv_heads);

/*
 * pa_reshape_and_cache -- scatter new key/value rows into the paged caches by slot.
 *
 * Defines: "paged_attn.py", write_to_paged_cache (-> reshape_and_cache with the flattened
 * slot_mapping) and split_kv_cache (the cache views).  For token t with
 * slot = slot_mapping[t] >= 0, b = slot / block_size, o = slot % block_size:
 *   key_cache[b][h][i / x][o][i % x] = enc(key[t][h][i]),
 *   value_cache[b][h][i][o]         = enc(value[t][h][i]).
 * enc is a bitwise copy when kv_cache_dtype == PA_KV_AUTO, and
 * round-to-nearest-even-with-saturation to e4m3fn of (float)x / k_scale (resp. v_scale),
 * the division in IEEE binary32, when kv_cache_dtype == PA_KV_FP8_E4M3.
 * A negative slot skips the token.
 *
 * Arguments:
 *   key, value            device [num_tokens][num_kv_heads][head_size] rows in src_dtype;
 *                         consecutive tokens are key_stride_t / value_stride_t ELEMENTS
 *                         apart (heads and head elements are contiguous inside a row).
 *   key_cache, value_cache  device, layouts above, 16-byte aligned.
 *   slot_mapping          device int64 [num_tokens].
 *   num_tokens >= 0, num_kv_heads > 0, head_size as for pa_v2_decode, block_size 8/16/32,
 *   num_blocks > 0; src_dtype PA_DT_F16 or PA_DT_BF16; k_scale, v_scale > 0 and finite.
 * Errors: as for pa_v2_decode; a slot at or beyond num_blocks * block_size is skipped on
 * the device and recorded in the device error flags.
 */
PA_API pa_status pa_reshape_and_cache(const void* key, const void* value, int64_t key_stride_t,
                               int64_t value_stride_t, void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                               int head_size, int block_size, int num_blocks,
                               pa_dtype src_dtype, pa_kv_cache_dtype kv_cache_dtype,
                               float k_scale, float v_scale, cudaStream_t stream);

/*
 * pa_reshape_and_cache_head_scales -- pa_reshape_and_cache with one k_scale and one v_scale
 * per kv head: for an fp8 cache head h's rows are encoded as e4m3fn((float)x / k_scales[h])
 * (resp. v_scales[h]); a PA_KV_AUTO cache is a bitwise copy as there.  The pages' writer
 * takes one float each; this is the per-head variant of the same encode.
 * Arguments: as pa_reshape_and_cache, with k_scale / v_scale replaced by device float arrays
 * k_scales, v_scales [num_kv_heads] (4-byte aligned; read after the previous kernel in the
 * stream has completed; a value that is not finite and > 0 is used as given and recorded in
 * the device error flags, bit 8).
 * Errors: as pa_reshape_and_cache; PA_ERR_INVALID_ARG also for a null or misaligned array.
 */
PA_API pa_status pa_reshape_and_cache_head_scales(const void* key, const void* value, int64_t key_stride_t,
                                                  int64_t value_stride_t, void* key_cache, void* value_cache,
                                                  const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                                  int head_size, int block_size, int num_blocks,
                                                  pa_dtype src_dtype, pa_kv_cache_dtype kv_cache_dtype,
                                                  const float* k_scales, const float* v_scales,
                                                  cudaStream_t stream);

/*
 * pa_copy_blocks -- copy whole blocks inside every layer's K and V cache (copy-on-write of
 * shared prefixes).
 *
 * Defines: "paged_attn.py", copy_blocks (-> ops.copy_blocks(key_caches, value_caches,
 * src_to_dists)).  For every layer l < num_layers and pair i < num_pairs with
 * (src, dst) = (block_mapping[2i], block_mapping[2i+1]):
 *   key_caches[l][dst] = key_caches[l][src] and value_caches[l][dst] = value_caches[l][src],
 * where a block is the block_bytes contiguous bytes of one physical block of one cache
 * (num_kv_heads * head_size * block_size * element size).
 *
 * Arguments:
 *   key_caches, value_caches  HOST arrays of num_layers device pointers, 16-byte aligned.
 *   block_mapping             device int64 [num_pairs][2] (src, dst).
 *   block_bytes               > 0, a multiple of 16.   num_blocks: blocks in each cache.
 * Pairs run in parallel, so no dst may also be the src of another pair in the same call.
 * Errors: PA_ERR_INVALID_ARG before anything is enqueued; an id outside [0, num_blocks) is
 * skipped on the device and recorded in pa_get_device_errors (bit 4).
 */
PA_API pa_status pa_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                                const int64_t* block_mapping, int num_pairs, int64_t block_bytes,
                                int num_blocks, cudaStream_t stream);

/*
 * pa_swap_blocks -- move whole blocks from one cache to another, typically between the
 * GPU cache and a pinned host cache.
 *
 * Defines: "paged_attn.py", swap_blocks (-> ops.swap_blocks(src, dst, src_to_dst), called
 * once for the K caches and once for the V caches).  For every pair (src, dst) of
 * block_mapping: dst_cache[dst] = src_cache[src], block_bytes bytes each.
 *
 * Arguments:
 *   src_cache, dst_cache  device or pinned host memory (any pair the runtime can copy).
 *   block_mapping         HOST int64 [num_pairs][2] (src, dst), checked on the host.
 *   block_bytes > 0; src_num_blocks / dst_num_blocks: blocks in each cache.
 * Where both caches are reachable from the current device (its own memory, managed memory,
 * or host memory pinned or registered while it was current, through its device mapping),
 * block_bytes is a multiple of 16 and both caches are 16-byte aligned, a kernel on `stream`
 * moves the blocks (one launch per 480 pairs, the pairs in its parameters); otherwise one
 * cudaMemcpyAsync per pair.
 * Errors: PA_ERR_INVALID_ARG (nothing enqueued) for a bad size or an id out of range;
 * PA_ERR_CUDA if a copy or launch cannot be enqueued.
 */
PA_API pa_status pa_swap_blocks(const void* src_cache, void* dst_cache, const int64_t* block_mapping,
                                int num_pairs, int64_t block_bytes, int src_num_blocks,
                                int dst_num_blocks, cudaStream_t stream);

/*
 * pa_prefix -- chunked-prefix (prefill) attention: new tokens of each sequence attend to the
 * sequence's cached context and, causally, to the new tokens before and at themselves.
 *
 * Defines: "paged_attn.py", forward_prefix / _forward_prefix_pytorch.  Sequence s has
 * ctx = context_lens[s] tokens in the paged cache (views as for pa_v2_decode) and
 * q_len = query_start_loc[s+1] - query_start_loc[s] new tokens, rows
 * query_start_loc[s] .. query_start_loc[s+1]-1 of query/key/value.  For new token j and
 * query head h (kv head h / (num_heads / num_kv_heads)):
 *   keys   = the ctx cached tokens (block_tables[s][t / block_size], slot t % block_size),
 *            then key rows 0..j of the chunk (the chunk is read from key/value, not the cache);
 *   output = softmax(scale * q . keys) . values, rounded once to the query dtype.
 * The pages fix scale = head_size^-0.5; it is an argument here.  The cache holds the query
 * dtype (fp8 caches have no prefix path on the pages).
 *
 * Arguments (device pointers unless noted):
 *   output       [T][num_heads][head_size] contiguous, T = query_start_loc[num_seqs].
 *   query        rows of q_row_stride elements, head h at h * head_size; key/value rows of
 *                kv_row_stride elements, kv head at kvh * head_size.  Strides are multiples
 *                of 8 elements; every pointer is 16-byte aligned.
 *   key_cache    [num_blocks][num_kv_heads][head_size/8][block_size][8]
 *   value_cache  [num_blocks][num_kv_heads][head_size][block_size]
 *   block_tables int32 [num_seqs][max_blocks_per_seq]
 *   query_start_loc int32 [num_seqs + 1] non-decreasing; context_lens int32 [num_seqs].
 *   max_query_len  host int >= every q_len (sizes the grid).
 *   head_size in {64, 80, 96, 112, 120, 128, 192, 256}; block_size in {8, 16, 32};
 *   num_blocks * num_kv_heads < 2^31 (pages are addressed by 32-bit copy coordinates);
 *   dtype PA_DT_F16 or PA_DT_BF16 (query, key, value, caches and output).
 *
 * Split contexts (not on the pages; it changes where the work runs, not the result): with a
 * workspace and max_splits > 1, a sequence whose context exceeds min_split_keys tokens
 * (a multiple of 64) is cut into at most max_splits equal parts of whole 64-token tiles, each
 * attended by its own CTAs (the chunk goes with the last part).  min_split_keys = 0 asks for
 * the library's plan: contexts over 16384 tokens are cut only where one sequence's row tiles
 * (of all its kv heads) would occupy fewer than half the GPU's SMs, since a grid that already
 * spreads each sequence over the GPU runs faster unsplit (4 sequences x 1024 new tokens over
 * contexts up to 96K at head size 256: 2.82 against 3.04 ms cut into up to 7 parts).  Each
 * part leaves its un-normalised output and its rows' (max, sum) in the workspace, and a second
 * kernel merges the parts by the log-sum-exp rule and writes the output rows of those
 * sequences.  Long contexts then spread over the GPU instead of leaving a tail of a few CTAs.
 *   workspace        device memory, 16-byte aligned, owned by the caller, at least
 *                    pa_prefix_workspace_size(num_seqs, num_heads, num_kv_heads, head_size,
 *                    max_query_len, max_splits) bytes; nothing in it needs initialising and
 *                    it must not be shared by calls that can overlap.  NULL (or max_splits
 *                    <= 1) leaves every sequence in one part and ignores the other two.
 *   max_splits       1 .. 32; the call uses no more parts than the longest context the
 *                    tables can hold (max_blocks_per_seq * block_size) needs.
 * Errors: PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED before anything is enqueued (a workspace
 * that is too small or misaligned, max_splits > 32, min_split_keys not a multiple of 64
 * included).  On the device, a cached block id outside [0, num_blocks) masks that page (bit 5
 * of pa_get_device_errors); a context longer than the table row is capped to the row, as the
 * pages do (bit 6); a sequence with q_len > max_query_len or a negative length is skipped
 * (bit 7).
 */
PA_API pa_status pa_prefix(void* output, const void* query, const void* key, const void* value,
                           const void* key_cache, const void* value_cache, int num_seqs,
                           int num_heads, int num_kv_heads, int head_size, float scale,
                           const int32_t* block_tables, int max_blocks_per_seq, int num_blocks,
                           const int32_t* query_start_loc, const int32_t* context_lens,
                           int max_query_len, int block_size, int64_t q_row_stride,
                           int64_t kv_row_stride, pa_dtype dtype, void* workspace,
                           size_t workspace_bytes, int max_splits, int min_split_keys,
                           cudaStream_t stream);

/* Bytes of workspace pa_prefix needs for up to max_splits parts per context:
 * num_seqs * num_kv_heads * ceil(max_query_len * (num_heads / num_kv_heads) / 128) *
 * max_splits * 128 * (head_size * 4 + 8).  0 when max_splits <= 1 or an argument is out of
 * range. */
PA_API size_t pa_prefix_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                       int head_size, int max_query_len, int max_splits);

/* Parts each context is cut into by a pa_prefix call with these arguments (has_workspace: a
 * non-NULL workspace is passed), written to *parts: 1 for no cut (one kernel), else the parts
 * (the attention kernel and the combine).  The library's plan (min_split_keys = 0) depends
 * on the current device's SM count.  Errors: PA_ERR_INVALID_ARG for a NULL parts or an
 * argument pa_prefix would reject; PA_ERR_UNSUPPORTED for a dtype or head size it does not
 * implement; PA_ERR_CUDA when the device cannot be queried. */
PA_API pa_status pa_prefix_num_parts(int num_heads, int num_kv_heads, int head_size, pa_dtype dtype,
                                     int max_query_len, int max_blocks_per_seq, int block_size,
                                     int max_splits, int min_split_keys, int has_workspace, int* parts);

/* Tokens per partition: 512 ("paged_attention_v2_pytorch.py", _PARTITION_SIZE). */
PA_API int pa_v2_partition_size(void);

/* A static, human-readable name for a status code. */
PA_API const char* pa_status_string(pa_status status);

/* Device-side error flags (bit 0: a block id outside [0, num_blocks) or a table row too
 * short; bit 1: a sequence longer than max_num_partitions * 512 or a negative length;
 * bit 2: a bounded wait for a shared-memory copy gave up (decode or pa_prefix; pa_prefix
 * also when its shared memory is not 1 KiB aligned); bit 3: a slot outside the
 * cache; bit 4: a pa_copy_blocks id outside the cache; bits 5-7: pa_prefix, see there;
 * bit 8: a per-kv-head k or v scale that is not finite and > 0; bit 9: a grid-order entry
 * outside [0, num_seqs), whose grid slice is then skipped).
 * Reads the flags of the current device (this synchronises the device) into
 * *flags, and clears them when reset != 0.  Not part of the pages' interface: it reports
 * what the kernels skipped instead of faulting. */
PA_API pa_status pa_get_device_errors(uint32_t* flags, int reset);

/* Timing hook (not part of the pages' interface): while begin and end are non-NULL, every
 * pa_v2_decode call records `begin` on its stream just before the phase-1 kernel launch and
 * `end` just after it, and every pa_prefix call does the same around its attention kernel
 * (not the combine of split contexts), so a caller can time that kernel alone.  Pass NULL,
 * NULL to stop.  Process-wide and not thread-safe. */
PA_API pa_status pa_v2_set_timing_events(cudaEvent_t begin, cudaEvent_t end);

/*
 * pa_v2_decode_noalloc -- pa_v2_decode for callers that cannot allocate device memory.
 *
 * Not part of the pages' interface (the paper has no counterpart); it exists for callers
 * that are handed a stream but no allocator: an inference runtime that runs this library as
 * a plugin with a device-memory budget fixed at start-up, or an embedded or real-time
 * service that must not grow its footprint after initialisation.  Such a caller cannot provide the exp_sums,
 * max_logits and tmp_output workspace that pa_v2_decode needs.
 *
 * Same computation and the same output as pa_v2_decode (argument meanings and layouts as
 * there, with max_num_partitions = ceil(max_seq_len / 512) and tmp_dtype = PA_DT_F32).
 * The workspace lives in a fixed array of PA_NOALLOC_SCRATCH_BYTES in device memory that
 * the library defines at file scope: every GPU that loads the library holds it until the
 * process exits.  This call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and later calls reuse it; the call works
 * on the current device, so make the device of the pointers current.  A device reset
 * (cudaDeviceReset, or the primary context destroyed and created again) moves the array, and
 * the address looked up before it is then stale: do not call this entry point again in a
 * process after resetting a device it ran on.  The partition statistics a caller of
 * pa_v2_decode would receive are not returned.
 *
 * Errors: as pa_v2_decode, plus PA_ERR_SCRATCH_TOO_SMALL when
 *   2 * align256(S*H*P*4) + S*H*P*head_size*4 > PA_NOALLOC_SCRATCH_BYTES,
 *   P = ceil(max_seq_len / 512)
 * (for example 64 sequences x 32 heads x head_size 128 up to 16K tokens, or 4 x 24 heads x
 * 256 at 100K tokens, fit).  The PA_CHECK host check is not performed (it would allocate
 * host memory).
 *
 * Concurrency: every call on a device shares the one array, which keeps whatever the last
 * call left there (every entry a call reads is written by that same call first, so no
 * clearing is needed).  Calls that can overlap on the GPU -- on different streams, or from
 * different threads without ordering -- race on it and may return wrong results: order them
 * on one stream or use pa_v2_decode with a workspace per stream.
 */
PA_API pa_status pa_v2_decode_noalloc(void* output, const void* query, const void* key_cache,
                                      const void* value_cache, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_size, float scale,
                                      const int32_t* block_tables, int max_blocks_per_seq,
                                      int num_blocks, const int32_t* seq_lens, int block_size,
                                      int max_seq_len, const float* alibi_slopes,
                                      pa_dtype q_dtype, pa_kv_cache_dtype kv_cache_dtype,
                                      float k_scale, float v_scale, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_V2_H_ */
