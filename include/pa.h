/*
 * pa.h -- C ABI of the paged-KV attention step for GB300 (sm_103a).
 *
 * One engine step's attention over a flattened, variable-length batch that
 * mixes prompt chunks and single-token decodes, against a paged KV cache:
 *
 *   pa_prepare_inputs  the per-step index tensors (request of each token,
 *                      positions, query_start_loc, seq_lens, slot_mapping,
 *                      logits_indices);
 *   pa_prepare_inputs_ex  the same plus input_ids (gathered through
 *                      token_indices), the discard mask and the sampled rows
 *                      of speculative decoding;
 *   pa_cache_write     each new token's K and V copied to its cache slot;
 *   pa_prepare_and_write  pa_prepare_inputs and pa_cache_write in one launch;
 *   pa_copy_blocks / pa_zero_blocks  whole-block copy-on-write copies and
 *                      the zeroing of newly allocated blocks;
 *   pa_attention       causal grouped-query attention of every token over
 *                      its own request's context, read through the block
 *                      table;
 *   pa_cache_write_ex / pa_attention_ex  the same over FP8 (E4M3) pools;
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and owns every buffer.  The library
 *     allocates nothing per call.  Its device state is file-scope device
 *     variables: one status word per device, and the fixed scratch array
 *     that only pa_attention_noalloc uses (below).
 *   - Pointers named "device" are CUDA device pointers (any memory a kernel
 *     can dereference); sizes and scalars are host values.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *     return value reports host-side argument checks and launch errors only:
 *       PA_OK               queued;
 *       PA_ERR_INVALID      an argument is malformed; nothing was launched;
 *       PA_ERR_UNSUPPORTED  well-formed but outside what the kernels handle
 *                           (e.g. head_dim not 64/128); nothing launched;
 *       PA_ERR_CUDA         a CUDA runtime call failed.
 *     Checks that need the data (a request with zero scheduled tokens, a
 *     block id outside the pool, a logical block past the table's width, a
 *     slot outside the pool, a wait inside a kernel that ran out) are made
 *     by the kernels, which skip the offending item and record the failure
 *     in the device status word; pa_get_status() reads and clears it.  A
 *     failed check never turns into an out-of-bounds access.
 *   - Ordering: calls on one stream run in order, so pa_cache_write followed
 *     by pa_attention on the same stream reads the freshly written K/V.
 *   - Index tensors are int32.  Q/K/V/output elements are bf16 or fp16.
 *   - KV cache layout: separate K and V pools, each contiguous
 *     [num_blocks][block_size][num_kv_heads][head_dim]; element
 *     (slot, h, d) of a pool is at ((slot * num_kv_heads) + h) * head_dim + d
 *     with slot = physical_block * block_size + offset.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; declared here so the header needs
 * no CUDA include. */
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,
    PA_ERR_CUDA = 2,
    PA_ERR_UNSUPPORTED = 3,
    PA_ERR_DEVICE_CHECK = 4,
    PA_ERR_TIMEOUT = 5,
    PA_ERR_WORKSPACE = 6
} pa_status;

/* Element types.  PA_FP8_E4M3 (the OCP E4M3 "fn" format: bias 7, no
 * infinities, largest finite 448) is a cache element type only: q, k, v and
 * out stay bf16 or fp16. */
typedef enum { PA_BF16 = 0, PA_FP16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Bits of the detail word returned by pa_get_status(). */
enum {
    PA_CHECK_EMPTY_REQUEST = 1u << 0,  /* num_scheduled_tokens[r] <= 0 */
    PA_CHECK_TOKEN_COUNT = 1u << 1,    /* sum(num_scheduled_tokens) != num_tokens,
                                          or query_start_loc[num_reqs] != num_tokens */
    PA_CHECK_BLOCK_ID = 1u << 2,       /* block_table entry outside [0, num_blocks) */
    PA_CHECK_LOGICAL_BLOCK = 1u << 3,  /* position / block_size >= max_blocks_per_req */
    PA_CHECK_SLOT = 1u << 4,           /* slot_mapping entry >= num_blocks * block_size */
    PA_CHECK_SEQ_LEN = 1u << 5,        /* seq_lens[r] < query length, qsl decreasing, a
                                          context wider than the table, or (attention)
                                          seq_lens[r] > max_seq_len */
    PA_CHECK_TIMEOUT = 1u << 6,        /* a bounded wait inside a kernel ran out */
    PA_CHECK_TOKEN_INDEX = 1u << 7,    /* a token's position >= max_model_len (its id
                                          would come from another request's row) */
    PA_CHECK_DRAFT_COUNT = 1u << 8     /* num_draft_tokens[r] < 0 or >=
                                          num_scheduled_tokens[r], or num_reqs +
                                          sum(num_draft_tokens) != num_logits */
};

/*
 * pa_prepare_inputs -- the step's index tensors.
 *
 * Defined by "Building the Batch", sections "How they are computed" and
 * "Reading and writing the KV cache" (and its Go program), and by "vLLM's
 * Model Runner", section "The two things this method returns":
 *   query_start_loc[0] = 0, query_start_loc[r+1] = query_start_loc[r] + nst[r];
 *   entries past num_reqs, up to qsl_capacity, hold num_tokens (so the
 *   array never decreases);
 *   for token t of request r at offset i (t = query_start_loc[r] + i):
 *     req_indices[t]  = r
 *     positions[t]    = num_computed_tokens[r] + i
 *     slot_mapping[t] = block_table[r][pos / block_size] * block_size
 *                       + pos % block_size
 *   seq_lens[r]       = num_computed_tokens[r] + num_scheduled_tokens[r]
 *   logits_indices[r] = query_start_loc[r+1] - 1
 *
 * Arguments (all device pointers are int32):
 *   num_scheduled_tokens [num_reqs]   tokens each request runs this step (>= 1)
 *   num_computed_tokens  [num_reqs]   tokens already in the cache (>= 0)
 *   block_table [num_reqs][max_blocks_per_req] row-major physical block ids
 *   block_size           tokens per cache block (> 0)
 *   num_tokens           T = sum(num_scheduled_tokens), known to the host
 *   num_blocks           physical blocks in the pool (ids are checked against it)
 *   req_indices, positions, slot_mapping   outputs [num_tokens]
 *   query_start_loc      output [qsl_capacity], qsl_capacity >= num_reqs + 1
 *   seq_lens, logits_indices               outputs [num_reqs]
 * Errors: PA_ERR_INVALID for negative sizes, a NULL buffer with a non-zero
 * size, qsl_capacity < num_reqs + 1, or num_blocks * block_size >= 2^31;
 * PA_ERR_UNSUPPORTED for more than 50,000 requests.
 * Data checks (status word): PA_CHECK_EMPTY_REQUEST, PA_CHECK_TOKEN_COUNT,
 * PA_CHECK_LOGICAL_BLOCK, PA_CHECK_BLOCK_ID; a token whose block fails a
 * check gets slot_mapping = -1.
 */
pa_status pa_prepare_inputs(const int32_t *num_scheduled_tokens,
                            const int32_t *num_computed_tokens,
                            const int32_t *block_table, int32_t num_reqs,
                            int32_t max_blocks_per_req, int32_t block_size,
                            int32_t num_tokens, int32_t num_blocks,
                            int32_t *req_indices, int32_t *positions,
                            int32_t *slot_mapping, int32_t *query_start_loc,
                            int32_t qsl_capacity, int32_t *seq_lens,
                            int32_t *logits_indices, pa_stream_t stream);

/*
 * pa_prepare_and_write -- pa_prepare_inputs and pa_cache_write_ex in one
 * launch.
 *
 * "How vLLM Works Internally", section "Fused Kernels" (one launch instead
 * of two, and no round trip of slot_mapping through global memory between
 * them), applied to "Building the Batch", section "How they are computed"
 * (the index tensors) and "Inside vLLM: Following One Request", the write op
 * (token t's K and V rows to slot_mapping[t]).  The outputs are bit for bit
 * those of pa_prepare_inputs followed, on the same stream, by
 * pa_cache_write_ex with the slot_mapping it produced: every index tensor,
 * and every pool row written (16-bit pools: a copy; PA_FP8_E4M3 pools:
 * E4M3(x / scale)).  A token whose slot fails a check (slot_mapping -1) is
 * not written, as a negative slot is skipped by pa_cache_write.
 *
 * Arguments: those of pa_prepare_inputs, then key, value [num_tokens] rows
 * of num_kv_heads * head_dim elements kv_token_stride elements apart (16-byte
 * aligned rows), the pools (layout as pa_cache_write; 16-byte aligned rows,
 * 8-byte for FP8 pools), num_kv_heads, head_dim, dtype (of key/value),
 * cache_dtype (dtype or PA_FP8_E4M3) and the FP8 scales (device scalars,
 * NULL = 1.0; ignored for 16-bit pools).  The pools hold
 * num_blocks * block_size slots.
 * Errors: those of pa_prepare_inputs and pa_cache_write_ex; PA_ERR_UNSUPPORTED
 * also when a row or base address is not aligned as above (the two separate
 * calls take any alignment).  Data checks as pa_prepare_inputs.
 */
pa_status pa_prepare_and_write(const int32_t *num_scheduled_tokens,
                               const int32_t *num_computed_tokens, const int32_t *block_table,
                               int32_t num_reqs, int32_t max_blocks_per_req, int32_t block_size,
                               int32_t num_tokens, int32_t num_blocks, int32_t *req_indices,
                               int32_t *positions, int32_t *slot_mapping,
                               int32_t *query_start_loc, int32_t qsl_capacity, int32_t *seq_lens,
                               int32_t *logits_indices, const void *key, const void *value,
                               int64_t kv_token_stride, void *key_cache, void *value_cache,
                               int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype,
                               pa_dtype cache_dtype, const float *k_scale, const float *v_scale,
                               pa_stream_t stream);

/*
 * pa_prepare_inputs_ex -- pa_prepare_inputs plus the rest of the step's
 * input preparation, in the same single launch.
 *
 * Defined by "Building the Batch", sections "How they are computed" (token
 * ids gathered through token_indices = positions + req_indices * M) and
 * "Only one row per request reaches the vocabulary" (with speculative
 * decoding a request needs one row per draft token plus one), and by "vLLM's
 * Model Runner", sections "Flattening the batch into one token axis", "The
 * two things this method returns" and "The batch contains rows that must not
 * be sampled" (the discard mask).  Everything pa_prepare_inputs computes is
 * computed identically; in addition, each optional group below runs when its
 * pointers are given:
 *
 *   token-id gather (max_model_len > 0):
 *     token_ids is the per-request token buffer [max_num_reqs][max_model_len]
 *     (int32, row-major; row r holds batch row r's ids).  It may be device
 *     memory or host memory the device can read (page-locked host memory
 *     from cudaHostAlloc / cudaMallocHost, or pageable memory on systems
 *     whose devices report pageable-memory access).
 *       token_indices[t] = positions[t] + req_indices[t] * max_model_len  (int64)
 *       input_ids[t]     = token_ids[token_indices[t]]
 *     A token whose position is >= max_model_len gets -1 in both and sets
 *     PA_CHECK_TOKEN_INDEX.
 *   discard mask (request_num_tokens != NULL):
 *     discard_request_mask[r] = (num_computed_tokens[r] + num_scheduled_tokens[r]
 *                                < request_num_tokens[r])   (one byte, 0 or 1)
 *     request_num_tokens[r] is the request's total known token count
 *     (prompt plus output so far).
 *   sampled rows:
 *     num_draft_tokens == NULL: num_logits must equal num_reqs, and
 *       logits_indices[r] = query_start_loc[r+1] - 1 (as pa_prepare_inputs);
 *     otherwise, with d = num_draft_tokens[r], request r owns the d + 1
 *       entries cu_num_logits[r] .. cu_num_logits[r+1] - 1 of logits_indices,
 *       cu_num_logits being the exclusive scan of (num_draft_tokens + 1), and
 *       logits_indices[cu_num_logits[r] + k] = query_start_loc[r+1] - 1 - d + k,
 *       k = 0..d: the last d + 1 rows of its slice.  num_logits must be
 *       num_reqs + sum(num_draft_tokens) (known to the host); a mismatch or a
 *       draft count outside [0, num_scheduled_tokens[r]) sets
 *       PA_CHECK_DRAFT_COUNT and no row past num_logits is written.
 *     cu_num_logits [num_reqs + 1] is optional (NULL skips it).
 *
 * Errors: as pa_prepare_inputs, plus PA_ERR_INVALID when a group is half
 * given (max_model_len > 0 without token_ids, or without token_indices /
 * input_ids while num_tokens > 0; max_model_len == 0 with any of the three;
 * request_num_tokens
 * without discard_request_mask or the reverse), max_num_reqs < num_reqs,
 * max_model_len < 0, num_logits != num_reqs without drafts, num_logits < 0,
 * or a token buffer the current device cannot read.
 */
pa_status pa_prepare_inputs_ex(const int32_t *num_scheduled_tokens,
                               const int32_t *num_computed_tokens,
                               const int32_t *block_table, int32_t num_reqs,
                               int32_t max_blocks_per_req, int32_t block_size,
                               int32_t num_tokens, int32_t num_blocks,
                               const int32_t *token_ids, int32_t max_num_reqs,
                               int32_t max_model_len,
                               const int32_t *request_num_tokens,
                               const int32_t *num_draft_tokens, int32_t num_logits,
                               int32_t *req_indices, int32_t *positions,
                               int32_t *slot_mapping, int32_t *query_start_loc,
                               int32_t qsl_capacity, int32_t *seq_lens,
                               int64_t *token_indices, int32_t *input_ids,
                               uint8_t *discard_request_mask,
                               int32_t *logits_indices, int32_t *cu_num_logits,
                               pa_stream_t stream);

/*
 * pa_cache_write -- scatter the step's new K and V into the cache.
 *
 * Defined by "Inside vLLM: Following One Request", the section on the write
 * op (reshape_and_cache_flash): for token i, its key and value vectors are
 * copied to slot slot_mapping[i].  A bit copy: no conversion, no scaling.
 *
 * Arguments:
 *   key, value        device [num_tokens][num_kv_heads][head_dim] elements,
 *                     token rows kv_token_stride elements apart (>= Hkv*D;
 *                     lets K and V be views of a fused QKV projection)
 *   key_cache, value_cache  device pools, layout above
 *   slot_mapping      device int32 [num_tokens]; a negative slot means the
 *                     token writes nothing (a padding row)
 *   block_size, num_blocks  pool geometry (slots = num_blocks * block_size)
 *   dtype             element type of all four buffers
 * Errors: PA_ERR_INVALID for non-positive head counts/sizes, NULL buffers
 * with num_tokens > 0, or kv_token_stride < num_kv_heads * head_dim.
 * Data check: PA_CHECK_SLOT (that token is skipped).
 */
pa_status pa_cache_write(const void *key, const void *value, int64_t kv_token_stride,
                         void *key_cache, void *value_cache,
                         const int32_t *slot_mapping, int32_t num_tokens,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_blocks, pa_dtype dtype, pa_stream_t stream);

/*
 * pa_cache_write_ex -- pa_cache_write into pools of another element type.
 *
 * Defined by "Inside vLLM: Following One Request", the write op's
 * kv_cache_dtype, k_scale and v_scale arguments, and "How vLLM Works
 * Internally", section "FP8 KV Cache" (the cache may hold FP8 instead of
 * 16-bit values).  cache_dtype == dtype: exactly pa_cache_write.
 * cache_dtype == PA_FP8_E4M3: the pools hold one byte per element, and
 *   key_cache[slot][h][d] = E4M3(key[t][h][d] / *k_scale)
 *   value_cache[slot][h][d] = E4M3(value[t][h][d] / *v_scale)
 * with the division in IEEE single precision and E4M3() rounding to nearest,
 * ties to even, magnitudes past 448 saturating to +-448 (NaN stays NaN).
 * k_scale / v_scale are device pointers to one float each (> 0); NULL means
 * 1.0.  The 16-bit sources need 16-byte aligned rows and token stride, the
 * pools 8-byte aligned rows (else PA_ERR_UNSUPPORTED).  Other arguments and
 * errors as pa_cache_write.
 */
pa_status pa_cache_write_ex(const void *key, const void *value, int64_t kv_token_stride,
                            void *key_cache, void *value_cache, const int32_t *slot_mapping,
                            int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                            pa_dtype cache_dtype, const float *k_scale, const float *v_scale,
                            pa_stream_t stream);

/*
 * pa_copy_blocks -- copy-on-write: make whole cache blocks copies of others.
 *
 * Defined by "How vLLM Works Internally", section "Copy-on-Write for Beam
 * Search", step 3 (the old block's contents are copied to the newly
 * allocated block).  Steps 1, 2, 4 and 5 (reference counts, allocation, the
 * block-table update) are the block manager's, on the host.
 *   for i in [0, num_pairs): block dst_blocks[i] of the K pool and of the V
 *   pool becomes a byte copy of block src_blocks[i] of the same pool
 *   (block_size * num_kv_heads * head_dim elements each).
 * The destinations must be distinct and none may be a source (they are new
 * blocks); otherwise the contents of the overlapping blocks are unspecified
 * (every access still stays inside the pools).
 *
 * Arguments: key_cache, value_cache device pools as in pa_cache_write
 * (16-byte aligned); src_blocks, dst_blocks device int32 [num_pairs].
 * dtype is the pools' element type (PA_BF16, PA_FP16 or PA_FP8_E4M3).
 * Errors: PA_ERR_INVALID for negative sizes, NULL buffers with num_pairs > 0,
 * unaligned pools or a bad dtype; PA_ERR_UNSUPPORTED when a block is not a
 * multiple of 16 bytes.  Data check: PA_CHECK_BLOCK_ID (that pair skipped).
 */
pa_status pa_copy_blocks(void *key_cache, void *value_cache, const int32_t *src_blocks,
                         const int32_t *dst_blocks, int32_t num_pairs, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                         pa_dtype dtype, pa_stream_t stream);

/*
 * pa_zero_blocks -- clear newly allocated cache blocks.
 *
 * Defined by "Inside vLLM: Following One Request", the scheduler output's
 * new_block_ids_to_zero: blocks that must be cleared before the forward pass
 * so that stale data or NaNs of an earlier owner cannot reach attention.
 *   every byte of block block_ids[i] of both pools becomes 0 (+0.0).
 * Arguments and errors as pa_copy_blocks; block_ids device int32 [num_ids].
 */
pa_status pa_zero_blocks(void *key_cache, void *value_cache, const int32_t *block_ids,
                         int32_t num_ids, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, int32_t num_blocks, pa_dtype dtype,
                         pa_stream_t stream);

/*
 * pa_attention_workspace_size -- bytes of workspace that let pa_attention
 * split every request's context into its preferred number of partitions
 * and, over bf16 pools at head_dim 128, convert the V of the requests with
 * more than 16 query tokens to f16 once (for up to 64 MiB of it) instead of
 * once per 256-row tile inside the tensor-core kernel.  The workspace is
 * laid out as 256 bytes of item counters, the split-K partials, then that
 * copy.  Any smaller workspace (including 0) is still correct and gives the
 * same prefill rows bit for bit: requests the copy has no room for are
 * converted in the kernel, the split-K kernel uses longer partitions so the
 * partial results fit (less parallelism for long contexts), and without
 * the first 256 bytes both kernels take their work items in a fixed order
 * instead of as their CTAs free up.  Arguments are host-known bounds of the
 * step.
 */
size_t pa_attention_workspace_size(int32_t num_reqs, int32_t num_tokens,
                                   int32_t max_query_len, int32_t max_seq_len,
                                   int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim);

/*
 * pa_attention -- paged causal grouped-query attention for the flat batch.
 *
 * Defined by "How vLLM Works Internally", section "How the Kernel Works"
 * (look up the block table, fetch K from the scattered blocks, scores,
 * softmax, weighted sum of V; the two-pass variant reduces partial softmax
 * results across partitions) and "Inside vLLM: Following One Request", the
 * read path (cu_seqlens_q = query_start_loc, seqused_k = seq_lens,
 * physical block = block_table[logical block]).  For token t of request r
 * at offset i, with n = query_start_loc[r+1] - query_start_loc[r] and
 * position p = seq_lens[r] - n + i, and q head h reading kv head
 * g = h / (num_q_heads / num_kv_heads):
 *     out[t][h] = sum_{j <= p} softmax_j(scale * q[t][h] . K_r[j][g]) V_r[j][g]
 * where K_r[j] is the cache entry at block_table[r][j / block_size],
 * offset j % block_size.  Accumulation is fp32 and the output is rounded
 * once to the element type.  The softmax weights enter the weighted sum of
 * V with at least 11 significant bits.  On the split-K kernel they are f16
 * over fp16 and FP8 pools, and two bf16 terms over bf16 pools (the weight
 * rounded, then the remainder rounded: 16 significant bits).  On the
 * tensor-core kernel they are f16, with V converted to f16 first: exactly,
 * apart from values below f16's normal range, which round to its subnormals
 * (an absolute error of at most 2^-25).  A 64-key half of a V tile holding a
 * value that f16 cannot represent keeps bf16 V, and its weights enter as two
 * bf16 terms, exactly.
 *
 * Requests with more than 16 query tokens run on the tensor-core (tcgen05)
 * kernel when num_q_heads / num_kv_heads <= 128 and scale > 0; every other
 * request runs on the split-K kernel.
 *
 * Arguments:
 *   q             device [num_tokens][num_q_heads][head_dim], contiguous
 *   key_cache, value_cache  device pools (layout above), already holding
 *                 this step's K/V (pa_cache_write first, same stream)
 *   block_table   device int32 [num_reqs][max_blocks_per_req]
 *   query_start_loc device int32 [num_reqs + 1]; seq_lens device int32 [num_reqs]
 *   max_query_len, max_seq_len  host upper bounds of q length / seq_lens (a
 *                 request with seq_lens[r] > max_seq_len is flagged
 *                 PA_CHECK_SEQ_LEN and left out)
 *   head_dim      64 or 128; block_size 16; num_q_heads % num_kv_heads == 0
 *   scale         softmax scale (usually 1/sqrt(head_dim))
 *   out           device [num_tokens][num_q_heads][head_dim]
 *   workspace     device scratch of workspace_bytes (256-byte aligned when
 *                 non-zero); contents need no initialisation and are
 *                 overwritten.  Calls that share a workspace must not
 *                 overlap on the GPU.
 * Errors: PA_ERR_INVALID (NULL buffers, bad sizes, misaligned buffers),
 * PA_ERR_UNSUPPORTED (head_dim, block_size, head ratio, a pool too large for
 * 32-bit slots).  Data checks: PA_CHECK_SEQ_LEN, PA_CHECK_BLOCK_ID (the
 * request is skipped, or its block replaced by block 0), PA_CHECK_TIMEOUT.
 */
pa_status pa_attention(const void *q, const void *key_cache, const void *value_cache,
                       const int32_t *block_table, int32_t max_blocks_per_req,
                       const int32_t *query_start_loc, const int32_t *seq_lens,
                       int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                       int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks,
                       float scale, pa_dtype dtype, void *out, void *workspace,
                       size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_ex -- pa_attention over pools of another element type.
 *
 * Defined as pa_attention, with the cached values read as in "How vLLM Works
 * Internally", section "FP8 KV Cache": cache_dtype == dtype is exactly
 * pa_attention; cache_dtype == PA_FP8_E4M3 reads one-byte E4M3 pools whose
 * cached key is element * *k_scale and cached value element * *v_scale
 * (device scalars; NULL = 1.0).  Requests go to the same two kernels as in
 * pa_attention (more than 16 query tokens: the tcgen05 kernel; the rest: the
 * split-K kernel); over FP8 pools both run their MMAs in f16 (E4M3 widens to
 * f16 exactly; bf16 q is rounded to f16, exact inside f16's range; the
 * softmax weights are f16).  The output is dtype.  Errors as
 * pa_attention, plus PA_ERR_INVALID for a cache_dtype that is neither dtype
 * nor PA_FP8_E4M3.
 *
 * flags: 0, or PA_ATTN_SHARED_BLOCKS (any other bit: PA_ERR_INVALID).
 * PA_ATTN_SHARED_BLOCKS declares that block tables may hold the same
 * physical block for several requests -- the copy-on-write sharing of "How
 * vLLM Works Internally", section "Copy-on-Write for Beam Search", or a
 * prefix reused by "Prefix Caching (Automatic Prefix Caching)".  Results are
 * the same with or without it.  With it, consecutive single-token requests
 * whose tables hold the same blocks over a whole KV partition (512 keys
 * with the workspace pa_attention_workspace_size() asks for) that their
 * query sees completely -- up to 32 / (num_q_heads / num_kv_heads) such
 * requests -- are computed together, reading those blocks once.  Without it
 * the kernel carries no code for this (a few percent faster when nothing is
 * shared).  The flag takes effect when a workspace is given and some context
 * is longer than one partition.
 */
#define PA_ATTN_SHARED_BLOCKS 1u
pa_status pa_attention_ex(const void *q, const void *key_cache, const void *value_cache,
                          const int32_t *block_table, int32_t max_blocks_per_req,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                          int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                          pa_dtype dtype, pa_dtype cache_dtype, const float *k_scale,
                          const float *v_scale, uint32_t flags, void *out, void *workspace,
                          size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_attention_noalloc -- pa_attention for callers that cannot allocate.
 *
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory when they call in -- an engine that has
 * given nearly all free HBM to its KV-cache pool, a decode loop where
 * cudaMalloc/cudaFree would synchronise the device, or a host program that
 * reaches this library through the C ABI with no device allocator of its
 * own.  Same inputs, outputs and results as pa_attention; the workspace is
 * a fixed PA_NOALLOC_SCRATCH_BYTES array in the library's own device memory
 * (every GPU that loads the library holds it until the process exits), and
 * the call itself allocates nothing.
 *   - Limit: num_reqs <= PA_NOALLOC_MAX_REQS, else PA_ERR_WORKSPACE and
 *     nothing is launched.  Long contexts are still handled: with less
 *     scratch than pa_attention_workspace_size() asks for, the kernel uses
 *     longer KV partitions.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept per device and per
 *     CUDA context (a context of one's own on the same device has its own
 *     copy of the array and is looked up on its first call).  A device reset
 *     (cudaDeviceReset) destroys the array with its context: the library
 *     does not support calls on a device after it was reset.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; nothing needs clearing (each call writes what it
 *     reads), but calls that overlap on the GPU (different streams, or
 *     threads without ordering) race on it and must be serialised.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
#define PA_NOALLOC_MAX_REQS 65536
pa_status pa_attention_noalloc(const void *q, const void *key_cache, const void *value_cache,
                               const int32_t *block_table, int32_t max_blocks_per_req,
                               const int32_t *query_start_loc, const int32_t *seq_lens,
                               int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                               int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int32_t num_blocks,
                               float scale, pa_dtype dtype, void *out, pa_stream_t stream);

/*
 * pa_get_status -- synchronise `stream`, then read and clear the current
 * device's status word.  Returns PA_OK when no kernel check failed since the
 * last call, PA_ERR_TIMEOUT when a bounded wait ran out, PA_ERR_DEVICE_CHECK
 * for any other failed check, PA_ERR_CUDA if the synchronisation failed.
 * When `detail` is non-NULL it receives the PA_CHECK_* bits.
 */
pa_status pa_get_status(pa_stream_t stream, uint32_t *detail);

/*
 * pa_selftest_wait_timeout -- diagnostic.  Launches one small kernel that
 * takes the library's bounded mbarrier wait on a barrier nothing ever
 * completes.  The wait gives up after its time limit (about one second),
 * the kernel records PA_CHECK_TIMEOUT and returns; the next pa_get_status()
 * then reports PA_ERR_TIMEOUT and the context stays usable.  No counterpart
 * on the pages: it checks this library's own failure handling.
 */
pa_status pa_selftest_wait_timeout(pa_stream_t stream);

/* A static, human-readable name for a status code. */
const char *pa_status_string(pa_status s);

/* Number of the library's kernel launches queued by this thread since the
 * last call to this function (returns and resets the count). */
uint64_t pa_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
