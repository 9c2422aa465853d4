/*
 * Oracle for one paged-KV attention step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the step computes.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this library; the CUDA library never links, includes or calls it, and it
 * shares no code with the CUDA library.  Floating point is fp64 throughout.
 *
 * The functions, each citing the passage it follows:
 *
 *   oracle_prepare_inputs  -- the per-step index tensors
 *       ("Building the Batch", sections "How they are computed" and
 *        "Reading and writing the KV cache": req_indices, query positions,
 *        positions = num_computed + offset, query_start_loc with its tail
 *        padded by the total, slot = block_table[pos / bs] * bs + pos % bs,
 *        logits_indices = query_start_loc[1:] - 1; and the same page's Go
 *        program, which builds the tensors with one loop over requests and
 *        one over each request's scheduled tokens).
 *   oracle_gather_input_ids -- "Building the Batch", section "How they are
 *        computed" (token_indices = positions + req_indices * M, M the width
 *        of the per-request token buffer, then one index_select of the
 *        flattened buffer) and "vLLM's Model Runner", section "Flattening
 *        the batch into one token axis".
 *   oracle_discard_request_mask -- "vLLM's Model Runner", sections "The two
 *        things this method returns" and "The batch contains rows that must
 *        not be sampled": optimistic seq len = computed + scheduled; a
 *        request's sample is discarded when that is below its total token
 *        count.
 *   oracle_spec_logits_indices -- "Building the Batch", section "Only one row
 *        per request reaches the vocabulary": without drafts one row per
 *        request, query_start_loc[1:] - 1; with d draft tokens a request
 *        needs d + 1 rows, read as the last d + 1 rows of its slice.
 *   oracle_copy_blocks     -- "How vLLM Works Internally", section
 *        "Copy-on-Write for Beam Search", step 3: the old block's contents
 *        are copied to the newly allocated one (every slot, every head, both
 *        the K and the V pool).  A byte copy.
 *   oracle_zero_blocks     -- "Inside vLLM: Following One Request", the
 *        scheduler output's new_block_ids_to_zero: freshly allocated blocks
 *        are cleared before the forward pass.  Every byte of the block, in
 *        both pools, becomes 0.
 *   oracle_e4m3_decode / oracle_e4m3_encode -- the FP8 E4M3 format
 *        ("How vLLM Works Internally", section "FP8 KV Cache": the cache may
 *        hold FP8 instead of FP16), written from the format's definition:
 *        decode exactly; encode by round to nearest, ties to even, with
 *        saturation to +-448.
 *   oracle_cache_write_fp8 -- the write op with kv_cache_dtype FP8 ("Inside
 *        vLLM: Following One Request", reshape_and_cache_flash's
 *        kv_cache_dtype, k_scale, v_scale): element / scale in single
 *        precision, then E4M3.
 *   oracle_attention_ex    -- oracle_attention over pools of any element
 *        type: the cached value is pool element * k_scale (or v_scale).
 *   oracle_cache_write     -- "Inside vLLM: Following One Request", section
 *        on reshape_and_cache_flash: token i's K and V are copied to slot
 *        slot_mapping[i].  A bit copy.
 *   oracle_attention       -- "How vLLM Works Internally", section "How the
 *        Kernel Works" (look up the block table, fetch K from the scattered
 *        blocks, scores, softmax, weighted sum of V) and "Inside vLLM", the
 *        CPU read loop (physical = block_table[logical]).  Each request's K/V
 *        is gathered into a contiguous buffer through its block table, then
 *        dense causal softmax attention runs in fp64.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - causal: query token at position p sees keys 0..p of its own request,
 *     itself included; its position is seq_len - q_len + offset.
 *   - grouped-query heads: q head h reads kv head h / (Hq / Hkv).
 *   - cache layout: separate K and V pools, each [num_blocks][block_size]
 *     [num_kv_heads][head_dim], so element (slot, h, d) is at
 *     (slot * Hkv + h) * D + d.
 *   - a negative slot means "no write" for that token.
 *   - a request must schedule at least one token.
 *   - FP8 cache: E4M3 with one scale per pool (k_scale, v_scale); the write
 *     stores round(x / scale) and a read returns element * scale.
 *
 * Return value: 0 on success, a negative number when an input breaks the
 * problem's rules (the outputs for the offending items are then unspecified).
 */
#define _POSIX_C_SOURCE 200809L
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_BF16 0
#define ORACLE_FP16 1
#define ORACLE_FP8_E4M3 2

/* ------------------------------------------------------------------------ */
/* Element decoding: the raw 16-bit patterns of bf16 / IEEE half to double.  */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b)
{
    /* bf16 is the upper half of an IEEE single. */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* zero / subnormal */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant + 1024), expo - 25);  /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

static double elem(uint16_t x, int dtype)
{
    return dtype == ORACLE_FP16 ? fp16_to_double(x) : bf16_to_double(x);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (the OCP "fn" variant: 1 sign, 4 exponent bits with bias 7, 3    */
/* mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448).     */
/* ------------------------------------------------------------------------ */

static double e4m3_to_double(uint8_t b)
{
    int sign = b >> 7;
    int expo = (b >> 3) & 0xf;
    int mant = b & 7;
    double v;
    if (expo == 15 && mant == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)mant, -9);                  /* 2^-6 * m/8 */
    else
        v = ldexp((double)(8 + mant), expo - 10);     /* 2^(e-7) * (1 + m/8) */
    return sign ? -v : v;
}

/* Round a float to the nearest E4M3 value, ties to the even mantissa;
 * magnitudes past the largest finite value give +-448 (saturation), NaN gives
 * the NaN code. */
static uint8_t float_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the first normal */
        double units = nearbyint(a * 512.0);
        return sign | (uint8_t)units;
    }
    int e2;
    frexp(a, &e2);                  /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                 /* a in [2^e, 2^(e+1)) */
    double steps = nearbyint(ldexp(a, 3 - e));     /* in [8, 16] */
    if (steps == 16.0) {
        steps = 8.0;
        e += 1;
    }
    return sign | (uint8_t)(((e + 7) << 3) | ((int)steps - 8));
}

/* Pool element `i` of a cache in `cache_dtype` (bf16, fp16, or fp8 e4m3). */
static double cache_elem(const void *pool, int64_t i, int cache_dtype)
{
    if (cache_dtype == ORACLE_FP8_E4M3)
        return e4m3_to_double(((const uint8_t *)pool)[i]);
    return elem(((const uint16_t *)pool)[i], cache_dtype);
}

int oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_to_double(codes[i]);
    return 0;
}

int oracle_e4m3_encode(const float *x, int64_t n, uint8_t *codes)
{
    for (int64_t i = 0; i < n; ++i)
        codes[i] = float_to_e4m3(x[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Index build                                                               */
/* ------------------------------------------------------------------------ */

int oracle_prepare_inputs(const int32_t *num_scheduled_tokens,
                          const int32_t *num_computed_tokens,
                          const int32_t *block_table, int32_t num_reqs,
                          int32_t max_blocks_per_req, int32_t block_size,
                          int32_t num_tokens, int32_t num_blocks,
                          int32_t *req_indices, int32_t *positions,
                          int32_t *slot_mapping, int32_t *query_start_loc,
                          int32_t qsl_capacity, int32_t *seq_lens,
                          int32_t *logits_indices)
{
    int err = 0;
    if (num_reqs < 0 || block_size <= 0 || num_tokens < 0 || qsl_capacity < num_reqs + 1)
        return -1;
    query_start_loc[0] = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t n = num_scheduled_tokens[r];
        int32_t c = num_computed_tokens[r];
        if (n <= 0 || c < 0) {
            err = -2;
            n = n < 0 ? 0 : n;
        }
        query_start_loc[r + 1] = query_start_loc[r] + n;
        seq_lens[r] = c + n;
        logits_indices[r] = query_start_loc[r + 1] - 1;
        for (int32_t i = 0; i < n; ++i) {
            int32_t t = query_start_loc[r] + i;
            if (t >= num_tokens) {          /* more scheduled tokens than T */
                err = -3;
                break;
            }
            int32_t pos = c + i;
            int32_t logical = pos / block_size;
            req_indices[t] = r;
            positions[t] = pos;
            if (logical >= max_blocks_per_req) {
                err = -4;
                slot_mapping[t] = -1;
                continue;
            }
            int32_t phys = block_table[(int64_t)r * max_blocks_per_req + logical];
            if (phys < 0 || phys >= num_blocks) {
                err = -5;
                slot_mapping[t] = -1;
                continue;
            }
            slot_mapping[t] = phys * block_size + pos % block_size;
        }
    }
    if (query_start_loc[num_reqs] != num_tokens)
        err = err ? err : -3;
    /* Pad the tail with the total so the array never decreases. */
    for (int32_t i = num_reqs + 1; i < qsl_capacity; ++i)
        query_start_loc[i] = num_tokens;
    return err;
}

/* ------------------------------------------------------------------------ */
/* Token ids, discard mask, sampled rows                                     */
/* ------------------------------------------------------------------------ */

/* The token buffer holds one row of max_model_len ids per request slot, so
 * the id at position p of row r sits at flat offset r * max_model_len + p.
 * Every token of the step is gathered from there in one pass. */
int oracle_gather_input_ids(const int32_t *req_indices, const int32_t *positions,
                            int32_t num_tokens, const int32_t *token_ids,
                            int32_t max_num_reqs, int32_t max_model_len,
                            int64_t *token_indices, int32_t *input_ids)
{
    int err = 0;
    if (num_tokens < 0 || max_num_reqs < 0 || max_model_len <= 0)
        return -1;
    /* Step 1: flat offsets into the [max_num_reqs][max_model_len] buffer. */
    for (int32_t t = 0; t < num_tokens; ++t)
        token_indices[t] = (int64_t)positions[t] + (int64_t)req_indices[t] * max_model_len;
    /* Step 2: index_select of the flattened buffer at those offsets. */
    for (int32_t t = 0; t < num_tokens; ++t) {
        if (req_indices[t] < 0 || req_indices[t] >= max_num_reqs || positions[t] < 0 ||
            positions[t] >= max_model_len) {
            err = -6;            /* the offset would leave its own row */
            token_indices[t] = -1;
            input_ids[t] = -1;
            continue;
        }
        input_ids[t] = token_ids[token_indices[t]];
    }
    return err;
}

int oracle_discard_request_mask(const int32_t *num_computed_tokens,
                                const int32_t *num_scheduled_tokens,
                                const int32_t *request_num_tokens, int32_t num_reqs,
                                uint8_t *discard_request_mask)
{
    if (num_reqs < 0)
        return -1;
    for (int32_t r = 0; r < num_reqs; ++r) {
        /* how long the sequence is once this step has run */
        int64_t optimistic_seq_len =
            (int64_t)num_computed_tokens[r] + (int64_t)num_scheduled_tokens[r];
        discard_request_mask[r] = optimistic_seq_len < (int64_t)request_num_tokens[r];
    }
    return 0;
}

/* Rows of the step's output that get a next-token distribution.  Request r
 * with d[r] draft tokens owns d[r] + 1 consecutive entries, starting at
 * cu_num_logits[r]; they are the last d[r] + 1 rows of its slice
 * [query_start_loc[r], query_start_loc[r+1]).  num_draft_tokens == NULL
 * means no drafts.  cu_num_logits (optional) gets the R + 1 starts. */
int oracle_spec_logits_indices(const int32_t *query_start_loc,
                               const int32_t *num_draft_tokens, int32_t num_reqs,
                               int32_t num_logits, int32_t *logits_indices,
                               int32_t *cu_num_logits)
{
    int err = 0;
    if (num_reqs < 0 || num_logits < 0)
        return -1;
    int32_t row = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t d = num_draft_tokens ? num_draft_tokens[r] : 0;
        int32_t q_len = query_start_loc[r + 1] - query_start_loc[r];
        if (d < 0 || d + 1 > q_len) {
            err = -7;           /* the drafts must be among the scheduled tokens */
            d = d < 0 ? 0 : (q_len > 0 ? q_len - 1 : 0);
        }
        if (cu_num_logits)
            cu_num_logits[r] = row;
        int32_t last = query_start_loc[r + 1] - 1;
        for (int32_t k = 0; k <= d; ++k) {
            if (row >= num_logits) {
                err = -3;
                break;
            }
            logits_indices[row++] = last - d + k;
        }
    }
    if (cu_num_logits)
        cu_num_logits[num_reqs] = row;
    if (row != num_logits)
        err = err ? err : -3;
    return err;
}

/* ------------------------------------------------------------------------ */
/* Whole-block operations: copy-on-write copy, zeroing                       */
/* ------------------------------------------------------------------------ */

/* A block of a pool is block_bytes consecutive bytes starting at
 * block * block_bytes (block_bytes = block_size * num_kv_heads * head_dim *
 * element size).  Pairs are copied in order; the destinations are new
 * blocks, so no destination is also a source. */
int oracle_copy_blocks(uint8_t *key_cache, uint8_t *value_cache, int64_t block_bytes,
                       int32_t num_blocks, const int32_t *src_blocks,
                       const int32_t *dst_blocks, int32_t num_pairs)
{
    int err = 0;
    if (block_bytes <= 0 || num_blocks < 0 || num_pairs < 0)
        return -1;
    for (int32_t i = 0; i < num_pairs; ++i) {
        int32_t s = src_blocks[i], d = dst_blocks[i];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            err = -5;             /* a block outside the pool: that pair is skipped */
            continue;
        }
        for (int64_t b = 0; b < block_bytes; ++b) {
            key_cache[(int64_t)d * block_bytes + b] = key_cache[(int64_t)s * block_bytes + b];
            value_cache[(int64_t)d * block_bytes + b] = value_cache[(int64_t)s * block_bytes + b];
        }
    }
    return err;
}

int oracle_zero_blocks(uint8_t *key_cache, uint8_t *value_cache, int64_t block_bytes,
                       int32_t num_blocks, const int32_t *block_ids, int32_t num_ids)
{
    int err = 0;
    if (block_bytes <= 0 || num_blocks < 0 || num_ids < 0)
        return -1;
    for (int32_t i = 0; i < num_ids; ++i) {
        int32_t blk = block_ids[i];
        if (blk < 0 || blk >= num_blocks) {
            err = -5;
            continue;
        }
        for (int64_t b = 0; b < block_bytes; ++b) {
            key_cache[(int64_t)blk * block_bytes + b] = 0;
            value_cache[(int64_t)blk * block_bytes + b] = 0;
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Cache write                                                               */
/* ------------------------------------------------------------------------ */

int oracle_cache_write(const uint16_t *key, const uint16_t *value,
                       int64_t kv_token_stride, uint16_t *key_cache,
                       uint16_t *value_cache, const int32_t *slot_mapping,
                       int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, int32_t num_blocks)
{
    int err = 0;
    int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;                         /* padding row: nothing to write */
        if (slot >= num_slots) {
            err = -1;
            continue;
        }
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = (int64_t)t * kv_token_stride + (int64_t)h * head_dim + d;
                int64_t dst = (slot * num_kv_heads + h) * head_dim + d;
                key_cache[dst] = key[src];
                value_cache[dst] = value[src];
            }
    }
    return err;
}

/* The write into an FP8 cache ("Inside vLLM: Following One Request", the
 * write op's kv_cache_dtype, k_scale and v_scale arguments): each element of
 * the new key is divided by k_scale in single precision and rounded to E4M3
 * (values of V likewise with v_scale).  src_dtype is the type of key/value. */
int oracle_cache_write_fp8(const uint16_t *key, const uint16_t *value,
                           int64_t kv_token_stride, uint8_t *key_cache,
                           uint8_t *value_cache, const int32_t *slot_mapping,
                           int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, int32_t src_dtype,
                           float k_scale, float v_scale)
{
    int err = 0;
    int64_t num_slots = (int64_t)num_blocks * block_size;
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f))
        return -1;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            err = -8;
            continue;
        }
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = (int64_t)t * kv_token_stride + (int64_t)h * head_dim + d;
                int64_t dst = (slot * num_kv_heads + h) * head_dim + d;
                float kq = (float)elem(key[src], src_dtype) / k_scale;
                float vq = (float)elem(value[src], src_dtype) / v_scale;
                key_cache[dst] = float_to_e4m3(kq);
                value_cache[dst] = float_to_e4m3(vq);
            }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Attention                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t req;        /* request */
    int32_t kv_head;    /* kv head g */
    int32_t first;      /* range [first, last) into the selected-token list */
    int32_t last;
} work_item;

typedef struct {
    const uint16_t *q;
    const void *key_cache, *value_cache;
    const int32_t *block_table, *query_start_loc, *seq_lens;
    int32_t max_blocks_per_req, num_q_heads, num_kv_heads, head_dim, block_size;
    int32_t dtype;                /* q */
    int32_t cache_dtype;          /* K/V pools */
    double k_scale, v_scale;      /* pool element * scale = the cached value */
    double scale;
    double *out;
    const int32_t *sel;           /* selected tokens, ascending */
    const work_item *items;
    int64_t num_items;
    int64_t next;                 /* shared work counter */
    int failed;
} attn_job;

/* Position of flat token t of request r: the request's last query token is
 * at seq_len - 1, so the chunk starts at seq_len - q_len (= num_computed). */
static int32_t token_position(const attn_job *jb, int32_t r, int32_t t)
{
    int32_t q_len = jb->query_start_loc[r + 1] - jb->query_start_loc[r];
    return jb->seq_lens[r] - q_len + (t - jb->query_start_loc[r]);
}

static void run_item(const attn_job *jb, const work_item *it, double *kc, double *vc,
                     double *w)
{
    const int32_t D = jb->head_dim, Hkv = jb->num_kv_heads, Hq = jb->num_q_heads;
    const int32_t group = Hq / Hkv;
    const int32_t r = it->req, g = it->kv_head;
    /* Keys needed by the chunk: up to the largest position in it. */
    int32_t keys = token_position(jb, r, jb->sel[it->last - 1]) + 1;

    /* Gather: logical key j lives in physical block block_table[r][j / bs]
     * at offset j % bs. */
    for (int32_t j = 0; j < keys; ++j) {
        int32_t phys = jb->block_table[(int64_t)r * jb->max_blocks_per_req + j / jb->block_size];
        int64_t slot = (int64_t)phys * jb->block_size + j % jb->block_size;
        for (int32_t d = 0; d < D; ++d) {
            int64_t a = (slot * Hkv + g) * D + d;
            kc[(int64_t)j * D + d] = cache_elem(jb->key_cache, a, jb->cache_dtype) * jb->k_scale;
            vc[(int64_t)j * D + d] = cache_elem(jb->value_cache, a, jb->cache_dtype) * jb->v_scale;
        }
    }

    for (int32_t s = it->first; s < it->last; ++s) {
        int32_t t = jb->sel[s];
        int32_t p = token_position(jb, r, t);
        for (int32_t h = g * group; h < (g + 1) * group; ++h) {
            const uint16_t *qv = jb->q + ((int64_t)t * Hq + h) * D;
            double m = -INFINITY;
            for (int32_t j = 0; j <= p; ++j) {
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    dot += elem(qv[d], jb->dtype) * kc[(int64_t)j * D + d];
                w[j] = jb->scale * dot;
                if (w[j] > m)
                    m = w[j];
            }
            double l = 0.0;
            for (int32_t j = 0; j <= p; ++j) {
                w[j] = exp(w[j] - m);
                l += w[j];
            }
            double *o = jb->out + ((int64_t)t * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int32_t j = 0; j <= p; ++j)
                    acc += w[j] * vc[(int64_t)j * D + d];
                o[d] = acc / l;
            }
        }
    }
}

static void *attn_worker(void *arg)
{
    attn_job *jb = (attn_job *)arg;
    int64_t cap = 0;
    double *kc = NULL, *vc = NULL, *w = NULL;
    for (;;) {
        int64_t i = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (i >= jb->num_items)
            break;
        const work_item *it = &jb->items[i];
        int64_t keys = token_position(jb, it->req, jb->sel[it->last - 1]) + 1;
        if (keys > cap) {
            free(kc);
            free(vc);
            free(w);
            cap = keys;
            kc = malloc(sizeof(double) * cap * jb->head_dim);
            vc = malloc(sizeof(double) * cap * jb->head_dim);
            w = malloc(sizeof(double) * cap);
            if (!kc || !vc || !w) {
                __atomic_store_n(&jb->failed, 1, __ATOMIC_RELAXED);
                cap = 0;
                continue;
            }
        }
        run_item(jb, it, kc, vc, w);
    }
    free(kc);
    free(vc);
    free(w);
    return NULL;
}

int oracle_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * out: fp64 [num_tokens][num_q_heads][head_dim].  When `tokens` is non-NULL
 * only those flat token indices (ascending) are computed and written.
 * num_threads <= 0 uses every online CPU.  Tokens are split into chunks of
 * at most `chunk` tokens per (request, kv head) so that the threads share a
 * long prefill.
 */
int oracle_attention_ex(const uint16_t *q, const void *key_cache,
                        const void *value_cache, const int32_t *block_table,
                        int32_t max_blocks_per_req, const int32_t *query_start_loc,
                        const int32_t *seq_lens, int32_t num_reqs, int32_t num_tokens,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, double scale,
                        int32_t dtype, int32_t cache_dtype, double k_scale, double v_scale,
                        double *out, const int32_t *tokens, int32_t num_selected,
                        int32_t num_threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads || head_dim <= 0 || block_size <= 0)
        return -1;
    if (query_start_loc[0] != 0 || query_start_loc[num_reqs] != num_tokens)
        return -2;
    /* Every logical block a request reads must name a pool block. */
    for (int32_t r = 0; r < num_reqs; ++r) {
        int32_t q_len = query_start_loc[r + 1] - query_start_loc[r];
        if (q_len < 0 || seq_lens[r] < q_len)
            return -3;
        int32_t nblk = (seq_lens[r] + block_size - 1) / block_size;
        if (nblk > max_blocks_per_req)
            return -4;
        for (int32_t b = 0; b < nblk; ++b) {
            int32_t phys = block_table[(int64_t)r * max_blocks_per_req + b];
            if (phys < 0 || phys >= num_blocks)
                return -5;
        }
    }

    int32_t n_sel = tokens ? num_selected : num_tokens;
    int32_t *sel = malloc(sizeof(int32_t) * (n_sel > 0 ? n_sel : 1));
    /* request of each selected token */
    int32_t *sel_req = malloc(sizeof(int32_t) * (n_sel > 0 ? n_sel : 1));
    if (!sel || !sel_req) {
        free(sel);
        free(sel_req);
        return -6;
    }
    for (int32_t i = 0; i < n_sel; ++i) {
        sel[i] = tokens ? tokens[i] : i;
        if (sel[i] < 0 || sel[i] >= num_tokens || (i && sel[i] <= sel[i - 1])) {
            free(sel);
            free(sel_req);
            return -7;
        }
    }
    for (int32_t i = 0, r = 0; i < n_sel; ++i) {
        while (sel[i] >= query_start_loc[r + 1])
            ++r;
        sel_req[i] = r;
    }

    const int32_t chunk = 32;
    int64_t cap_items = 0;
    for (int32_t i = 0; i < n_sel;) {
        int32_t j = i;
        while (j < n_sel && sel_req[j] == sel_req[i] && j - i < chunk)
            ++j;
        cap_items += num_kv_heads;
        i = j;
    }
    work_item *items = malloc(sizeof(work_item) * (cap_items > 0 ? cap_items : 1));
    if (!items) {
        free(sel);
        free(sel_req);
        return -6;
    }
    int64_t n_items = 0;
    for (int32_t i = 0; i < n_sel;) {
        int32_t j = i;
        while (j < n_sel && sel_req[j] == sel_req[i] && j - i < chunk)
            ++j;
        for (int32_t g = 0; g < num_kv_heads; ++g) {
            work_item it = {sel_req[i], g, i, j};
            items[n_items++] = it;
        }
        i = j;
    }

    attn_job jb = {q, key_cache, value_cache, block_table, query_start_loc, seq_lens,
                   max_blocks_per_req, num_q_heads, num_kv_heads, head_dim, block_size,
                   dtype, cache_dtype, k_scale, v_scale, scale, out, sel, items, n_items, 0, 0};
    int nt = num_threads > 0 ? num_threads : oracle_num_cpus();
    if (nt > n_items)
        nt = n_items > 0 ? (int)n_items : 1;
    pthread_t *th = malloc(sizeof(pthread_t) * nt);
    int started = 0;
    if (th)
        for (; started < nt - 1; ++started)
            if (pthread_create(&th[started], NULL, attn_worker, &jb))
                break;
    attn_worker(&jb);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(th);
    free(items);
    free(sel);
    free(sel_req);
    return jb.failed ? -6 : 0;
}

/* Attention over 16-bit pools of the same type as q (scales 1). */
int oracle_attention(const uint16_t *q, const uint16_t *key_cache,
                     const uint16_t *value_cache, const int32_t *block_table,
                     int32_t max_blocks_per_req, const int32_t *query_start_loc,
                     const int32_t *seq_lens, int32_t num_reqs, int32_t num_tokens,
                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int32_t num_blocks, double scale,
                     int32_t dtype, double *out, const int32_t *tokens,
                     int32_t num_selected, int32_t num_threads)
{
    return oracle_attention_ex(q, key_cache, value_cache, block_table, max_blocks_per_req,
                               query_start_loc, seq_lens, num_reqs, num_tokens, num_q_heads,
                               num_kv_heads, head_dim, block_size, num_blocks, scale, dtype,
                               dtype, 1.0, 1.0, out, tokens, num_selected, num_threads);
}
