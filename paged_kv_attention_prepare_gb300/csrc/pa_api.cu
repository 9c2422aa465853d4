// The C ABI (include/pa.h): host-side argument checks, the per-device status
// word, TMA descriptor encoding, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.cuh"

// The one piece of device state the library keeps: a word of PA_CHECK_* bits
// that kernels OR into when a data-dependent check fails.
static __device__ unsigned int g_pa_status;

namespace pa {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int *g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
thread_local uint64_t t_launches = 0;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

unsigned int *status_word() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_status_ptr[dev];
}

void note_launch(int n) { t_launches += (uint64_t)n; }

int num_sms() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool encode_pool_map_swizzled(CUtensorMap *map, const void *pool, int64_t num_slots, int Hkv,
                              int D, int elt, int box_rows) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return false;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    const int row = D * elt;
    const int inner = row >= 128 ? 128 : row;  // bytes of one box row
    if (inner != 128 && inner != 64) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)num_slots};
    const cuuint64_t strides[2] = {(cuuint64_t)row, (cuuint64_t)Hkv * row};
    const cuuint32_t box[3] = {(cuuint32_t)(inner / elt), 1u, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = g_encode(map, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                          3, const_cast<void *>(pool), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pa

using namespace pa;

namespace {

// Checks and argument packing shared by both index-build entry points.
pa_status check_prepare_core(const PrepArgs &a) {
    if (a.R < 0 || a.T < 0 || a.bs <= 0 || a.NB < 0 || a.MB < 0 || a.qsl_cap < a.R + 1)
        return PA_ERR_INVALID;
    if (!a.qsl) return PA_ERR_INVALID;
    if (a.R > 0 && (!a.nst || !a.nct || !a.seq_lens || (a.MB > 0 && !a.bt)))
        return PA_ERR_INVALID;
    if (a.num_logits > 0 && !a.logits) return PA_ERR_INVALID;
    if (a.T > 0 && (!a.req || !a.pos || !a.slot)) return PA_ERR_INVALID;
    if ((int64_t)a.NB * a.bs >= (int64_t)INT32_MAX) return PA_ERR_INVALID;
    return PA_OK;
}

// True when a kernel on the current device can dereference `p` as given.
bool device_readable(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        return true;
    case cudaMemoryTypeHost:
        // Page-locked host memory: readable at the same address under
        // unified addressing.
        return at.devicePointer == p;
    default: {
        int dev = current_device(), pageable = 0;
        if (dev < 0 || cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) !=
                           cudaSuccess)
            return false;
        return pageable != 0;
    }
    }
}

}  // namespace

extern "C" {

pa_status pa_prepare_inputs(const int32_t *num_scheduled_tokens, const int32_t *num_computed_tokens,
                            const int32_t *block_table, int32_t num_reqs,
                            int32_t max_blocks_per_req, int32_t block_size, int32_t num_tokens,
                            int32_t num_blocks, int32_t *req_indices, int32_t *positions,
                            int32_t *slot_mapping, int32_t *query_start_loc, int32_t qsl_capacity,
                            int32_t *seq_lens, int32_t *logits_indices, pa_stream_t stream) {
    PrepArgs a{};
    a.nst = num_scheduled_tokens;
    a.nct = num_computed_tokens;
    a.bt = block_table;
    a.R = num_reqs;
    a.MB = max_blocks_per_req;
    a.bs = block_size;
    a.T = num_tokens;
    a.NB = num_blocks;
    a.num_logits = num_reqs;
    a.req = req_indices;
    a.pos = positions;
    a.slot = slot_mapping;
    a.qsl = query_start_loc;
    a.qsl_cap = qsl_capacity;
    a.seq_lens = seq_lens;
    a.logits = logits_indices;
    const pa_status st = check_prepare_core(a);
    if (st != PA_OK) return st;
    return launch_prepare(a, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_prepare_inputs_ex(const int32_t *num_scheduled_tokens,
                               const int32_t *num_computed_tokens, const int32_t *block_table,
                               int32_t num_reqs, int32_t max_blocks_per_req, int32_t block_size,
                               int32_t num_tokens, int32_t num_blocks, const int32_t *token_ids,
                               int32_t max_num_reqs, int32_t max_model_len,
                               const int32_t *request_num_tokens,
                               const int32_t *num_draft_tokens, int32_t num_logits,
                               int32_t *req_indices, int32_t *positions, int32_t *slot_mapping,
                               int32_t *query_start_loc, int32_t qsl_capacity, int32_t *seq_lens,
                               int64_t *token_indices, int32_t *input_ids,
                               uint8_t *discard_request_mask, int32_t *logits_indices,
                               int32_t *cu_num_logits, pa_stream_t stream) {
    PrepArgs a{};
    a.nst = num_scheduled_tokens;
    a.nct = num_computed_tokens;
    a.bt = block_table;
    a.R = num_reqs;
    a.MB = max_blocks_per_req;
    a.bs = block_size;
    a.T = num_tokens;
    a.NB = num_blocks;
    a.token_ids = token_ids;
    a.max_num_reqs = max_num_reqs;
    a.M = max_model_len;
    a.req_num_tokens = request_num_tokens;
    a.num_draft = num_draft_tokens;
    a.num_logits = num_logits;
    a.req = req_indices;
    a.pos = positions;
    a.slot = slot_mapping;
    a.qsl = query_start_loc;
    a.qsl_cap = qsl_capacity;
    a.seq_lens = seq_lens;
    a.token_indices = token_indices;
    a.input_ids = input_ids;
    a.discard = discard_request_mask;
    a.logits = logits_indices;
    a.cu_logits = cu_num_logits;
    const pa_status st = check_prepare_core(a);
    if (st != PA_OK) return st;
    if (num_logits < 0 || (!num_draft_tokens && num_logits != num_reqs)) return PA_ERR_INVALID;
    // token-id gather group
    if (max_model_len < 0) return PA_ERR_INVALID;
    if (max_model_len > 0) {
        if (!token_ids || max_num_reqs < num_reqs ||
            (num_tokens > 0 && (!token_indices || !input_ids)))
            return PA_ERR_INVALID;
        if (!device_readable(token_ids)) return PA_ERR_INVALID;
    } else if (token_ids || token_indices || input_ids) {
        return PA_ERR_INVALID;
    }
    // discard group
    if ((request_num_tokens == nullptr) != (discard_request_mask == nullptr))
        return PA_ERR_INVALID;
    return launch_prepare(a, reinterpret_cast<cudaStream_t>(stream));
}

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
                               pa_stream_t stream) {
    PrepArgs a{};
    a.nst = num_scheduled_tokens;
    a.nct = num_computed_tokens;
    a.bt = block_table;
    a.R = num_reqs;
    a.MB = max_blocks_per_req;
    a.bs = block_size;
    a.T = num_tokens;
    a.NB = num_blocks;
    a.num_logits = num_reqs;
    a.req = req_indices;
    a.pos = positions;
    a.slot = slot_mapping;
    a.qsl = query_start_loc;
    a.qsl_cap = qsl_capacity;
    a.seq_lens = seq_lens;
    a.logits = logits_indices;
    const pa_status st = check_prepare_core(a);
    if (st != PA_OK) return st;
    // the write's checks, as pa_cache_write_ex
    if (num_kv_heads <= 0 || head_dim <= 0 || (dtype != PA_BF16 && dtype != PA_FP16) ||
        (cache_dtype != dtype && cache_dtype != PA_FP8_E4M3))
        return PA_ERR_INVALID;
    if (kv_token_stride < (int64_t)num_kv_heads * head_dim) return PA_ERR_INVALID;
    if (num_tokens > 0 && (!key || !value || !key_cache || !value_cache)) return PA_ERR_INVALID;
    if ((int64_t)num_kv_heads * head_dim > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
    return launch_prepare_write(a, key, value, kv_token_stride, key_cache, value_cache,
                                num_kv_heads * head_dim, dtype, cache_dtype, k_scale, v_scale,
                                reinterpret_cast<cudaStream_t>(stream));
}

static pa_status check_block_op(void *kc, void *vc, const void *a, const void *b, int32_t n,
                                int32_t bs, int32_t hkv, int32_t d, int32_t nb, pa_dtype dtype,
                                int64_t *block_bytes) {
    if (n < 0 || bs <= 0 || hkv <= 0 || d <= 0 || nb < 0 ||
        (dtype != PA_BF16 && dtype != PA_FP16 && dtype != PA_FP8_E4M3))
        return PA_ERR_INVALID;
    if (n > 0 && (!kc || !vc || !a || !b)) return PA_ERR_INVALID;
    if (n > 0 && (!aligned(kc, 16) || !aligned(vc, 16))) return PA_ERR_INVALID;
    const int64_t bb = (int64_t)bs * hkv * d * (dtype == PA_FP8_E4M3 ? 1 : 2);
    if (bb % 16 != 0) return PA_ERR_UNSUPPORTED;
    *block_bytes = bb;
    return PA_OK;
}

pa_status pa_copy_blocks(void *key_cache, void *value_cache, const int32_t *src_blocks,
                         const int32_t *dst_blocks, int32_t num_pairs, int32_t block_size,
                         int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                         pa_dtype dtype, pa_stream_t stream) {
    int64_t bb = 0;
    const pa_status st = check_block_op(key_cache, value_cache, src_blocks, dst_blocks, num_pairs,
                                        block_size, num_kv_heads, head_dim, num_blocks, dtype, &bb);
    if (st != PA_OK) return st;
    return launch_copy_blocks(key_cache, value_cache, bb, num_blocks, src_blocks, dst_blocks,
                              num_pairs, reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_zero_blocks(void *key_cache, void *value_cache, const int32_t *block_ids,
                         int32_t num_ids, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim, int32_t num_blocks, pa_dtype dtype,
                         pa_stream_t stream) {
    int64_t bb = 0;
    const pa_status st = check_block_op(key_cache, value_cache, block_ids, block_ids, num_ids,
                                        block_size, num_kv_heads, head_dim, num_blocks, dtype, &bb);
    if (st != PA_OK) return st;
    return launch_zero_blocks(key_cache, value_cache, bb, num_blocks, block_ids, num_ids,
                              reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_cache_write_ex(const void *key, const void *value, int64_t kv_token_stride,
                            void *key_cache, void *value_cache, const int32_t *slot_mapping,
                            int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                            pa_dtype cache_dtype, const float *k_scale, const float *v_scale,
                            pa_stream_t stream) {
    if (cache_dtype == dtype)
        return pa_cache_write(key, value, kv_token_stride, key_cache, value_cache, slot_mapping,
                              num_tokens, num_kv_heads, head_dim, block_size, num_blocks, dtype,
                              stream);
    if (cache_dtype != PA_FP8_E4M3) return PA_ERR_INVALID;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || (dtype != PA_BF16 && dtype != PA_FP16))
        return PA_ERR_INVALID;
    if (kv_token_stride < (int64_t)num_kv_heads * head_dim) return PA_ERR_INVALID;
    if (num_tokens > 0 && (!key || !value || !key_cache || !value_cache || !slot_mapping))
        return PA_ERR_INVALID;
    if ((int64_t)num_kv_heads * head_dim > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
    return launch_cache_write_fp8(key, value, kv_token_stride, key_cache, value_cache,
                                  slot_mapping, num_tokens, num_kv_heads * head_dim,
                                  (int64_t)num_blocks * block_size, dtype, k_scale, v_scale,
                                  reinterpret_cast<cudaStream_t>(stream));
}

pa_status pa_cache_write(const void *key, const void *value, int64_t kv_token_stride,
                         void *key_cache, void *value_cache, const int32_t *slot_mapping,
                         int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                         pa_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || (dtype != PA_BF16 && dtype != PA_FP16))
        return PA_ERR_INVALID;
    if (kv_token_stride < (int64_t)num_kv_heads * head_dim) return PA_ERR_INVALID;
    if (num_tokens > 0 && (!key || !value || !key_cache || !value_cache || !slot_mapping))
        return PA_ERR_INVALID;
    if ((int64_t)num_kv_heads * head_dim > INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
    return launch_cache_write(key, value, kv_token_stride, key_cache, value_cache, slot_mapping,
                              num_tokens, num_kv_heads * head_dim,
                              (int64_t)num_blocks * block_size,
                              reinterpret_cast<cudaStream_t>(stream));
}

size_t pa_attention_workspace_size(int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                                   int32_t max_seq_len, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim) {
    if (num_reqs <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0) return 0;
    const size_t dec = decode_workspace_size(num_reqs, num_tokens, max_query_len, max_seq_len,
                                             num_q_heads, num_kv_heads, head_dim);
    return kCtrlBytes + (dec + 255) / 256 * 256 +
           prefill_widen_size(num_reqs, num_tokens, max_query_len, max_seq_len, num_kv_heads,
                              head_dim);
}

pa_status pa_attention(const void *q, const void *key_cache, const void *value_cache,
                       const int32_t *block_table, int32_t max_blocks_per_req,
                       const int32_t *query_start_loc, const int32_t *seq_lens, int32_t num_reqs,
                       int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, int32_t num_blocks, float scale, pa_dtype dtype,
                       void *out, void *workspace, size_t workspace_bytes, pa_stream_t stream) {
    return pa_attention_ex(q, key_cache, value_cache, block_table, max_blocks_per_req,
                           query_start_loc, seq_lens, num_reqs, num_tokens, max_query_len,
                           max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, scale, dtype, dtype, nullptr, nullptr, 0u, out, workspace,
                           workspace_bytes, stream);
}

pa_status pa_attention_ex(const void *q, const void *key_cache, const void *value_cache,
                          const int32_t *block_table, int32_t max_blocks_per_req,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          int32_t num_reqs, int32_t num_tokens, int32_t max_query_len,
                          int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                          pa_dtype dtype, pa_dtype cache_dtype, const float *k_scale,
                          const float *v_scale, uint32_t flags, void *out, void *workspace,
                          size_t workspace_bytes, pa_stream_t stream) {
    if (flags & ~PA_ATTN_SHARED_BLOCKS) return PA_ERR_INVALID;
    if (num_reqs < 0 || num_tokens < 0 || max_query_len < 0 || max_seq_len < 0 ||
        num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks < 0 || max_blocks_per_req < 0 || (dtype != PA_BF16 && dtype != PA_FP16))
        return PA_ERR_INVALID;
    if (cache_dtype != dtype && cache_dtype != PA_FP8_E4M3) return PA_ERR_INVALID;
    if (workspace_bytes > 0 && (!workspace || !aligned(workspace, 256))) return PA_ERR_INVALID;
    if (num_tokens == 0 || num_reqs == 0) return PA_OK;
    if (!q || !key_cache || !value_cache || !block_table || !query_start_loc || !seq_lens || !out)
        return PA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(key_cache, 16) ||
        !aligned(value_cache, 16))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (block_size != 16) return PA_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size >= (int64_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (num_blocks == 0 || max_blocks_per_req == 0) return PA_ERR_INVALID;
    AttnArgs a;
    a.q = q;
    a.kc = key_cache;
    a.vc = value_cache;
    a.bt = block_table;
    a.MB = max_blocks_per_req;
    a.qsl = query_start_loc;
    a.seq_lens = seq_lens;
    a.R = num_reqs;
    a.T = num_tokens;
    a.max_q = max_query_len;
    a.max_seq = max_seq_len;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.D = head_dim;
    a.bs = block_size;
    a.NB = num_blocks;
    a.scale = scale;
    a.dtype = dtype;
    a.cache_dtype = cache_dtype;
    a.k_scale = cache_dtype == PA_FP8_E4M3 ? k_scale : nullptr;
    a.v_scale = cache_dtype == PA_FP8_E4M3 ? v_scale : nullptr;
    a.out = out;
    a.flags = flags;
    // The workspace starts with a small control block (the kernels' item
    // counters); the split-K partials take the rest.
    a.ctrl = nullptr;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    a.pf_ws = nullptr;
    a.pf_bytes = 0;
    if (workspace && workspace_bytes >= kCtrlBytes) {
        a.ctrl = static_cast<unsigned int *>(workspace);
        a.ws = static_cast<unsigned char *>(workspace) + kCtrlBytes;
        a.ws_bytes = workspace_bytes - kCtrlBytes;
        // Past what the decode partials can use, the rest goes to the
        // prefill kernel (a widened copy of bf16 V).
        const size_t dec = (decode_workspace_size(num_reqs, num_tokens, max_query_len,
                                                  max_seq_len, num_q_heads, num_kv_heads,
                                                  head_dim) + 255) / 256 * 256;
        if (a.ws_bytes > dec) {
            a.pf_ws = static_cast<unsigned char *>(a.ws) + dec;
            a.pf_bytes = a.ws_bytes - dec;
            a.ws_bytes = dec;
        }
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (a.ctrl) PA_TRY_CUDA(cudaMemsetAsync(a.ctrl, 0, kCtrlWords * sizeof(unsigned int), st));
    const int tau = prefill_tau(a);
    a.pdl = false;
    a.decode_part = 0;
    // Both request classes possible: the two kernels side by side.
    if (a.ctrl && tau != INT_MAX && max_query_len > tau && num_reqs > 1)
        return launch_attention_overlapped(a, tau, st);
    const pa_status r = launch_decode(a, tau, st);
    if (r != PA_OK) return r;
    return launch_prefill(a, tau, st);
}

pa_status pa_get_status(pa_stream_t stream, uint32_t *detail) {
    if (detail) *detail = 0;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    unsigned int v = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_pa_status, sizeof v) != cudaSuccess) return PA_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_pa_status, &zero, sizeof zero) != cudaSuccess) return PA_ERR_CUDA;
    if (detail) *detail = v;
    if (!v) return PA_OK;
    return (v & PA_CHECK_TIMEOUT) ? PA_ERR_TIMEOUT : PA_ERR_DEVICE_CHECK;
}

const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID: return "invalid argument";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
        case PA_ERR_DEVICE_CHECK: return "a device-side data check failed";
        case PA_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
        case PA_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

uint64_t pa_launch_count(void) {
    const uint64_t n = t_launches;
    t_launches = 0;
    return n;
}

}  // extern "C"
