// pa_attention_noalloc: pa_attention with scratch the library owns.
//
// Some callers cannot allocate device memory when they call us: a serving
// engine that hands almost all free HBM to its KV-cache pool at start-up
// (a later cudaMalloc for scratch can then fail), a latency-sensitive decode
// loop where cudaMalloc/cudaFree would synchronise the device and stall
// other streams, or a host program that reaches the library through the
// plain C ABI and has no device allocator of its own.  This entry point
// takes the same inputs and outputs as pa_attention and uses a fixed array
// in the library's own device memory as the workspace instead of one the
// caller passes.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.cuh"

namespace {

// The scratch: 32 MiB per GPU that loads the library, held until exit.
// Every call on a device shares it; nothing in it needs clearing because each
// call writes every byte it later reads (per-request partition metadata and
// partial results) before reading it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
// The array's address as last looked up on each device, and the CUDA context
// that was current then.  A module -- and with it the array -- is loaded once
// per context, so a caller that makes another context current on the same
// device (driver-API contexts) gets the lookup again.
void *g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch in the current context.  Host code must not
// hand the array's name to a kernel: on the host it is only a stand-in.
pa_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ctx_current) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return PA_ERR_CUDA;
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    }
    // No context is current before the runtime's first call on this thread
    // that needs one; the lookup below makes the device's primary context
    // current in that case.
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
    if (!ctx || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return PA_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_attention_noalloc(
    const void *q, const void *key_cache, const void *value_cache, const int32_t *block_table,
    int32_t max_blocks_per_req, const int32_t *query_start_loc, const int32_t *seq_lens,
    int32_t num_reqs, int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float scale, pa_dtype dtype, void *out, pa_stream_t stream) {
    if (num_reqs > PA_NOALLOC_MAX_REQS) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    return pa_attention(q, key_cache, value_cache, block_table, max_blocks_per_req,
                        query_start_loc, seq_lens, num_reqs, num_tokens, max_query_len,
                        max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                        scale, dtype, out, scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
