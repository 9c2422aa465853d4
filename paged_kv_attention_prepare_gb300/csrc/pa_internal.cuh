// Internal helpers shared by the library's translation units: launch
// plumbing, the status-word bits, and thin inline-PTX wrappers for mbarriers,
// TMA bulk-tensor copies and bounded waits on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// Device address of this device's status word (set up once per device).
unsigned int *status_word();
// Count one kernel launch queued by the calling thread.
void note_launch(int n = 1);
int num_sms();

// Inputs and outputs of the index build.  The three optional groups are off
// when their pointers are NULL: the token-id gather (M > 0), the discard mask
// and the draft tokens (then num_logits == R, one row per request).
struct PrepArgs {
    const int32_t *nst, *nct, *bt;
    int32_t R, MB, bs, T, NB;
    const int32_t *token_ids;       // [max_num_reqs][M], device-readable
    int32_t max_num_reqs, M;
    const int32_t *req_num_tokens;  // [R]
    const int32_t *num_draft;       // [R]
    int32_t num_logits;
    int32_t *req, *pos, *slot, *qsl;
    int32_t qsl_cap;
    int32_t *seq_lens;
    int64_t *token_indices;
    int32_t *input_ids;
    uint8_t *discard;
    int32_t *logits, *cu_logits;
};

pa_status launch_prepare(const PrepArgs &a, cudaStream_t stream);
// The index build (no optional groups) and the cache write in one launch;
// PA_ERR_UNSUPPORTED when the rows are not 16-byte aligned (8-byte FP8 pool
// rows).
pa_status launch_prepare_write(const PrepArgs &a, const void *key, const void *value,
                               int64_t stride_elems, void *kc, void *vc, int32_t row_elems,
                               pa_dtype dtype, pa_dtype cache_dtype, const float *k_scale,
                               const float *v_scale, cudaStream_t stream);

pa_status launch_copy_blocks(void *kc, void *vc, int64_t block_bytes, int32_t num_blocks,
                             const int32_t *src, const int32_t *dst, int32_t n,
                             cudaStream_t stream);
pa_status launch_zero_blocks(void *kc, void *vc, int64_t block_bytes, int32_t num_blocks,
                             const int32_t *ids, int32_t n, cudaStream_t stream);

pa_status launch_cache_write(const void *key, const void *value, int64_t stride_elems,
                             void *kc, void *vc, const int32_t *slots, int32_t T,
                             int32_t row_elems, int64_t num_slots, cudaStream_t stream);
// The write into FP8 pools: element / scale, rounded to E4M3 (satfinite).
pa_status launch_cache_write_fp8(const void *key, const void *value, int64_t stride_elems,
                                 void *kc, void *vc, const int32_t *slots, int32_t T,
                                 int32_t row_elems, int64_t num_slots, pa_dtype src,
                                 const float *k_scale, const float *v_scale, cudaStream_t stream);

struct AttnArgs {
    const void *q;
    const void *kc, *vc;
    const int32_t *bt;
    int32_t MB;
    const int32_t *qsl, *seq_lens;
    int32_t R, T, max_q, max_seq, Hq, Hkv, D, bs, NB;
    float scale;
    pa_dtype dtype;        // q and out
    pa_dtype cache_dtype;  // the pools: dtype, or PA_FP8_E4M3
    const float *k_scale;  // FP8 pools: device scalars (NULL = 1)
    const float *v_scale;
    void *out;
    void *ws;              // decode partials (after the control block)
    size_t ws_bytes;
    void *pf_ws;           // the workspace past the decode partials (NULL: none)
    size_t pf_bytes;
    unsigned int *ctrl;    // control block at the workspace's start (NULL: none)
    uint32_t flags;        // PA_ATTN_* bits
    bool pdl;              // launch the split-K kernel as a programmatic dependent
    int decode_part;       // launch_decode: 0 split-K grid + merge, 1 the grid only, 2 the merge only
};

// Bytes at the start of a caller's workspace kept for per-call counters.
constexpr size_t kCtrlBytes = 256;
// Words of the control block: the kernels' item counters, zeroed by one
// memset before each attention call's launches.
constexpr int kCtrlPrefillCounter = 0;
constexpr int kCtrlDecodeCounter = 1;
constexpr int kCtrlWords = 2;

size_t decode_workspace_size(int32_t R, int32_t T, int32_t max_q, int32_t max_seq,
                             int32_t Hq, int32_t Hkv, int32_t D);
// Requests with at most `tau` query tokens run on the split-K kernel, longer
// ones on the tensor-core kernel (tau == INT_MAX: everything split-K).
int prefill_tau(const AttnArgs &a);
// Workspace for the prefill kernel's widened copy of bf16 V (past the decode
// partials); 0 when no request can take the prefill kernel or head_dim is
// not 128.
size_t prefill_widen_size(int32_t R, int32_t T, int32_t max_q, int32_t max_seq, int32_t Hkv,
                          int32_t D);
pa_status launch_decode(const AttnArgs &a, int tau, cudaStream_t stream);
pa_status launch_prefill(const AttnArgs &a, int tau, cudaStream_t stream);
// A batch that may hold both request classes: the tensor-core kernel's first
// grid on two fifths of the SMs, the split-K kernel beside it on the rest, a
// second tensor-core grid that takes the remaining prefill items as SMs free
// up, then the merge pass.  Same results as launch_decode then
// launch_prefill.
pa_status launch_attention_overlapped(const AttnArgs &a, int tau, cudaStream_t stream);

// Encode a 3-D TMA map over one pool viewed as [NB*bs][Hkv][D] elements of
// `elt` bytes, with a box of min(128 bytes, a row) x 1 kv head x `box_rows`
// slots and the swizzle that matches the box's row (128 or 64 bytes).
bool encode_pool_map_swizzled(CUtensorMap *map, const void *pool, int64_t num_slots, int Hkv,
                              int D, int elt, int box_rows);

// ---------------------------------------------------------------------------
// Device side
// ---------------------------------------------------------------------------

__device__ __forceinline__ void flag(unsigned int *status, unsigned int bit) {
    atomicOr(status, bit);
}

// Block-wide exclusive scan of one value per thread.  Returns the thread's
// exclusive prefix and sets `total` to the block's sum.  `sh` is 33 shared
// ints (one per warp plus the total); it is free again on return.
__device__ __forceinline__ int block_exclusive_scan(int v, int *sh, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w0 = lane < nwarps ? sh[lane] : 0;
        int w = w0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < nwarps) sh[lane] = w - w0;
        if (lane == 31) sh[32] = w;
    }
    __syncthreads();
    const int r = sh[warp] + incl - v;
    total = sh[32];
    __syncthreads();
    return r;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Upper bound for any single wait inside a kernel.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false after the
// time limit (the caller records the timeout and winds down).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// The same wait taken by a whole warp: every lane gets one answer, so the
// warp stays converged for the warp-collective instructions that follow.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

// 3-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Programmatic dependent launch.  A grid launched with programmatic stream
// serialization may start before the grid ahead of it in the stream ends;
// grid_dependency_wait() returns once that grid has completed and its
// memory writes are visible (at once for a grid launched without the
// attribute).  grid_launch_dependents() lets the dependent grid be scheduled
// once every CTA of this grid has called it or exited.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Element traits: packed 16-bit elements -> floats, and two floats -> a
// packed pair rounded to nearest even.
template <typename T> struct Elt;

template <> struct Elt<__nv_bfloat16> {
    __device__ __forceinline__ static void unpack2(uint32_t w, float &a, float &b) {
        a = __uint_as_float(w << 16);
        b = __uint_as_float(w & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

template <> struct Elt<__half> {
    __device__ __forceinline__ static void unpack2(uint32_t w, float &a, float &b) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w);
        float2 x = __half22float2(h);
        a = x.x;
        b = x.y;
    }
    __device__ __forceinline__ static uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// Eight 16-bit elements (one 16-byte load, element 0 in the low half of the
// first word) to E4M3 codes (element 0 in the low byte): each divided by
// `scale` in IEEE single precision (correctly rounded), then rounded to the
// nearest E4M3 value, ties to even, saturating at +-448 (NaN stays NaN).
template <typename T>
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4 src, float scale) {
    const uint32_t w[4] = {src.x, src.y, src.z, src.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float x0, x1;
        Elt<T>::unpack2(w[e], x0, x1);
        const uint32_t q = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale)), __NV_SATFINITE, __NV_E4M3);
        out[e >> 1] |= (q & 0xffffu) << (16 * (e & 1));
    }
    return make_uint2(out[0], out[1]);
}

}  // namespace pa

#define PA_TRY_CUDA(expr)                                  \
    do {                                                   \
        cudaError_t e_ = (expr);                           \
        if (e_ != cudaSuccess) return PA_ERR_CUDA;         \
    } while (0)
