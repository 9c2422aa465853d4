// Index build and KV cache write in one launch: the results of
// pa_prepare_inputs followed by pa_cache_write_ex on the same stream.
//
// "Building the Batch", sections "How they are computed" (the index tensors
// and slot = block_table[pos / bs] * bs + pos % bs) and "Reading and writing
// the KV cache"; "Inside vLLM: Following One Request", the write op (token
// i's K and V rows go to slot slot_mapping[i], before attention reads the
// cache); "How vLLM Works Internally", section "Fused Kernels" (one launch
// and no round trip of slot_mapping through global memory between the two).
//
// Every CTA scans num_scheduled_tokens in shared memory as the index build
// does (the request count is small); CTA 0 writes the per-request outputs.
// Then one warp per token: its K and V rows' first units loaded, its request
// by binary search, its position and slot (lane 0 stores the three indices),
// and the rows stored at that slot by the whole warp -- 16-byte vectors of
// 16-bit pools, or eight elements quantised to E4M3 per lane and unit for FP8
// pools.  The grid is sized for the copy, not for the index build alone.
#include "pa_internal.cuh"

namespace pa {

constexpr int kFusedThreads = 256;
constexpr int kFusedCtasPerSm = 4;   // 32 warps an SM, 64 registers a thread
constexpr int kUnroll = 4;   // 16-byte units of each row in flight per lane

struct WriteArgs {
    const void *key, *value;  // [T] rows of Hkv*D elements, `stride` elements apart
    int64_t stride;
    void *kc, *vc;            // pools [NB*bs][Hkv*D]
    int32_t row;              // elements per row (Hkv*D)
    const float *k_scale, *v_scale;  // FP8 pools only (NULL = 1)
};

// kMode 0: 16-bit pools (a row is row * 2 / 16 16-byte vectors); 1: FP8
// pools, bf16 source; 2: FP8 pools, fp16 source.
template <int kMode>
__global__ void __launch_bounds__(kFusedThreads, kFusedCtasPerSm)
prepare_write_kernel(const PrepArgs a, const WriteArgs w, unsigned int *status) {
    extern __shared__ int32_t s_start[];  // [R + 1]: first flat token of each request
    __shared__ int32_t s_scan[33];
    const int tid = threadIdx.x, lane = tid & 31;
    const int nthreads = blockDim.x;
    const int R = a.R;

    // The warp's first token's K and V row units are loaded before the scan:
    // their addresses depend only on the token, so the copy's first memory
    // round trip overlaps the scan's.
    using Src = uint4;
    using Dst = typename std::conditional<kMode == 0, uint4, uint2>::type;
    const int nu = w.row / 8;   // 16-byte source units per row (and pool units)
    Src kx[kUnroll], vx[kUnroll];
    auto load_first = [&](long long t) {
        const Src *ksrc = static_cast<const Src *>(w.key) + t * (w.stride / 8);
        const Src *vsrc = static_cast<const Src *>(w.value) + t * (w.stride / 8);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (lane + 32 * u < nu) {
                kx[u] = __ldg(ksrc + lane + 32 * u);
                vx[u] = __ldg(vsrc + lane + 32 * u);
            }
    };
    const long long t_first = (long long)blockIdx.x * (nthreads / 32) + (tid >> 5);
    if (t_first < a.T) load_first(t_first);

    // ---- the scan of num_scheduled_tokens, as in the index build
    const int per = (R + nthreads - 1) / nthreads;
    const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
    int local = 0;
    bool empty_req = false;
    for (int r = r0; r < r1; ++r) {
        const int n = a.nst[r];
        if (n <= 0) empty_req = true;
        local += max(n, 0);
    }
    int total = 0;
    int run = block_exclusive_scan(local, s_scan, total);
    for (int r = r0; r < r1; ++r) {
        s_start[r] = run;
        run += max(a.nst[r], 0);
    }
    if (tid == 0) s_start[R] = total;
    __syncthreads();

    if (blockIdx.x == 0) {
        for (int r = tid; r < R; r += nthreads) {
            const int n = max(a.nst[r], 0);
            a.qsl[r] = s_start[r];
            a.seq_lens[r] = a.nct[r] + n;
            a.logits[r] = s_start[r] + n - 1;
        }
        for (int i = R + tid; i < a.qsl_cap; i += nthreads) a.qsl[i] = i == R ? total : a.T;
        if (tid == 0 && total != a.T) flag(status, PA_CHECK_TOKEN_COUNT);
    }
    if (empty_req) flag(status, PA_CHECK_EMPTY_REQUEST);

    // ---- one warp per token: indices, then the row copy
    const float ks = (kMode != 0 && w.k_scale) ? *w.k_scale : 1.f;
    const float vs = (kMode != 0 && w.v_scale) ? *w.v_scale : 1.f;
    const long long nwarps = (long long)gridDim.x * (nthreads / 32);
    for (long long t = t_first; t < a.T; t += nwarps) {
        if (t >= total || R == 0) {
            if (lane == 0) {
                a.req[t] = -1;
                a.pos[t] = -1;
                a.slot[t] = -1;
            }
            continue;
        }
        // A later token's first row units are loaded before its slot is
        // known (their addresses do not depend on it): the latencies overlap.
        if (t != t_first) load_first(t);
        const Src *ksrc = static_cast<const Src *>(w.key) + t * (w.stride / 8);
        const Src *vsrc = static_cast<const Src *>(w.value) + t * (w.stride / 8);
        // The request holding t: the last one whose start is <= t (every
        // lane searches, so the result needs no broadcast).
        int lo = 0, hi = R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_start[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo;
        const int p = a.nct[r] + ((int)t - s_start[r]);
        int s = -1;
        const int logical = p >= 0 ? p / a.bs : -1;
        if (logical < 0 || logical >= a.MB) {
            if (lane == 0) flag(status, PA_CHECK_LOGICAL_BLOCK);
        } else {
            const int phys = a.bt[(long long)r * a.MB + logical];
            if (phys < 0 || phys >= a.NB) {
                if (lane == 0) flag(status, PA_CHECK_BLOCK_ID);
            } else {
                s = phys * a.bs + p % a.bs;
            }
        }
        if (lane == 0) {
            a.req[t] = r;
            a.pos[t] = p;
            a.slot[t] = s;
        }
        if (s < 0) continue;   // no write for a token without a slot
        Dst *kd = static_cast<Dst *>(w.kc) + (int64_t)s * nu;
        Dst *vd = static_cast<Dst *>(w.vc) + (int64_t)s * nu;
        for (int i = lane;; i += 32 * kUnroll) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i + 32 * u < nu) {
                    if constexpr (kMode == 0) {
                        kd[i + 32 * u] = kx[u];
                        vd[i + 32 * u] = vx[u];
                    } else {
                        using T = typename std::conditional<kMode == 1, __nv_bfloat16, __half>::type;
                        kd[i + 32 * u] = quantize8_e4m3<T>(kx[u], ks);
                        vd[i + 32 * u] = quantize8_e4m3<T>(vx[u], vs);
                    }
                }
            if (i + 32 * kUnroll >= nu) break;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (i + 32 * (kUnroll + u) < nu) {
                    kx[u] = __ldg(ksrc + i + 32 * (kUnroll + u));
                    vx[u] = __ldg(vsrc + i + 32 * (kUnroll + u));
                }
        }
    }
}

pa_status launch_prepare_write(const PrepArgs &a, const void *key, const void *value,
                               int64_t stride_elems, void *kc, void *vc, int32_t row_elems,
                               pa_dtype dtype, pa_dtype cache_dtype, const float *k_scale,
                               const float *v_scale, cudaStream_t stream) {
    constexpr int kMaxReqs = 50000;
    if (a.R > kMaxReqs) return PA_ERR_UNSUPPORTED;
    const bool fp8 = cache_dtype == PA_FP8_E4M3;
    // 16-byte source rows; 16-byte (16-bit pools) or 8-byte (FP8) pool rows.
    const uintptr_t src = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                          (uintptr_t)(stride_elems * 2) | (uintptr_t)(row_elems * 2);
    const uintptr_t dst = reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc) |
                          (uintptr_t)(row_elems * (fp8 ? 1 : 2));
    if (a.T > 0 && ((src & 15) != 0 || (dst & (fp8 ? 7 : 15)) != 0)) return PA_ERR_UNSUPPORTED;
    const size_t smem = ((size_t)a.R + 1) * sizeof(int32_t);
    auto kernel = fp8 ? (dtype == PA_BF16 ? prepare_write_kernel<1> : prepare_write_kernel<2>)
                      : prepare_write_kernel<0>;
    if (smem > 48 * 1024)
        PA_TRY_CUDA(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem));
    const int warps = kFusedThreads / 32;
    long long blocks = ((long long)a.T + warps - 1) / warps;
    const long long cap = (long long)kFusedCtasPerSm * num_sms();   // one wave
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    WriteArgs w{key, value, stride_elems, kc, vc, row_elems, k_scale, v_scale};
    kernel<<<(int)blocks, kFusedThreads, smem, stream>>>(a, w, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
