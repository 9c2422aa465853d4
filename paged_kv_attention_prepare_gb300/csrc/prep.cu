// Index build for one step ("Building the Batch", sections "How they are
// computed" and "Reading and writing the KV cache"; "vLLM's Model Runner",
// section "The two things this method returns").
//
// One launch.  Every CTA recomputes the exclusive scan of
// num_scheduled_tokens in shared memory (a block-wide warp-shuffle scan; the
// request count is small), so no CTA waits on another.  CTA 0 writes the
// per-request outputs (query_start_loc with its padded tail, seq_lens,
// logits_indices); all CTAs then stride over the flat tokens, find each
// token's request by binary search in the scanned starts, and write
// req_indices, positions and slot_mapping.
#include "pa_internal.cuh"

namespace pa {

constexpr int kPrepThreads = 1024;
constexpr int kPrepMaxReqs = 50000;

__global__ void __launch_bounds__(kPrepThreads)
prepare_inputs_kernel(const int32_t *__restrict__ nst, const int32_t *__restrict__ nct,
                      const int32_t *__restrict__ bt, int32_t R, int32_t MB, int32_t bs,
                      int32_t T, int32_t NB, int32_t *__restrict__ req,
                      int32_t *__restrict__ pos, int32_t *__restrict__ slot,
                      int32_t *__restrict__ qsl, int32_t qsl_cap, int32_t *__restrict__ seq_lens,
                      int32_t *__restrict__ logits, unsigned int *status) {
    extern __shared__ int32_t s_start[];  // [R + 1]: first flat token of each request
    __shared__ int32_t s_warp[kPrepThreads / 32];
    __shared__ int32_t s_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads >> 5;

    // Each thread owns a contiguous run of requests.
    const int per = (R + nthreads - 1) / nthreads;
    const int r0 = min(R, tid * per), r1 = min(R, r0 + per);
    int local = 0;
    bool empty_req = false;
    for (int r = r0; r < r1; ++r) {
        const int n = nst[r];
        if (n <= 0) empty_req = true;
        local += max(n, 0);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < nwarps ? s_warp[lane] : 0;
        int w = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < nwarps) s_warp[lane] = w - v;
        if (lane == 31) s_total = w;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - local;
    for (int r = r0; r < r1; ++r) {
        s_start[r] = run;
        run += max(nst[r], 0);
    }
    const int total = s_total;
    if (tid == 0) s_start[R] = total;
    __syncthreads();

    if (blockIdx.x == 0) {
        for (int r = tid; r < R; r += nthreads) {
            const int n = max(nst[r], 0);
            qsl[r] = s_start[r];
            seq_lens[r] = nct[r] + n;
            logits[r] = s_start[r] + n - 1;
        }
        // Entry R holds the total; the tail up to the capacity holds T so the
        // array never decreases.
        for (int i = R + tid; i < qsl_cap; i += nthreads) qsl[i] = i == R ? total : T;
        if (tid == 0 && total != T) flag(status, PA_CHECK_TOKEN_COUNT);
    }
    if (empty_req) flag(status, PA_CHECK_EMPTY_REQUEST);

    for (int t = blockIdx.x * nthreads + tid; t < T; t += gridDim.x * nthreads) {
        if (t >= total || R == 0) {
            req[t] = -1;
            pos[t] = -1;
            slot[t] = -1;
            continue;
        }
        // The request holding t: the last one whose start is <= t.
        int lo = 0, hi = R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_start[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo;
        const int p = nct[r] + (t - s_start[r]);
        req[t] = r;
        pos[t] = p;
        int s = -1;
        const int logical = p >= 0 ? p / bs : -1;
        if (logical < 0 || logical >= MB) {
            flag(status, PA_CHECK_LOGICAL_BLOCK);
        } else {
            const int phys = bt[(long long)r * MB + logical];
            if (phys < 0 || phys >= NB) flag(status, PA_CHECK_BLOCK_ID);
            else s = phys * bs + p % bs;
        }
        slot[t] = s;
    }
}

pa_status launch_prepare(const int32_t *nst, const int32_t *nct, const int32_t *bt, int32_t R,
                         int32_t MB, int32_t bs, int32_t T, int32_t NB, int32_t *req,
                         int32_t *pos, int32_t *slot, int32_t *qsl, int32_t qsl_cap,
                         int32_t *seq_lens, int32_t *logits, cudaStream_t stream) {
    if (R > kPrepMaxReqs) return PA_ERR_UNSUPPORTED;
    const size_t smem = ((size_t)R + 1) * sizeof(int32_t);
    if (smem > 48 * 1024) {
        PA_TRY_CUDA(cudaFuncSetAttribute(prepare_inputs_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    }
    long long blocks = ((long long)T + kPrepThreads - 1) / kPrepThreads;
    const long long cap = 2LL * num_sms();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    prepare_inputs_kernel<<<(int)blocks, kPrepThreads, smem, stream>>>(
        nst, nct, bt, R, MB, bs, T, NB, req, pos, slot, qsl, qsl_cap, seq_lens, logits, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
