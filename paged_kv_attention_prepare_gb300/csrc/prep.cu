// Index build for one step ("Building the Batch", sections "How they are
// computed", "Reading and writing the KV cache" and "Only one row per request
// reaches the vocabulary"; "vLLM's Model Runner", sections "The two things
// this method returns" and "The batch contains rows that must not be
// sampled").
//
// One launch.  Every CTA recomputes the exclusive scan of
// num_scheduled_tokens in shared memory (a block-wide warp-shuffle scan; the
// request count is small), so no CTA waits on another.  CTA 0 writes the
// per-request outputs (query_start_loc with its padded tail, seq_lens, the
// discard mask, the sampled rows with their own scan over drafts + 1); all
// CTAs then stride over the flat tokens, find each token's request by binary
// search in the scanned starts, and write req_indices, positions,
// slot_mapping and, when a token buffer is given, token_indices and input_ids.
#include "pa_internal.cuh"

namespace pa {

constexpr int kPrepThreads = 1024;
constexpr int kPrepMaxReqs = 50000;

__global__ void __launch_bounds__(kPrepThreads)
prepare_inputs_kernel(const PrepArgs a, unsigned int *status) {
    extern __shared__ int32_t s_start[];  // [R + 1]: first flat token of each request
    __shared__ int32_t s_scan[33];
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int R = a.R;

    // Each thread owns a contiguous run of requests.
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
            // Sampled anyway, thrown away later: the request has not reached
            // its known token count yet.
            if (a.discard)
                a.discard[r] = (int64_t)a.nct[r] + n < (int64_t)a.req_num_tokens[r] ? 1 : 0;
            if (!a.num_draft) {
                a.logits[r] = s_start[r] + n - 1;
                if (a.cu_logits) a.cu_logits[r] = r;
            }
        }
        if (!a.num_draft && a.cu_logits && tid == 0) a.cu_logits[R] = R;
        // Entry R holds the total; the tail up to the capacity holds T so the
        // array never decreases.
        for (int i = R + tid; i < a.qsl_cap; i += nthreads) a.qsl[i] = i == R ? total : a.T;
        if (tid == 0 && total != a.T) flag(status, PA_CHECK_TOKEN_COUNT);

        if (a.num_draft) {
            // Request r verifies d drafts: d + 1 rows, the last d + 1 of its
            // slice, starting at the exclusive scan of (d + 1).
            int lrows = 0;
            bool bad_draft = false;
            for (int r = r0; r < r1; ++r) {
                const int n = max(a.nst[r], 0);
                int d = a.num_draft[r];
                if (d < 0 || d + 1 > n) {
                    bad_draft = true;
                    d = d < 0 ? 0 : max(n - 1, 0);
                }
                lrows += d + 1;
            }
            int rows_total = 0;
            int row = block_exclusive_scan(lrows, s_scan, rows_total);
            for (int r = r0; r < r1; ++r) {
                const int n = max(a.nst[r], 0);
                const int d = min(max(a.num_draft[r], 0), max(n - 1, 0));
                if (a.cu_logits) a.cu_logits[r] = row;
                const int last = s_start[r] + n - 1;
                for (int k = 0; k <= d; ++k, ++row)
                    if (row < a.num_logits) a.logits[row] = last - d + k;
            }
            if (tid == 0) {
                if (a.cu_logits) a.cu_logits[R] = rows_total;
                if (rows_total != a.num_logits) flag(status, PA_CHECK_DRAFT_COUNT);
            }
            if (bad_draft) flag(status, PA_CHECK_DRAFT_COUNT);
        }
    }
    if (empty_req) flag(status, PA_CHECK_EMPTY_REQUEST);

    const bool gather = a.M > 0;
    for (int t = blockIdx.x * nthreads + tid; t < a.T; t += gridDim.x * nthreads) {
        if (t >= total || R == 0) {
            a.req[t] = -1;
            a.pos[t] = -1;
            a.slot[t] = -1;
            if (gather) {
                a.token_indices[t] = -1;
                a.input_ids[t] = -1;
            }
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
        const int p = a.nct[r] + (t - s_start[r]);
        a.req[t] = r;
        a.pos[t] = p;
        int s = -1;
        const int logical = p >= 0 ? p / a.bs : -1;
        if (logical < 0 || logical >= a.MB) {
            flag(status, PA_CHECK_LOGICAL_BLOCK);
        } else {
            const int phys = a.bt[(long long)r * a.MB + logical];
            if (phys < 0 || phys >= a.NB) flag(status, PA_CHECK_BLOCK_ID);
            else s = phys * a.bs + p % a.bs;
        }
        a.slot[t] = s;
        if (gather) {
            // Row r of the token buffer holds request r's ids; position p sits
            // at flat offset r * M + p.
            if (r >= a.max_num_reqs || p < 0 || p >= a.M) {
                flag(status, PA_CHECK_TOKEN_INDEX);
                a.token_indices[t] = -1;
                a.input_ids[t] = -1;
            } else {
                const int64_t ti = (int64_t)r * a.M + p;
                a.token_indices[t] = ti;
                a.input_ids[t] = a.token_ids[ti];
            }
        }
    }
}

pa_status launch_prepare(const PrepArgs &a, cudaStream_t stream) {
    if (a.R > kPrepMaxReqs) return PA_ERR_UNSUPPORTED;
    const size_t smem = ((size_t)a.R + 1) * sizeof(int32_t);
    if (smem > 48 * 1024) {
        PA_TRY_CUDA(cudaFuncSetAttribute(prepare_inputs_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    }
    long long blocks = ((long long)a.T + kPrepThreads - 1) / kPrepThreads;
    const long long cap = 2LL * num_sms();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    prepare_inputs_kernel<<<(int)blocks, kPrepThreads, smem, stream>>>(a, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
