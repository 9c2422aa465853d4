// Paged attention, split-K over KV partitions, on the CUDA cores.
//
// "How vLLM Works Internally", section "How the Kernel Works": look up the
// block table, fetch K from the scattered blocks, scores, softmax, weighted
// sum of V; the two-pass variant computes partial softmax results per
// partition and reduces them across partitions in a second pass.
//
// GB300 design (HBM-bound: ~2 flops per byte of K/V for grouped heads):
//   * Work item = (request, kv head g, row chunk, KV partition).  A row is one
//     (query token, q head of group g) pair, so each K/V page is read once
//     for all Hq/Hkv heads that share it and for all query tokens of a short
//     chunk.  Rows per item (RPI) is a template parameter.
//   * Persistent CTAs (3 per SM).  Every warp walks the request list itself
//     (a warp-wide scan over 32 requests at a time) to map its CTA's next
//     item index to (r, g, chunk, partition), so no work list is stored and
//     no planning launch is needed.
//   * One producer warp issues 3-D TMA copies of one 16-token page of one kv
//     head (box D x 1 x 16) into a 12-stage shared-memory ring, driven by the
//     block table; four consumer warps compute.  mbarriers: full (TMA bytes)
//     and empty (one arrive per consumer warp).  Every wait is bounded.
//   * Keys are processed in chunks of 256 (16 pages): all K pages of the
//     chunk -> scores in shared memory -> exact chunk max/sum, combined
//     online across chunks -> all V pages of the chunk.  QK: one warp per
//     key, D/32 dims per lane, reduce-scatter shuffles across lanes.  PV: one
//     warp per key, lanes over dims, per-warp partial accumulators combined
//     through shared memory once per item.
//   * A request whose context fits one partition writes its output directly;
//     otherwise (m, l, unnormalised o) go to the workspace and the merge
//     kernel combines them.
#include <climits>
#include <cstring>

#include "pa_internal.cuh"

namespace pa {
namespace decode {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kCtasPerSm = 3;
constexpr int kStages = 12;
constexpr int kPage = 16;         // tokens per cache block
constexpr int kChunkPages = 16;   // pages per softmax chunk
constexpr int kChunkKeys = kPage * kChunkPages;
constexpr int kCandidates = 8;    // partition lengths p_min << k
constexpr int kSingle = INT_MAX / 2;

struct Params {
    CUtensorMap tmK;
    CUtensorMap tmV;
    const void *q;
    void *out;
    const int32_t *bt;
    const int32_t *qsl;
    const int32_t *seq_lens;
    float *part_o;        // [pslot][RPI][D]
    float *part_ml;       // [pslot][RPI][2]
    int32_t *req_meta;    // [R][4]: pslot base (lo, hi), nsplit, nchunks
    long long pslot_cap;  // partial items the workspace holds
    int R, T, MB, NB, Hq, Hkv, G;
    int tau;              // requests with more query tokens are not handled here
    int p_min;            // preferred partition length in keys (multiple of 256)
    float qscale;         // softmax scale * log2(e)
    unsigned int *status;
};

template <int D, int RPI>
struct Smem {
    static constexpr int kPageBytes = kPage * D * 2;
    static constexpr int kScores = RPI * kChunkKeys;             // floats
    static constexpr int kRed = kConsumerWarps * RPI * D;        // floats
    static constexpr int kUnion = kScores > kRed ? kScores : kRed;
    static constexpr int kStageBytes = kStages * kPageBytes;
    static constexpr int kBytes = kStageBytes + kUnion * 4 + 3 * RPI * 4 + 2 * kStages * 8 +
                                  kCandidates * 8 + 16 + 128;  // + alignment slack
};

// Per-warp walk over the request list: maps a global item index to its
// request and coordinates.  All warps of all CTAs compute the same mapping.
template <int RPI>
struct Walker {
    const Params *p;
    int part;              // chosen partition length in keys
    int rb;                // first request of the current 32-request window
    long long item_base;   // items before the window
    long long pslot_base;  // partial slots before the window
    // the lane's request in the window
    int n, L, nchunks, nsplit;
    int items, incl, pincl;
    int total, ptotal;

    __device__ void load_window(int lane) {
        const int r = rb + lane;
        n = 0;
        L = 0;
        nchunks = 0;
        nsplit = 0;
        items = 0;
        if (r < p->R) {
            const int a = p->qsl[r], b = p->qsl[r + 1];
            n = b - a;
            L = p->seq_lens[r];
            const bool sane = a >= 0 && b <= p->T && n >= 0 && L >= n &&
                              (L + kPage - 1) / kPage <= p->MB;
            if (!sane) flag(p->status, PA_CHECK_SEQ_LEN);
            if (sane && n >= 1 && n <= p->tau) {
                nchunks = (n * p->G + RPI - 1) / RPI;
                nsplit = (L + part - 1) / part;
                items = p->Hkv * nchunks * nsplit;
            }
        }
        incl = items;
        pincl = nsplit > 1 ? items : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            const int w = __shfl_up_sync(0xffffffffu, pincl, o);
            if (lane >= o) {
                incl += v;
                pincl += w;
            }
        }
        total = __shfl_sync(0xffffffffu, incl, 31);
        ptotal = __shfl_sync(0xffffffffu, pincl, 31);
    }

    __device__ void begin(const Params *params, int partition, int lane) {
        p = params;
        part = partition;
        rb = 0;
        item_base = 0;
        pslot_base = 0;
        load_window(lane);
    }

    __device__ bool next_window(int lane) {
        item_base += total;
        pslot_base += ptotal;
        rb += 32;
        if (rb >= p->R) return false;
        load_window(lane);
        return true;
    }

    struct Item {
        int r, g, chunk, split, n, L, nsplit;
        long long pslot;  // -1: single partition, write the output directly
    };

    // Find item i (non-decreasing across calls).  False when past the end.
    __device__ bool find(long long i, int lane, Item &it) {
        while (i >= item_base + total)
            if (!next_window(lane)) return false;
        const int local_i = (int)(i - item_base);
        const unsigned m = __ballot_sync(0xffffffffu, incl > local_i);
        const int src = __ffs(m) - 1;
        const int excl = __shfl_sync(0xffffffffu, incl - items, src);
        const int pexcl = __shfl_sync(0xffffffffu, pincl - (nsplit > 1 ? items : 0), src);
        it.n = __shfl_sync(0xffffffffu, n, src);
        it.L = __shfl_sync(0xffffffffu, L, src);
        const int nc = __shfl_sync(0xffffffffu, nchunks, src);
        it.nsplit = __shfl_sync(0xffffffffu, nsplit, src);
        it.r = rb + src;
        const int local = local_i - excl;
        it.split = local % it.nsplit;
        const int rest = local / it.nsplit;
        it.chunk = rest % nc;
        it.g = rest / nc;
        it.pslot = it.nsplit > 1 ? pslot_base + pexcl + local : -1;
        return true;
    }
};

// Key range of an item: its partition, clipped to the context and to the
// last position any of its rows can see (causal).
template <int RPI>
__device__ __forceinline__ void item_keys(const Params &p, const typename Walker<RPI>::Item &it,
                                          int part, int &k0, int &k1) {
    const int last_row = min((it.chunk + 1) * RPI, it.n * p.G) - 1;
    const int max_pos = it.L - it.n + last_row / p.G;
    k0 = it.split * part;
    k1 = min(min(k0 + part, it.L), max_pos + 1);
}

// Reduce v[RPI] across the 32 lanes so that each row's full sum ends in the
// lanes whose low (5 - log2 RPI) bits are zero; returns the row the lane holds
// in v[0].  Each halving step trades half of the rows with the partner lane,
// so RPI rows cost RPI - 1 + (5 - log2 RPI) shuffles instead of 5 * RPI.
template <int RPI>
__device__ __forceinline__ int reduce_scatter(float (&v)[RPI], int lane) {
    int row = 0;
#pragma unroll
    for (int step = 0; (1 << step) < RPI; ++step) {
        const int half = RPI >> (step + 1);
        const int mask = 16 >> step;
        const bool upper = lane & mask;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
        if (upper) row += half;
    }
#pragma unroll
    for (int m = 32 / RPI / 2; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
    return row;
}

// Load this lane's DPL elements of a 16-bit row as floats.
template <typename T, int DPL>
__device__ __forceinline__ void load_lane(const void *row, int lane, float (&f)[DPL]) {
    if constexpr (DPL == 4) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const char *>(row) + lane * 8);
        Elt<T>::unpack2(raw.x, f[0], f[1]);
        Elt<T>::unpack2(raw.y, f[2], f[3]);
    } else {
        const uint32_t raw = *reinterpret_cast<const uint32_t *>(static_cast<const char *>(row) + lane * 4);
        Elt<T>::unpack2(raw, f[0], f[1]);
    }
}

template <typename T, int D, int RPI>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
paged_decode_kernel(const __grid_constant__ Params p) {
    using S = Smem<D, RPI>;
    constexpr int DPL = D / 32;  // dims per lane
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    unsigned char *stages = base;
    float *uni = reinterpret_cast<float *>(base + S::kStageBytes);
    float *row_m = uni + S::kUnion;
    float *row_l = row_m + RPI;
    float *row_a = row_l + RPI;
    uint64_t *full = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(row_a + RPI) + 7) & ~uintptr_t(7));
    uint64_t *empty = full + kStages;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(empty + kStages);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid < kCandidates) cand[tid] = 0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensor_map(&p.tmK);
        prefetch_tensor_map(&p.tmV);
    }
    __syncthreads();

    // ---- choose the partition length: the shortest candidate whose partial
    //      results fit the workspace (every CTA reaches the same answer).
    {
        unsigned long long local[kCandidates];
#pragma unroll
        for (int k = 0; k < kCandidates; ++k) local[k] = 0;
        if (p.p_min < kSingle) {
            for (int r = tid; r < p.R; r += kThreads) {
                const int a = p.qsl[r], b = p.qsl[r + 1];
                const int n = b - a;
                const int L = p.seq_lens[r];
                if (a < 0 || b > p.T || n < 1 || n > p.tau || L < n ||
                    (L + kPage - 1) / kPage > p.MB)
                    continue;
                const long long per = (long long)p.Hkv * ((n * p.G + RPI - 1) / RPI);
#pragma unroll
                for (int k = 0; k < kCandidates; ++k) {
                    const long long part = (long long)p.p_min << k;
                    const long long ns = (L + part - 1) / part;
                    if (ns > 1) local[k] += per * ns;
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kCandidates; ++k)
            if (local[k]) atomicAdd(&cand[k], local[k]);
    }
    __syncthreads();
    int part = kSingle;
    if (p.p_min < kSingle) {
        for (int k = kCandidates - 1; k >= 0; --k)
            if (cand[k] <= (unsigned long long)p.pslot_cap) part = p.p_min << k;
    }

    // ---- CTA 0 records, per request, where its partials live (merge pass).
    if (blockIdx.x == 0 && warp == 0 && p.req_meta != nullptr) {
        Walker<RPI> w;
        w.begin(&p, part, lane);
        do {
            const int r = w.rb + lane;
            if (r < p.R) {
                const long long pb = w.pslot_base + w.pincl - (w.nsplit > 1 ? w.items : 0);
                reinterpret_cast<int4 *>(p.req_meta)[r] =
                    make_int4((int)(pb & 0xffffffff), (int)(pb >> 32), w.nsplit, w.nchunks);
            }
        } while (w.next_window(lane));
    }

    Walker<RPI> walk;
    walk.begin(&p, part, lane);
    typename Walker<RPI>::Item it;

    if (warp == kConsumerWarps) {
        // =================== producer warp ===================
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long i = blockIdx.x; ok && walk.find(i, lane, it); i += gridDim.x) {
            int k0, k1;
            item_keys<RPI>(p, it, part, k0, k1);
            const int32_t *row = p.bt + (long long)it.r * p.MB;
            for (int c0 = k0; ok && c0 < k1; c0 += kChunkKeys) {
                const int npages = (min(c0 + kChunkKeys, k1) - c0 + kPage - 1) / kPage;
                int blk = 0;
                if (lane < npages) {
                    blk = row[c0 / kPage + lane];
                    if (blk < 0 || blk >= p.NB) {
                        flag(p.status, PA_CHECK_BLOCK_ID);
                        blk = 0;
                    }
                }
                for (int kv = 0; ok && kv < 2; ++kv) {
                    for (int pg = 0; pg < npages; ++pg) {
                        const int b = __shfl_sync(0xffffffffu, blk, pg);
                        if (lane == 0) {
                            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                                flag(p.status, PA_CHECK_TIMEOUT);
                                ok = false;
                            } else {
                                mbar_arrive_expect_tx(&full[stage], S::kPageBytes);
                                tma_load_3d(stages + stage * S::kPageBytes, kv ? &p.tmV : &p.tmK,
                                            &full[stage], 0, it.g, b * kPage);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) break;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
        }
        // Drain: wait (bounded) until the consumers have released every stage,
        // so no copy is still landing when the CTA exits.
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s) {
                if (!mbar_wait(&empty[stage], phase ^ 1)) {
                    flag(p.status, PA_CHECK_TIMEOUT);
                    break;
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        return;
    }

    // =================== consumer warps ===================
    const T *q = reinterpret_cast<const T *>(p.q);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (long long i = blockIdx.x; ok && walk.find(i, lane, it); i += gridDim.x) {
        int k0, k1;
        item_keys<RPI>(p, it, part, k0, k1);
        const int qstart = p.qsl[it.r];
        const int nrows = it.n * p.G;
        const int pos0 = it.L - it.n;  // position of the request's first query token

        // Q rows of this item, this lane's dims, pre-scaled by scale*log2(e).
        float qr[RPI][DPL];
#pragma unroll
        for (int j = 0; j < RPI; ++j) {
            const int rr = it.chunk * RPI + j;
            if (rr < nrows) {
                const int h = it.g * p.G + rr % p.G;
                load_lane<T, DPL>(q + ((long long)(qstart + rr / p.G) * p.Hq + h) * D, lane, qr[j]);
#pragma unroll
                for (int d = 0; d < DPL; ++d) qr[j][d] *= p.qscale;
            } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) qr[j][d] = 0.f;
            }
        }
        float acc[RPI][DPL];
#pragma unroll
        for (int j = 0; j < RPI; ++j)
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[j][d] = 0.f;
        if (tid < RPI) {
            row_m[tid] = -INFINITY;
            row_l[tid] = 0.f;
        }

        for (int c0 = k0; ok && c0 < k1; c0 += kChunkKeys) {
            const int nkeys = min(c0 + kChunkKeys, k1) - c0;
            const int npages = (nkeys + kPage - 1) / kPage;
            // ---- scores for the chunk's keys
            for (int pg = 0; pg < npages; ++pg) {
                if (!mbar_wait(&full[stage], phase)) {
                    flag(p.status, PA_CHECK_TIMEOUT);
                    ok = false;
                    break;
                }
                const unsigned char *page = stages + stage * S::kPageBytes;
#pragma unroll
                for (int u = 0; u < kPage / kConsumerWarps; ++u) {
                    const int tk = warp + u * kConsumerWarps;
                    float kf[DPL];
                    load_lane<T, DPL>(page + tk * D * 2, lane, kf);
                    float s[RPI];
#pragma unroll
                    for (int j = 0; j < RPI; ++j) {
                        float a = 0.f;
#pragma unroll
                        for (int d = 0; d < DPL; ++d) a = fmaf(qr[j][d], kf[d], a);
                        s[j] = a;
                    }
                    const int row = reduce_scatter<RPI>(s, lane);
                    if ((lane & (32 / RPI - 1)) == 0) {
                        const int kk = pg * kPage + tk;
                        const int rr = it.chunk * RPI + row;
                        const bool vis =
                            rr < nrows && c0 + kk < k1 && c0 + kk <= pos0 + rr / p.G;
                        uni[row * kChunkKeys + kk] = vis ? s[0] : -INFINITY;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            named_bar_sync(1, kConsumers);
            // ---- online softmax update, one warp per row
            for (int j = warp; j < RPI; j += kConsumerWarps) {
                float *srow = uni + j * kChunkKeys;
                float mx = -INFINITY;
                for (int k = lane; k < nkeys; k += 32) mx = fmaxf(mx, srow[k]);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = row_m[j];
                const float m_new = fmaxf(m_old, mx);
                float sum = 0.f;
                for (int k = lane; k < nkeys; k += 32) {
                    const float e = m_new == -INFINITY ? 0.f : fast_exp2(srow[k] - m_new);
                    srow[k] = e;
                    sum += e;
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                if (lane == 0) {
                    const float alpha = m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new);
                    row_a[j] = alpha;
                    row_l[j] = row_l[j] * alpha + sum;
                    row_m[j] = m_new;
                }
            }
            named_bar_sync(1, kConsumers);
#pragma unroll
            for (int j = 0; j < RPI; ++j) {
                const float a = row_a[j];
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[j][d] *= a;
            }
            // ---- weighted sum of the chunk's values
            for (int pg = 0; pg < npages; ++pg) {
                if (!mbar_wait(&full[stage], phase)) {
                    flag(p.status, PA_CHECK_TIMEOUT);
                    ok = false;
                    break;
                }
                const unsigned char *page = stages + stage * S::kPageBytes;
#pragma unroll
                for (int u = 0; u < kPage / kConsumerWarps; ++u) {
                    const int tk = warp + u * kConsumerWarps;
                    const int kk = pg * kPage + tk;
                    if (c0 + kk < k1) {  // never touch slots past the context
                        float vf[DPL];
                        load_lane<T, DPL>(page + tk * D * 2, lane, vf);
#pragma unroll
                        for (int j = 0; j < RPI; ++j) {
                            const float pj = uni[j * kChunkKeys + kk];
#pragma unroll
                            for (int d = 0; d < DPL; ++d) acc[j][d] = fmaf(pj, vf[d], acc[j][d]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            named_bar_sync(1, kConsumers);  // the chunk's weights are no longer read
        }
        if (!ok) break;

        // ---- combine the consumer warps' partial sums and write the item out
#pragma unroll
        for (int j = 0; j < RPI; ++j)
#pragma unroll
            for (int d = 0; d < DPL; ++d) uni[(warp * RPI + j) * D + lane * DPL + d] = acc[j][d];
        named_bar_sync(1, kConsumers);
        for (int o = tid; o < RPI * D / 2; o += kConsumers) {
            const int j = o / (D / 2);
            const int d = (o % (D / 2)) * 2;
            const int rr = it.chunk * RPI + j;
            if (rr >= nrows) continue;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                s0 += uni[(w * RPI + j) * D + d];
                s1 += uni[(w * RPI + j) * D + d + 1];
            }
            if (it.pslot < 0) {
                const float inv = 1.f / row_l[j];
                const int h = it.g * p.G + rr % p.G;
                T *dst = reinterpret_cast<T *>(p.out) +
                         ((long long)(qstart + rr / p.G) * p.Hq + h) * D + d;
                *reinterpret_cast<uint32_t *>(dst) = Elt<T>::pack2(s0 * inv, s1 * inv);
            } else {
                float *po = p.part_o + (it.pslot * RPI + j) * D + d;
                *reinterpret_cast<float2 *>(po) = make_float2(s0, s1);
                if (d == 0) {
                    *reinterpret_cast<float2 *>(p.part_ml + (it.pslot * RPI + j) * 2) =
                        make_float2(row_m[j], row_l[j]);
                }
            }
        }
        named_bar_sync(1, kConsumers);  // the union buffer is free again
    }
    // Consumers that stop early (a timed-out wait) release every stage once so
    // the producer's bounded drain can finish.
    if (!ok && lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_arrive(&empty[s]);
    }
}

// Second pass: for each (token, q head) of a request whose context was split,
// combine the partitions' (m, l, o): M = max m_s, o = sum 2^(m_s-M) o_s /
// sum 2^(m_s-M) l_s.  One CTA per token, one warp per head.
template <typename T, int D, int RPI>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ Params p) {
    constexpr int DPL = D / 32;
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ int s_r;
    if (threadIdx.x == 0) {
        // the last request whose start is <= t
        int lo = 0, hi = p.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.qsl[mid] <= t) lo = mid;
            else hi = mid - 1;
        }
        s_r = lo;
    }
    __syncthreads();
    const int r = s_r;
    const int4 meta = reinterpret_cast<const int4 *>(p.req_meta)[r];
    const int nsplit = meta.z, nchunks = meta.w;
    if (nsplit <= 1) return;
    const int tl = t - p.qsl[r];
    if (tl < 0 || tl >= p.qsl[r + 1] - p.qsl[r]) return;
    const long long pbase = (long long)(unsigned)meta.x | ((long long)meta.y << 32);
    for (int h = warp; h < p.Hq; h += 8) {
        const int g = h / p.G;
        const int rr = tl * p.G + h % p.G;
        const int chunk = rr / RPI, j = rr % RPI;
        const long long first = pbase + ((long long)g * nchunks + chunk) * nsplit;
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.part_ml[((first + s) * RPI + j) * 2]);
        float o[DPL];
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[d] = 0.f;
        float Lsum = 0.f;
        for (int s = 0; s < nsplit; ++s) {
            const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + ((first + s) * RPI + j) * 2);
            const float w = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
            Lsum += w * ml.y;
            const float *po = p.part_o + ((first + s) * RPI + j) * D + lane * DPL;
#pragma unroll
            for (int d = 0; d < DPL; ++d) o[d] = fmaf(w, po[d], o[d]);
        }
        const float inv = 1.f / Lsum;
        T *dst = reinterpret_cast<T *>(p.out) + ((long long)t * p.Hq + h) * D + lane * DPL;
#pragma unroll
        for (int d = 0; d < DPL; d += 2)
            *reinterpret_cast<uint32_t *>(dst + d) = Elt<T>::pack2(o[d] * inv, o[d + 1] * inv);
    }
}

template <typename T, int D, int RPI>
pa_status launch_typed(Params &prm, int grid, bool merge, cudaStream_t stream) {
    using S = Smem<D, RPI>;
    static bool configured[64] = {};
    int dev = 0;
    PA_TRY_CUDA(cudaGetDevice(&dev));
    if (dev >= 64 || !configured[dev]) {
        PA_TRY_CUDA(cudaFuncSetAttribute(paged_decode_kernel<T, D, RPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes));
        if (dev < 64) configured[dev] = true;
    }
    paged_decode_kernel<T, D, RPI><<<grid, kThreads, S::kBytes, stream>>>(prm);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    if (merge && prm.T > 0) {
        merge_kernel<T, D, RPI><<<prm.T, 256, 0, stream>>>(prm);
        PA_TRY_CUDA(cudaGetLastError());
        note_launch();
    }
    return PA_OK;
}

template <typename T, int D>
pa_status dispatch_rpi(int rpi, Params &prm, int grid, bool merge, cudaStream_t stream) {
    switch (rpi) {
        case 1: return launch_typed<T, D, 1>(prm, grid, merge, stream);
        case 2: return launch_typed<T, D, 2>(prm, grid, merge, stream);
        case 4: return launch_typed<T, D, 4>(prm, grid, merge, stream);
        default: return launch_typed<T, D, 8>(prm, grid, merge, stream);
    }
}

// Rows per item: enough for all heads of a group and a few query tokens, at
// most 8 (register budget).
inline int rows_per_item(int G, int max_q) {
    const long long rows = (long long)G * (max_q > 0 ? max_q : 1);
    int rpi = 1;
    while (rpi < 8 && rpi < rows) rpi <<= 1;
    return rpi;
}

constexpr int kPreferredPartition = 512;
constexpr size_t kAlign = 256;

inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace decode

size_t decode_workspace_size(int32_t R, int32_t T, int32_t max_q, int32_t max_seq, int32_t Hq,
                             int32_t Hkv, int32_t D) {
    using namespace decode;
    if (R <= 0 || Hkv <= 0) return 0;
    const int G = Hq / Hkv;
    const int rpi = rows_per_item(G, max_q);
    const size_t meta = round_up((size_t)R * 16);
    const long long splits = (max_seq + kPreferredPartition - 1) / kPreferredPartition;
    if (splits <= 1) return meta;
    // every request's rows, in chunks of rpi, for every kv head and partition
    const long long chunks = (long long)R + ((long long)T * G + rpi - 1) / rpi;
    const long long items = (long long)Hkv * chunks * splits;
    const size_t bytes = meta + round_up((size_t)items * rpi * 2 * sizeof(float)) +
                         (size_t)items * rpi * D * sizeof(float);
    const size_t cap = (size_t)1 << 30;  // past this, longer partitions instead
    return bytes < cap ? bytes : cap;
}

pa_status launch_decode(const AttnArgs &a, cudaStream_t stream) {
    using namespace decode;
    Params prm;
    memset(&prm, 0, sizeof prm);
    const int64_t slots = (int64_t)a.NB * a.bs;
    if (!encode_pool_map(&prm.tmK, a.kc, slots, a.Hkv, a.D, kPage) ||
        !encode_pool_map(&prm.tmV, a.vc, slots, a.Hkv, a.D, kPage))
        return PA_ERR_CUDA;
    prm.q = a.q;
    prm.out = a.out;
    prm.bt = a.bt;
    prm.qsl = a.qsl;
    prm.seq_lens = a.seq_lens;
    prm.R = a.R;
    prm.T = a.T;
    prm.MB = a.MB;
    prm.NB = a.NB;
    prm.Hq = a.Hq;
    prm.Hkv = a.Hkv;
    prm.G = a.Hq / a.Hkv;
    prm.tau = INT_MAX;
    prm.qscale = a.scale * 1.4426950408889634f;
    prm.status = status_word();
    if (!prm.status) return PA_ERR_CUDA;
    const int rpi = rows_per_item(prm.G, a.max_q);

    // Workspace: per-request metadata, then (m, l) and o partials.
    const size_t meta = round_up((size_t)a.R * 16);
    bool merge = false;
    prm.p_min = kSingle;
    if (a.ws && a.ws_bytes > meta && a.max_seq > kPreferredPartition) {
        const size_t rest = a.ws_bytes - meta;
        const size_t per = (size_t)rpi * (a.D + 2) * sizeof(float);
        long long cap = (long long)(rest / per);
        while (cap > 0 && round_up((size_t)cap * rpi * 2 * sizeof(float)) +
                                  (size_t)cap * rpi * a.D * sizeof(float) > rest)
            --cap;
        if (cap > 0) {
            unsigned char *w = static_cast<unsigned char *>(a.ws);
            prm.req_meta = reinterpret_cast<int32_t *>(w);
            prm.part_ml = reinterpret_cast<float *>(w + meta);
            prm.part_o = reinterpret_cast<float *>(
                w + meta + round_up((size_t)cap * rpi * 2 * sizeof(float)));
            prm.pslot_cap = cap;
            prm.p_min = kPreferredPartition;
            merge = true;
        }
    }

    // Grid: persistent, kCtasPerSm per SM, no more CTAs than there can be items.
    const long long splits = prm.p_min >= kSingle ? 1 : (a.max_seq + prm.p_min - 1) / prm.p_min;
    const long long chunks = (long long)a.R + ((long long)a.T * prm.G + rpi - 1) / rpi;
    const long long ub = (long long)a.Hkv * chunks * splits;
    long long grid = (long long)kCtasPerSm * num_sms();
    if (ub < grid) grid = ub;
    if (grid < 1) grid = 1;

    const bool bf16 = a.dtype == PA_BF16;
    if (a.D == 128)
        return bf16 ? dispatch_rpi<__nv_bfloat16, 128>(rpi, prm, (int)grid, merge, stream)
                    : dispatch_rpi<__half, 128>(rpi, prm, (int)grid, merge, stream);
    return bf16 ? dispatch_rpi<__nv_bfloat16, 64>(rpi, prm, (int)grid, merge, stream)
                : dispatch_rpi<__half, 64>(rpi, prm, (int)grid, merge, stream);
}

}  // namespace pa
