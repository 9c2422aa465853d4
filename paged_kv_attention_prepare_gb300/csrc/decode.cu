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
//   * Persistent CTAs (3 per SM; 2 for 8-row items, which need more registers).  Every warp walks the request list itself
//     (a warp-wide scan over 32 requests at a time) to map its CTA's next
//     item index to (r, g, chunk, partition), so no work list is stored and
//     no planning launch is needed.
//   * One producer warp issues 3-D TMA copies of one 16-token page of one kv
//     head (box D x 1 x 16) into a 16-stage shared-memory ring, driven by the
//     block table, in the order K0 V0 K1 V1 ...; four consumer warps take the
//     (K, V) page pairs round-robin.  mbarriers: full (TMA bytes) and empty
//     (one arrive by the owning warp).  Every wait is bounded.
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
#include <type_traits>

#include "pa_internal.cuh"

namespace pa {
namespace decode {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kCtasPerSm = 3;
constexpr int kStages = 16;
// Page pairs (K, V) are dealt round-robin to the consumer warps.  With
// (kStages / 2) a multiple of the warp count, pair n always lands on stages
// 2n mod kStages and 2n+1 mod kStages owned by warp n mod 4 alone, so every
// round of a stage is consumed by the same warp in order: a warp can never run
// a whole ring round ahead on a stage (where mbarrier parity could not tell
// the rounds apart).
static_assert((kStages / 2) % kConsumerWarps == 0, "stages must split evenly among warps");
static_assert((kStages & (kStages - 1)) == 0, "ring index arithmetic uses a power-of-two ring");
constexpr int kPage = 16;         // tokens per cache block
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

// Compile-time shape of the consumer work for head_dim D and RPI rows.
template <int D, int RPI>
struct Cfg {
    // QK: LPT lanes share one key; each holds DQ dims of q for every row.
    static constexpr int LPT = (D == 128 && RPI >= 4) ? 16 : 8;
    static constexpr int TPP = 32 / LPT;           // keys per pass of a warp
    static constexpr int NPASS = kPage / TPP;      // passes per page
    static constexpr int CPL = D / 8 / LPT;        // 16-byte chunks per lane per key row
    static constexpr int DQ = CPL * 8;             // q dims per lane
    // PV: lanes over dims.
    static constexpr int DPL = D / 32;
    static constexpr int kPageBytes = kPage * D * 2;
    static constexpr int kStageBytes = kStages * kPageBytes;
    // per warp: p[key][row], alpha[row]; padded to 16 bytes so every warp's
    // buffer (and the float4 reads of it) stays aligned for any RPI
    static constexpr int kPbuf = (kPage * RPI + RPI + 3) / 4 * 4;
    static constexpr int kComb = RPI * (D + 2);       // per warp: acc[row][D], m[row], l[row]
    static constexpr int kBytes = kStageBytes + kConsumerWarps * (kPbuf + kComb) * 4 +
                                  (2 * kStages + 2) * 8 + kCandidates * 8 + 256;
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
    // A chunk of a long prompt can end before this partition starts: the item
    // is then empty (k1 == k0), never negative, so page counts stay >= 0.
    k1 = max(k0, min(min(k0 + part, it.L), max_pos + 1));
}

// Reduce v[RPI] across the LPT lanes of a key group so that each row's full
// sum ends in v[0] of the lanes whose low log2(LPT/RPI) bits are zero.  Each
// halving step trades half of the rows with the partner lane; the lane's q
// rows are stored XOR-permuted by the row it ends up holding (slot i holds
// row i ^ myrow), which makes "keep the low half, send the high half" right
// for every lane and needs no selects.  RPI rows cost RPI - 1 + log2(LPT/RPI)
// shuffles.
template <int RPI, int LPT>
__device__ __forceinline__ void reduce_scatter(float (&v)[RPI]) {
#pragma unroll
    for (int step = 0; (1 << step) < RPI; ++step) {
        const int half = RPI >> (step + 1);
        const int mask = (LPT / 2) >> step;
#pragma unroll
        for (int i = 0; i < half; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + half], mask);
    }
#pragma unroll
    for (int m = LPT / RPI / 2; m >= 1; m >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
}

// Unpack a word of two 16-bit elements into a float pair (element order kept).
template <typename T>
__device__ __forceinline__ float2 unpack_pair(uint32_t w) {
    float2 f;
    Elt<T>::unpack2(w, f.x, f.y);
    return f;
}

// Bounded barrier among the consumer warps (an mbarrier with one arrival per
// warp): a warp that timed out elsewhere cannot leave the others waiting.
__device__ __forceinline__ bool consumer_sync(uint64_t *bar, uint32_t &parity, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = mbar_wait_warp(bar, parity);
    parity ^= 1;
    return ok;
}

template <typename T, int D, int RPI>
__global__ void __launch_bounds__(kThreads, RPI == 8 ? 2 : kCtasPerSm)
paged_decode_kernel(const __grid_constant__ Params p) {
    using C = Cfg<D, RPI>;
    constexpr int LPT = C::LPT, TPP = C::TPP, NPASS = C::NPASS, CPL = C::CPL, DQ = C::DQ;
    constexpr int DPL = C::DPL;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    unsigned char *stages = base;
    float *pbuf = reinterpret_cast<float *>(base + C::kStageBytes);
    float *comb = pbuf + kConsumerWarps * C::kPbuf;
    uint64_t *full = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(comb + kConsumerWarps * C::kComb) + 7) & ~uintptr_t(7));
    uint64_t *empty = full + kStages;
    uint64_t *cbar = empty + kStages;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(cbar + 2);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid < kCandidates) cand[tid] = 0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(cbar, kConsumerWarps);
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
        // Ring order: K page 0, V page 0, K page 1, V page 1, ... of each item.
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (long long i = blockIdx.x; ok && walk.find(i, lane, it); i += gridDim.x) {
            int k0, k1;
            item_keys<RPI>(p, it, part, k0, k1);
            const int npages = (k1 - k0 + kPage - 1) / kPage;
            const int32_t *row = p.bt + (long long)it.r * p.MB + k0 / kPage;
            for (int g0 = 0; ok && g0 < npages; g0 += 32) {
                int blk = 0;
                if (g0 + lane < npages) {
                    blk = row[g0 + lane];
                    if (blk < 0 || blk >= p.NB) {
                        flag(p.status, PA_CHECK_BLOCK_ID);
                        blk = 0;
                    }
                }
                const int n = min(32, npages - g0);
                for (int pg = 0; ok && pg < n; ++pg) {
                    const int b = __shfl_sync(0xffffffffu, blk, pg);
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        if (lane == 0) {
                            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                                flag(p.status, PA_CHECK_TIMEOUT);
                                ok = false;
                            } else {
                                mbar_arrive_expect_tx(&full[stage], C::kPageBytes);
                                tma_load_3d(stages + stage * C::kPageBytes, kv ? &p.tmV : &p.tmK,
                                            &full[stage], 0, it.g, b * kPage);
                            }
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
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
    // Warp w takes the page pairs whose running index (over all items of this
    // CTA) is w mod 4, and keeps its own online-softmax state for its rows;
    // the four states are combined once per item.
    const T *q = reinterpret_cast<const T *>(p.q);
    const int j = lane % LPT;        // lane within its key group
    const int tq = lane / LPT;       // key group: keys tq, tq + TPP, ... of a page
    const int dup = j & (LPT / RPI - 1);
    int myrow = 0;                   // the row whose score this lane ends up holding
#pragma unroll
    for (int step = 0; (1 << step) < RPI; ++step)
        if (j & ((LPT / 2) >> step)) myrow += RPI >> (step + 1);
    float *pb = pbuf + warp * C::kPbuf;
    float *cw = comb + warp * C::kComb;
    int pair_base = 0;               // page pairs of earlier items
    uint32_t cpar = 0;
    bool ok = true;
    for (long long i = blockIdx.x; ok && walk.find(i, lane, it); i += gridDim.x) {
        int k0, k1;
        item_keys<RPI>(p, it, part, k0, k1);
        const int npages = (k1 - k0 + kPage - 1) / kPage;
        const int qstart = p.qsl[it.r];
        const int nrows = it.n * p.G;
        const int pos0 = it.L - it.n;  // position of the request's first query token
        int lim;                       // last key this lane's row may see
        {
            const int rr = it.chunk * RPI + myrow;
            lim = rr < nrows ? min(pos0 + rr / p.G, k1 - 1) : -1;
        }
        // Pages whose last key every row of the item sees need no mask (rows
        // past the request's end may then pick up scores, but they are never
        // written out and stay in their own accumulators).
        const int lim_all = min(pos0 + (it.chunk * RPI) / p.G, k1 - 1);

        // q rows of this item, this lane's QK dims, pre-scaled by scale*log2(e);
        // slot r holds row r ^ myrow (see reduce_scatter).
        float2 qv[RPI][DQ / 2];
#pragma unroll
        for (int r = 0; r < RPI; ++r) {
            const int rr = it.chunk * RPI + (r ^ myrow);
            if (rr < nrows) {
                const T *qrow = q + ((long long)(qstart + rr / p.G) * p.Hq + it.g * p.G + rr % p.G) * D;
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(qrow + (j + c * LPT) * 8);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 f = unpack_pair<T>(w4[e]);
                        qv[r][c * 4 + e] = make_float2(f.x * p.qscale, f.y * p.qscale);
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < DQ / 2; ++e) qv[r][e] = make_float2(0.f, 0.f);
            }
        }
        float2 acc[RPI][DPL / 2];
#pragma unroll
        for (int r = 0; r < RPI; ++r)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e) acc[r][e] = make_float2(0.f, 0.f);
        float m_run = -INFINITY, l_run = 0.f;

        for (int pg = (warp - pair_base % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
             pg < npages; pg += kConsumerWarps) {
            const int n2 = 2 * (pair_base + pg);
            const int stK = n2 & (kStages - 1), stV = (n2 + 1) & (kStages - 1);
            const uint32_t phK = (uint32_t)(n2 / kStages) & 1u, phV = (uint32_t)((n2 + 1) / kStages) & 1u;
            const int key0 = k0 + pg * kPage;
            const bool page_visible = key0 + kPage - 1 <= lim_all;

            // ---- scores of the page's 16 keys for this warp's rows
            if (!mbar_wait_warp(&full[stK], phK)) {
                flag(p.status, PA_CHECK_TIMEOUT);
                ok = false;
                break;
            }
            const unsigned char *kpage = stages + stK * C::kPageBytes;
            float sc[NPASS];
            float alpha;
            // Scores and the online-softmax update for this lane's row.  With
            // every key of the page visible to every row (the common case) no
            // mask is applied and the running max is always finite.
            auto qk_softmax = [&](auto all_visible) {
                constexpr bool kVis = decltype(all_visible)::value;
#pragma unroll
                for (int ps = 0; ps < NPASS; ++ps) {
                    const int t = ps * TPP + tq;
                    float2 kf[DQ / 2];
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(kpage + t * D * 2 + (j + c * LPT) * 16);
                        kf[c * 4 + 0] = unpack_pair<T>(raw.x);
                        kf[c * 4 + 1] = unpack_pair<T>(raw.y);
                        kf[c * 4 + 2] = unpack_pair<T>(raw.z);
                        kf[c * 4 + 3] = unpack_pair<T>(raw.w);
                    }
                    float sr[RPI];
#pragma unroll
                    for (int r = 0; r < RPI; ++r) {
                        float2 a = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < DQ / 2; ++e) a = __ffma2_rn(qv[r][e], kf[e], a);
                        sr[r] = a.x + a.y;
                    }
                    reduce_scatter<RPI, LPT>(sr);
                    sc[ps] = (kVis || key0 + t <= lim) ? sr[0] : -INFINITY;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stK]);
                float mp = sc[0];
#pragma unroll
                for (int ps = 1; ps < NPASS; ++ps) mp = fmaxf(mp, sc[ps]);
#pragma unroll
                for (int m = LPT; m < 32; m <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, m));
                const float m_new = fmaxf(m_run, mp);
                float sum = 0.f;
                if (kVis) {
                    alpha = fast_exp2(m_run - m_new);
#pragma unroll
                    for (int ps = 0; ps < NPASS; ++ps) {
                        sc[ps] = fast_exp2(sc[ps] - m_new);
                        sum += sc[ps];
                    }
                } else {
                    alpha = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
#pragma unroll
                    for (int ps = 0; ps < NPASS; ++ps) {
                        const float e = m_new == -INFINITY ? 0.f : fast_exp2(sc[ps] - m_new);
                        sc[ps] = e;
                        sum += e;
                    }
                }
#pragma unroll
                for (int m = LPT; m < 32; m <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
                l_run = l_run * alpha + sum;
                m_run = m_new;
            };
            if (page_visible) qk_softmax(std::true_type{});
            else qk_softmax(std::false_type{});
            if (dup == 0) {
#pragma unroll
                for (int ps = 0; ps < NPASS; ++ps) pb[(ps * TPP + tq) * RPI + myrow] = sc[ps];
                if (tq == 0) pb[kPage * RPI + myrow] = alpha;
            }
            __syncwarp();

            // ---- weighted values
            if (!mbar_wait_warp(&full[stV], phV)) {
                flag(p.status, PA_CHECK_TIMEOUT);
                ok = false;
                break;
            }
            const unsigned char *vpage = stages + stV * C::kPageBytes;
#pragma unroll
            for (int r = 0; r < RPI; ++r) {
                const float a = pb[kPage * RPI + r];
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[r][e] = __fmul2_rn(acc[r][e], make_float2(a, a));
            }
            const int nvalid = min(kPage, k1 - key0);  // never touch slots past the context
            auto pv_key = [&](int t) {
                float2 vf[DPL / 2];
                if constexpr (DPL == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2 *>(vpage + t * D * 2 + lane * 8);
                    vf[0] = unpack_pair<T>(raw.x);
                    vf[1] = unpack_pair<T>(raw.y);
                } else {
                    vf[0] = unpack_pair<T>(*reinterpret_cast<const uint32_t *>(vpage + t * D * 2 + lane * 4));
                }
                float pr[RPI];
                if constexpr (RPI >= 4) {
#pragma unroll
                    for (int r = 0; r < RPI; r += 4) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(pb + t * RPI + r);
                        pr[r] = v4.x;
                        pr[r + 1] = v4.y;
                        pr[r + 2] = v4.z;
                        pr[r + 3] = v4.w;
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < RPI; ++r) pr[r] = pb[t * RPI + r];
                }
#pragma unroll
                for (int r = 0; r < RPI; ++r)
#pragma unroll
                    for (int e = 0; e < DPL / 2; ++e)
                        acc[r][e] = __ffma2_rn(make_float2(pr[r], pr[r]), vf[e], acc[r][e]);
            };
            if (nvalid == kPage) {
#pragma unroll
                for (int t = 0; t < kPage; ++t) pv_key(t);
            } else {
                for (int t = 0; t < nvalid; ++t) pv_key(t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stV]);
        }
        if (!ok) break;
        pair_base += npages;

        // ---- combine the four warps' states and write the item out
#pragma unroll
        for (int r = 0; r < RPI; ++r)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e)
                *reinterpret_cast<float2 *>(cw + r * D + lane * DPL + 2 * e) = acc[r][e];
        if (dup == 0 && tq == 0) {
            cw[RPI * D + myrow] = m_run;
            cw[RPI * D + RPI + myrow] = l_run;
        }
        if (!consumer_sync(cbar, cpar, lane)) {
            flag(p.status, PA_CHECK_TIMEOUT);
            ok = false;
            break;
        }
        for (int o = tid; o < RPI * D / 2; o += kConsumers) {
            const int r = o / (D / 2);
            const int d = (o % (D / 2)) * 2;
            const int rr = it.chunk * RPI + r;
            if (rr >= nrows) continue;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb[w * C::kComb + RPI * D + r]);
            float Ls = 0.f, s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float *c = comb + w * C::kComb;
                const float mw = c[RPI * D + r];
                const float sw = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                Ls += sw * c[RPI * D + RPI + r];
                const float2 a = *reinterpret_cast<const float2 *>(c + r * D + d);
                s0 += sw * a.x;
                s1 += sw * a.y;
            }
            if (it.pslot < 0) {
                const float inv = 1.f / Ls;
                const int h = it.g * p.G + rr % p.G;
                T *dst = reinterpret_cast<T *>(p.out) +
                         ((long long)(qstart + rr / p.G) * p.Hq + h) * D + d;
                *reinterpret_cast<uint32_t *>(dst) = Elt<T>::pack2(s0 * inv, s1 * inv);
            } else {
                float *po = p.part_o + (it.pslot * RPI + r) * D + d;
                *reinterpret_cast<float2 *>(po) = make_float2(s0, s1);
                if (d == 0)
                    *reinterpret_cast<float2 *>(p.part_ml + (it.pslot * RPI + r) * 2) =
                        make_float2(M, Ls);
            }
        }
        if (!consumer_sync(cbar, cpar, lane)) {  // the combine buffer is free again
            flag(p.status, PA_CHECK_TIMEOUT);
            ok = false;
            break;
        }
    }
    // A consumer that stops early (a timed-out wait) releases every stage and
    // the item barrier once, so the others' bounded waits and the producer's
    // drain can finish.
    if (!ok && lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_arrive(&empty[s]);
        mbar_arrive(cbar);
    }
}

// Second pass: for each (token, q head) of a request whose context was split,
// combine the partitions' (m, l, o): M = max m_s, o = sum 2^(m_s-M) o_s /
// sum 2^(m_s-M) l_s.  One CTA per (token, group of 8 heads), one warp per
// head, so a long request's partitions are combined on many SMs at once.
// Lanes take 32 partitions at a time for (m, l); the weighted sum then walks
// those 32 with lanes over dims, eight independent partial-row loads in flight.
constexpr int kMergeHeadsPerCta = 8;

template <typename T, int D, int RPI>
__global__ void __launch_bounds__(32 * kMergeHeadsPerCta) merge_kernel(const __grid_constant__ Params p) {
    constexpr int DPL = D / 32;
    const int groups = (p.Hq + kMergeHeadsPerCta - 1) / kMergeHeadsPerCta;
    const int t = blockIdx.x / groups;
    const int h = (blockIdx.x % groups) * kMergeHeadsPerCta + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
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
    if (h >= p.Hq) return;
    const int r = s_r;
    const int4 meta = reinterpret_cast<const int4 *>(p.req_meta)[r];
    const int nsplit = meta.z, nchunks = meta.w;
    if (nsplit <= 1) return;
    const int tl = t - p.qsl[r];
    if (tl < 0 || tl >= p.qsl[r + 1] - p.qsl[r]) return;
    const long long pbase = (long long)(unsigned)meta.x | ((long long)meta.y << 32);
    const int g = h / p.G;
    const int rr = tl * p.G + h % p.G;
    const int chunk = rr / RPI, j = rr % RPI;
    const long long first = pbase + ((long long)g * nchunks + chunk) * nsplit;
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, ml[(first + s) * RPI + j].x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float Lsum = 0.f;
    float o[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += 32) {
        float w = 0.f;
        if (s0 + lane < nsplit) {
            const float2 v = ml[(first + s0 + lane) * RPI + j];
            w = v.x == -INFINITY ? 0.f : fast_exp2(v.x - M);
            Lsum += w * v.y;
        }
        const int cnt = min(32, nsplit - s0);
#pragma unroll 8
        for (int k = 0; k < cnt; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            const float *po = p.part_o + ((first + s0 + k) * RPI + j) * D + lane * DPL;
            if constexpr (DPL == 4) {
                const float4 v = *reinterpret_cast<const float4 *>(po);
                o[0] = fmaf(wk, v.x, o[0]);
                o[1] = fmaf(wk, v.y, o[1]);
                o[2] = fmaf(wk, v.z, o[2]);
                o[3] = fmaf(wk, v.w, o[3]);
            } else {
                const float2 v = *reinterpret_cast<const float2 *>(po);
                o[0] = fmaf(wk, v.x, o[0]);
                o[1] = fmaf(wk, v.y, o[1]);
            }
        }
    }
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, s);
    const float inv = 1.f / Lsum;
    T *dst = reinterpret_cast<T *>(p.out) + ((long long)t * p.Hq + h) * D + lane * DPL;
#pragma unroll
    for (int d = 0; d < DPL; d += 2)
        *reinterpret_cast<uint32_t *>(dst + d) = Elt<T>::pack2(o[d] * inv, o[d + 1] * inv);
}

template <typename T, int D, int RPI>
pa_status launch_typed(Params &prm, long long max_items, bool merge, cudaStream_t stream) {
    using S = Cfg<D, RPI>;
    static int resident[64] = {};  // CTAs per SM, per device
    int dev = 0;
    PA_TRY_CUDA(cudaGetDevice(&dev));
    int per_sm = dev < 64 ? resident[dev] : 0;
    if (per_sm == 0) {
        PA_TRY_CUDA(cudaFuncSetAttribute(paged_decode_kernel<T, D, RPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes));
        PA_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, paged_decode_kernel<T, D, RPI>, kThreads, S::kBytes));
        if (per_sm < 1) return PA_ERR_UNSUPPORTED;
        if (dev < 64) resident[dev] = per_sm;
    }
    // Persistent grid: every resident slot once, no more CTAs than items.
    long long grid = (long long)per_sm * num_sms();
    if (max_items < grid) grid = max_items;
    if (grid < 1) grid = 1;
    paged_decode_kernel<T, D, RPI><<<(int)grid, kThreads, S::kBytes, stream>>>(prm);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    if (merge && prm.T > 0) {
        const long long groups = (prm.Hq + kMergeHeadsPerCta - 1) / kMergeHeadsPerCta;
        merge_kernel<T, D, RPI><<<(unsigned)(prm.T * groups), 32 * kMergeHeadsPerCta, 0, stream>>>(prm);
        PA_TRY_CUDA(cudaGetLastError());
        note_launch();
    }
    return PA_OK;
}

template <typename T, int D>
pa_status dispatch_rpi(int rpi, Params &prm, long long grid, bool merge, cudaStream_t stream) {
    switch (rpi) {
        case 1: return launch_typed<T, D, 1>(prm, grid, merge, stream);
        case 2: return launch_typed<T, D, 2>(prm, grid, merge, stream);
        case 4: return launch_typed<T, D, 4>(prm, grid, merge, stream);
        default: return launch_typed<T, D, 8>(prm, grid, merge, stream);
    }
}

// Rows per item: all heads of a kv group (at most 8, the register budget).
// With 4+ heads per group a single-token decode already fills the item, so
// short multi-token requests are split into more items rather than making
// every decode item carry empty rows; with fewer heads per group a few query
// tokens share an item.
inline int rows_per_item(int G, int max_q) {
    long long rows = (long long)G * (max_q > 0 ? max_q : 1);
    if (G >= 4) rows = G;
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

pa_status launch_decode(const AttnArgs &a, int tau, cudaStream_t stream) {
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
    prm.tau = tau;
    prm.qscale = a.scale * 1.4426950408889634f;
    prm.status = status_word();
    if (!prm.status) return PA_ERR_CUDA;
    const int rpi = rows_per_item(prm.G, a.max_q < tau ? a.max_q : tau);

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

    // Upper bound on the work items (the grid never exceeds it).
    const long long splits = prm.p_min >= kSingle ? 1 : (a.max_seq + prm.p_min - 1) / prm.p_min;
    const long long chunks = (long long)a.R + ((long long)a.T * prm.G + rpi - 1) / rpi;
    const long long grid = (long long)a.Hkv * chunks * splits;

    const bool bf16 = a.dtype == PA_BF16;
    if (a.D == 128)
        return bf16 ? dispatch_rpi<__nv_bfloat16, 128>(rpi, prm, grid, merge, stream)
                    : dispatch_rpi<__half, 128>(rpi, prm, grid, merge, stream);
    return bf16 ? dispatch_rpi<__nv_bfloat16, 64>(rpi, prm, grid, merge, stream)
                : dispatch_rpi<__half, 64>(rpi, prm, grid, merge, stream);
}

}  // namespace pa
