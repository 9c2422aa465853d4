// Paged attention, split-K over KV partitions.
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
//   * Persistent CTAs, 3 per SM (128 registers; at 8 rows and head_dim 128
//     the warps' states are combined in two passes of 64 dims, so the
//     combine buffer fits).  The producer warp takes its CTA's own index first, then
//     each next item index from a counter in the workspace as its CTA frees
//     up (a fixed stride when there is no workspace), and passes it to the
//     consumer warps through a small shared-memory queue.  Every warp walks the request list itself (a
//     warp-wide scan over 32 requests at a time) to map an item index to
//     (r, g, chunk, partition), so no work list is stored and no planning
//     launch is needed.
//   * One producer warp issues swizzled 3-D TMA copies of 16-token pages of
//     one kv head into a 16-stage shared-memory ring, driven by the block
//     table: K unit, V unit, ... where a unit is the consecutive pages that
//     fill 4 KiB (one 16-bit page at head_dim 128, up to four FP8 pages at
//     head_dim 64).  Unit j of an item goes to consumer warp j mod 4.
//     mbarriers: full (TMA bytes) and empty (the consumers' release); every
//     wait is bounded.
//   * Consumers run on the tensor cores with mma.sync (m16n8k16, f32
//     accumulate): S^T = K Q^T and O^T += V^T P^T per page, the item's rows
//     as the MMA's N, an online softmax per warp, the four warps' states
//     combined once per item.  FP8 E4M3 pages widen to f16 in registers.
//   * A request whose context fits one partition writes its output directly;
//     otherwise (m, l, unnormalised o) go to the workspace and the merge
//     kernel combines them.
//   * With kGroups (callers whose block tables share blocks), single-token
//     requests holding the same blocks over a whole partition form group
//     items: the pages are read once and each consumer warp computes 8 of up
//     to 32 rows over every page.
#include <climits>
#include <cstring>
#include <type_traits>

#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {
namespace decode {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kCtasPerSm = 3;
constexpr int kPage = 16;         // tokens per cache block
constexpr int kCandidates = 8;    // partition lengths p_min << k
constexpr int kSingle = INT_MAX / 2;
constexpr int kQueue = 8;         // item queue entries (producer -> consumer warps)
constexpr int kGroupRows = 32;    // rows of a shared-partition group item (8 per consumer warp)
constexpr int kGroupShift = 48;   // queue entry = item index | members << kGroupShift

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
    unsigned int *item_counter;  // zeroed before launch: CTAs take the next item as they
                                 // free up (NULL: fixed stride over the items)
    int R, T, MB, NB, Hq, Hkv, G;
    int tau;              // requests with more query tokens are not handled here
    int max_seq;          // the caller's bound on seq_lens (longer requests are flagged)
    int p_min;            // preferred partition length in keys (multiple of 256)
    int part_fixed;       // the workspace holds every partial at p_min: no choice to make
    float qscale;         // softmax scale * log2(e)
    const float *k_scale; // FP8 pools: cached value = element * scale (device scalars)
    const float *v_scale;
    unsigned int *status;
    int launch_pdl;       // host side: the split-K grid as a programmatic dependent of the grid before
    int launch_part;      // host side: 0 split-K grid and merge pass, 1 the grid only, 2 the merge only
};

// Marker for an FP8 E4M3 cache element.
struct Fp8E4M3 {};

// Shared-memory layout of one cache page (16 slots of one kv head) as the
// TMA writes it: rows of min(128, D * elt) bytes with the matching TMA
// swizzle (128 B, or 64 B for 64-byte rows); a 256-byte row is split into two
// 16-row boxes, one per 128-byte half, stored back to back.
template <typename TC, int D>
struct Lay {
    static constexpr int E = std::is_same<TC, Fp8E4M3>::value ? 1 : 2;  // bytes per element
    static constexpr int RB = D * E;                  // bytes per slot row
    static constexpr int SR = RB >= 128 ? 128 : RB;   // bytes per smem row
    static constexpr int NSUB = RB / SR;              // TMA boxes per page
    static constexpr int kSubBytes = kPage * SR;
    static constexpr int kPageBytes = kPage * RB;
    static constexpr int CPR = SR / 16;               // 16-byte chunks per smem row
    static constexpr int NCH = RB / 64;               // chunks of a key row per lane (4 lanes per key)
    static constexpr int KPC = 4 / E;                 // MMA k-steps per chunk (4 dims per lane per step)
    static constexpr int KS = D / 16;                 // k-steps of QK = m-tiles of PV
    static constexpr int kSwzMask = SR == 128 ? 7 : 3;
    static_assert(RB % 64 == 0 && (SR == 128 || SR == 64), "head_dim 64 or 128");
    // byte offset of 16-byte chunk c of page row `key`
    __device__ __forceinline__ static int chunk_off(int key, int c) {
        const int off = (c / CPR) * kSubBytes + key * SR + (c % CPR) * 16;
        return off ^ (((off >> 7) & kSwzMask) << 4);
    }
};

// The MMA's input type: the cache's own type for 16-bit caches (the same as
// q's); f16 for an FP8 cache (E4M3 widens to f16 exactly).
template <typename TQ, typename TC> struct MmaIn { using type = TC; };
template <typename TQ> struct MmaIn<TQ, Fp8E4M3> { using type = __half; };

template <typename TC, int D, int RPI>
struct Cfg {
    using L = Lay<TC, D>;
    // Pages per ring stage: consecutive pages of a request share a stage and
    // one handoff up to 4 KiB (one 16-bit page at head_dim 128; two at
    // head_dim 64 or FP8; four FP8 pages at head_dim 64), so every layout
    // keeps the same bytes in flight.  With 2 KiB stages head_dim 64 streamed
    // at 4.6 TB/s, with 4 KiB at 5.5-6.0.
    static constexpr int kSP = L::kPageBytes >= 4096 ? 1 : 4096 / L::kPageBytes;
    static constexpr int kUnitBytes = kSP * L::kPageBytes;
    // 64 KB of pages in flight per CTA at head_dim 128
    static constexpr int kStages = 16;
    // Unit pairs (K, V) of an item are dealt to the consumer warps by their
    // index in the item: unit j goes to warp j mod 4, so an item's arithmetic
    // never depends on what the CTA ran before it.  Each warp owns
    // kPairsPerWarp pairs of stages and fills them in turn (pair_stage), so
    // every round of a stage is consumed by the same warp in order: a warp can
    // never run a whole round ahead on a stage (where mbarrier parity could
    // not tell the rounds apart).
    static constexpr int kPairsPerWarp = kStages / 2 / kConsumerWarps;
    static_assert(kPairsPerWarp * 2 * kConsumerWarps == kStages, "stages must split evenly among warps");
    static_assert((kPairsPerWarp & (kPairsPerWarp - 1)) == 0, "per-warp counters wrap at a power of two");
    static constexpr int kStageBytes = kStages * kUnitBytes;
    // The four warps' states are combined through shared memory in kCombPasses
    // passes of kDC dims each: at 8 rows and head_dim 128 two passes keep the
    // buffer at the 4-row size, so three CTAs still fit an SM.
    static constexpr int kCombPasses = (RPI == 8 && D == 128) ? 2 : 1;
    static constexpr int kDC = D / kCombPasses;
    static constexpr int kComb = RPI * (kDC + 2);     // per warp: acc[row][kDC], m[row], l[row]
    static constexpr int kBytes = kStageBytes + kConsumerWarps * kComb * 4 +
                                  (2 * kStages + 2) * 8 + kCandidates * 8 + kQueue * 3 * 8 +
                                  1024;
};

// First stage of warp w's c-th (K, V) unit pair (the V unit takes the next
// stage); that round's mbarrier parity is (c / kPW) & 1.
template <int kPW>
__device__ __forceinline__ int pair_stage(int w, uint32_t c) {
    return 2 * (w + kConsumerWarps * (int)(c % kPW));
}

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
            const bool sane = a >= 0 && b <= p->T && n >= 0 && L >= n && L <= p->max_seq &&
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

// Bounded barrier among the consumer warps (an mbarrier with one arrival per
// warp): a warp that timed out elsewhere cannot leave the others waiting.
__device__ __forceinline__ bool consumer_sync(uint64_t *bar, uint32_t &parity, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    const bool ok = mbar_wait_warp(bar, parity);
    parity ^= 1;
    return ok;
}

// ---- warp-level tensor-core helpers (mma.sync m16n8k16, f32 accumulate) ----

template <typename TM> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    // P enters the PV product as two bf16 terms, hi = bf16(p) and
    // lo = bf16(p - hi): 16 significant bits instead of 8, so the weights
    // add about 2^-17 of |v| to the error instead of 2^-9 (a near one-hot row
    // with |v| near 4 would otherwise be off by 0.008 before the output's own
    // rounding).
    static constexpr bool kSplitP = true;
    __device__ __forceinline__ static uint32_t residual(float lo, float hi, uint32_t packed) {
        return pack(lo - __uint_as_float(packed << 16), hi - __uint_as_float(packed & 0xffff0000u));
    }
};
template <> struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    // f16 P carries 11 significant bits (P <= 256 stays far from f16's
    // limits): one term is enough.
    static constexpr bool kSplitP = false;
    __device__ __forceinline__ static uint32_t residual(float, float, uint32_t) { return 0u; }
};

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}

// Transpose an 8x8 matrix of 16-bit elements held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Four E4M3 codes (bytes 0..3 of w) to two f16 pairs, exactly: bytes (0, 1)
// -> lo (byte 0 in the low half), bytes (2, 3) -> hi.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n"
        ".reg .b16 l, h;\n"
        "mov.b32 {l, h}, %2;\n"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n"
        "}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// 16-bit Q elements to the MMA's input type (the f16 path of an FP8 cache
// takes bf16 q through float: exact inside f16's range).
template <typename TQ, typename TM> struct QConv {
    __device__ __forceinline__ static uint32_t run(uint32_t w) { return w; }
};
template <> struct QConv<__nv_bfloat16, __half> {
    __device__ __forceinline__ static uint32_t run(uint32_t w) {
        const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

// Logical key k (the MMA's index, 0..15) of a page lives in page row
// perm16(k): rows 0,5,3,6,4,1,7,2 then the same + 8.  With this order every
// shared-memory load of the consumer below is free of bank conflicts under
// the TMA swizzle, for each element size and head_dim.
__device__ __forceinline__ int perm16(int k) { return ((0x27146350u >> (4 * (k & 7))) & 0xf) | (k & 8); }

// kGroups: shared-partition group items (callers whose block tables may
// share physical blocks); the kernel without them has no code for them.
template <typename TQ, typename TC, int D, int RPI, bool kGroups>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
paged_decode_kernel(const __grid_constant__ Params p) {
    using L = Lay<TC, D>;
    using TM = typename MmaIn<TQ, TC>::type;
    using C = Cfg<TC, D, RPI>;
    constexpr int kSt = C::kStages;
    constexpr int KS = L::KS, NCH = L::NCH, KPC = L::KPC;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *stages = base;
    float *comb = reinterpret_cast<float *>(base + C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(comb + kConsumerWarps * C::kComb) + 7) & ~uintptr_t(7));
    uint64_t *empty = full + kSt;
    uint64_t *cbar = empty + kSt;
    unsigned long long *cand = reinterpret_cast<unsigned long long *>(cbar + 2);
    uint64_t *qfull = reinterpret_cast<uint64_t *>(cand + kCandidates);
    uint64_t *qempty = qfull + kQueue;
    long long *qitem = reinterpret_cast<long long *>(qempty + kQueue);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // arrivals that release a stage: group items need all four warps
    constexpr uint32_t kRelease = kGroups ? kConsumerWarps : 1;

    if (tid < kCandidates) cand[tid] = 0;
    if (tid == 0) {
        for (int s = 0; s < kSt; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kRelease);   // every warp of a group item, or the owner for all
        }
        mbar_init(cbar, kConsumerWarps);
        for (int e = 0; e < kQueue; ++e) {
            mbar_init(&qfull[e], 1);
            mbar_init(&qempty[e], kConsumerWarps);
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
        if (p.p_min < kSingle && !p.part_fixed) {
            for (int r = tid; r < p.R; r += kThreads) {
                const int a = p.qsl[r], b = p.qsl[r + 1];
                const int n = b - a;
                const int L = p.seq_lens[r];
                if (a < 0 || b > p.T || n < 1 || n > p.tau || L < n || L > p.max_seq ||
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
    if (p.part_fixed) {
        part = p.p_min;
    } else if (p.p_min < kSingle) {
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
    // With an item counter the producer takes its CTA's own index first, then
    // grid + each next value of the counter, and publishes the index in queue
    // entry k % kQueue (-1: no more items) for the consumer warps; without
    // one, CTA b takes items b, b + grid, ...  Either way a CTA's indices
    // rise, as the walker needs.

    // ---- shared-partition groups.  Requests of one query token whose block
    // tables hold the same physical blocks over a whole partition that their
    // query sees completely (a prefix shared after a fork or by prefix
    // caching) read the same K/V there.  Runs of such requests, cut at
    // multiples of kGroupRows / G in batch order, form one group item: the
    // first request's item reads the pages once for every member's rows and
    // the others' items for that partition are skipped.  Only with an item
    // queue (the producer publishes the member count) and a partial slot for
    // every partition.
    const int gcap = (kGroups && p.item_counter && p.part_o && p.G <= 8 && kGroupRows % p.G == 0)
                         ? kGroupRows / p.G : 0;   // members per group (0: no groups)
    // partition s of the window's request at lane rl, fully visible to its
    // single query token and part of a single row chunk
    auto groupable = [&](int rl, int s) {
        const int n = __shfl_sync(0xffffffffu, walk.n, rl);
        const int L = __shfl_sync(0xffffffffu, walk.L, rl);
        const int nc = __shfl_sync(0xffffffffu, walk.nchunks, rl);
        return n == 1 && nc == 1 && (long long)(s + 1) * part <= L - 1;
    };
    // the same blocks for partition s in requests ra and rb (warp-wide)
    auto same_blocks = [&](int ra, int rb, int s) {
        const int P = part / kPage;
        const int32_t *a = p.bt + (long long)ra * p.MB + (long long)s * P;
        const int32_t *b = p.bt + (long long)rb * p.MB + (long long)s * P;
        bool same = true;
        for (int c0 = 0; same && c0 < P; c0 += 32)
            same = __ballot_sync(0xffffffffu, c0 + lane < P && a[c0 + lane] != b[c0 + lane]) == 0;
        return same;
    };

    if (warp == kConsumerWarps) {
        // =================== producer warp ===================
        // Issue order: K unit 0, V unit 0, K unit 1, V unit 1, ... of each
        // item, a unit being C::kSP consecutive pages of the request, unit j
        // into the next stage pair of warp j mod 4.  A page is L::NSUB swizzled
        // boxes of 16 rows (one per 128 bytes of a row), landing back to back.
        constexpr int kSP = C::kSP;
        constexpr int kPW = C::kPairsPerWarp;
        // pairs handed to each consumer warp so far, mod 256: one byte per warp
        uint32_t handed = 0;
        auto handed_to = [&](int w) { return (handed >> (8 * w)) & 0xffu; };
        int blk0 = 0;            // the item's first 32 block ids, when already loaded
        bool have_blk0 = false;
        bool first_fetch = true; // a CTA's first item is its own index: no atomic storm at launch
        bool ok = true;
        for (long long k = 0; ok; ++k) {   // k: items published
            if (p.item_counter) {
                unsigned int cand = 0;
                bool valid;
                long long members = 0;
                for (;;) {   // the next item that is not a group member's
                    if (first_fetch) {
                        cand = blockIdx.x;
                        first_fetch = false;
                    } else {
                        if (lane == 0) cand = gridDim.x + atomicAdd(p.item_counter, 1u);
                        cand = __shfl_sync(0xffffffffu, cand, 0);
                    }
                    valid = walk.find((long long)cand, lane, it);
                    have_blk0 = false;
                    if (!valid || gcap == 0) break;
                    const int rl = it.r - walk.rb;
                    if (!groupable(rl, it.split)) break;
                    // The item's first 32 block ids (its copies need them) and, in
                    // the same round trip, the partition's first block id in the
                    // neighbouring requests: only a match there calls for a full
                    // comparison.
                    const long long pg = (long long)it.split * (part / kPage);
                    const bool prev_ok = it.r % gcap != 0 && groupable(rl - 1, it.split);
                    const bool next_ok = (it.r + 1) % gcap != 0 && it.r + 1 < p.R &&
                                         groupable(rl + 1, it.split);
                    blk0 = p.bt[(long long)it.r * p.MB + pg + lane];   // a full partition: >= 32 pages
                    int nb = -1;
                    if (lane == 0 && prev_ok) nb = p.bt[(long long)(it.r - 1) * p.MB + pg];
                    if (lane == 1 && next_ok) nb = p.bt[(long long)(it.r + 1) * p.MB + pg];
                    have_blk0 = true;
                    const int first = __shfl_sync(0xffffffffu, blk0, 0);
                    const int prev = __shfl_sync(0xffffffffu, nb, 0), next = __shfl_sync(0xffffffffu, nb, 1);
                    if (prev_ok && prev == first && same_blocks(it.r, it.r - 1, it.split))
                        continue;   // a member: its group's first request covers it
                    int m = 1;
                    if (next_ok && next == first)
                        while (m < gcap && (it.r + m) % gcap != 0 && it.r + m < p.R &&
                               groupable(rl + m, it.split) && same_blocks(it.r + m, it.r, it.split))
                            ++m;
                    if (m > 1) members = m;
                    break;
                }
                const int e = (int)(k % kQueue);
                if (lane == 0) {
                    if (!mbar_wait(&qempty[e], (uint32_t)(((k / kQueue) & 1) ^ 1))) {
                        flag(p.status, PA_CHECK_TIMEOUT);
                        ok = false;
                    } else {
                        qitem[e] = valid ? ((long long)cand | (members << kGroupShift)) : -1;
                        mbar_arrive(&qfull[e]);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || !valid) break;
            } else if (!walk.find(blockIdx.x + k * gridDim.x, lane, it)) {
                break;
            }
            int k0, k1;
            item_keys<RPI>(p, it, part, k0, k1);
            const int npages = (k1 - k0 + kPage - 1) / kPage;
            const int32_t *row = p.bt + (long long)it.r * p.MB + k0 / kPage;
            for (int g0 = 0; ok && g0 < npages; g0 += 32) {
                int blk = 0;
                if (g0 + lane < npages) {
                    blk = (g0 == 0 && have_blk0) ? blk0 : row[g0 + lane];
                    if (blk < 0 || blk >= p.NB) {
                        flag(p.status, PA_CHECK_BLOCK_ID);
                        blk = 0;
                    }
                }
                const int n = min(32, npages - g0);
                for (int pu = 0; ok && pu < n; pu += kSP) {
                    const int cnt = min(kSP, n - pu);   // pages in this unit
                    int b[kSP];
#pragma unroll
                    for (int sp = 0; sp < kSP; ++sp) b[sp] = __shfl_sync(0xffffffffu, blk, min(pu + sp, 31));
                    const int w = ((g0 + pu) / kSP) % kConsumerWarps;
                    const uint32_t c = handed_to(w);
                    const uint32_t phase = (c / kPW) & 1u;
                    handed = (handed & ~(0xffu << (8 * w))) | (((c + 1) & 0xffu) << (8 * w));
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        const int stage = pair_stage<kPW>(w, c) + kv;
                        if (lane == 0) {
                            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                                flag(p.status, PA_CHECK_TIMEOUT);
                                ok = false;
                            } else {
                                mbar_arrive_expect_tx(&full[stage], cnt * L::kPageBytes);
#pragma unroll
                                for (int sp = 0; sp < kSP; ++sp) {
                                    if (sp >= cnt) break;
#pragma unroll
                                    for (int sub = 0; sub < L::NSUB; ++sub)
                                        tma_load_3d(stages + stage * C::kUnitBytes + sp * L::kPageBytes +
                                                        sub * L::kSubBytes,
                                                    kv ? &p.tmV : &p.tmK, &full[stage],
                                                    sub * (L::SR / L::E), it.g, b[sp] * kPage);
                                }
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
            }
        }
        // No items left for this CTA: the merge pass may be scheduled (it
        // still waits for this grid to finish before reading).
        if (lane == 0) grid_launch_dependents();
        // Drain: wait (bounded) until the consumers have released every stage
        // (each warp's next kPW pairs find their stages free), so no copy is
        // still landing when the CTA exits.
        if (lane == 0) {
            bool drained = true;
            for (int w = 0; drained && w < kConsumerWarps; ++w)
                for (int j = 0; drained && j < kPW; ++j) {
                    const uint32_t c = handed_to(w) + j;
                    for (int kv = 0; drained && kv < 2; ++kv)
                        if (!mbar_wait(&empty[pair_stage<kPW>(w, c) + kv], ((c / kPW) & 1u) ^ 1)) {
                            flag(p.status, PA_CHECK_TIMEOUT);
                            drained = false;
                        }
                }
        }
        return;
    }

    // =================== consumer warps ===================
    // Warp w takes the unit pairs w, w + 4, ... of each item and keeps its
    // own online-softmax state; the four states are combined once per item
    // (in warp order, so an item's result is the same whichever CTA runs it).  Per page pair, on the tensor cores:
    //   S^T (16 keys x 8 rows) = K (16 x D) . Q^T      (D/16 MMAs, k = dims)
    //   O^T (D x 8 rows)      += V^T (D x 16) . P^T    (D/16 MMAs, k = keys)
    // Lane (gq = lane/4, tq = lane%4) holds S^T for keys perm16(gq), perm16(gq+8)
    // and rows 2tq, 2tq+1; the rows of an item (its (token, head) pairs, at most
    // 8) are the MMAs' N.  P^T is moved from the S^T layout to the B-operand
    // layout by two 8x8 transposes (movmatrix).
    const TQ *q = reinterpret_cast<const TQ *>(p.q);
    const int gq = lane >> 2, tq = lane & 3;
    const float qs = p.qscale * (p.k_scale ? *p.k_scale : 1.f);
    const float vs = p.v_scale ? *p.v_scale : 1.f;
    const int key_a = perm16(gq), key_b = perm16(gq + 8);   // page rows of this lane's keys
    // Byte offsets inside a page, fixed per lane.  K: the lane's chunks of
    // keys key_a / key_b.  V (16-bit): the row this lane gives ldmatrix for
    // m-tile mt (logical key (lane & 7) + 8 * (matrix >> 1), dims 16 mt +
    // 8 * (matrix & 1)).  V (FP8): the lane's D/8 bytes (dims gq * D/8 ..) of
    // keys 2tq, 2tq + 1, 2tq + 8, 2tq + 9.
    // Offsets of later chunks follow from the first by flipping swizzle bits
    // (chunk c + 4 of a 128-byte row: bit 6) and adding whole 16-row boxes,
    // so each needs one register.  (A 64-byte row has one chunk per lane.)
    static_assert(L::SR == 128 || NCH == 1, "one chunk per lane on 64-byte rows");
    const int koff_a = L::chunk_off(key_a, tq), koff_b = L::chunk_off(key_b, tq);
    auto koff = [&](int base, int jj) { return (base ^ (64 * (jj & 1))) + (jj >> 1) * L::kSubBytes; };
    // page rows of keys 2tq, 2tq + 1, 2tq + 8, 2tq + 9 (recomputed where
    // needed, which is only on partial pages: no registers held for them)
    auto vkey = [&](int e) { return perm16(2 * tq + (e & 1) + 8 * (e >> 1)); };
    int voff[L::E == 2 ? 1 : 4];
    if constexpr (L::E == 2) {
        const int mi = lane >> 3;
        voff[0] = L::chunk_off(perm16((lane & 7) + 8 * (mi >> 1)), mi & 1);
    } else {
        const int byte = gq * (D / 8);
#pragma unroll
        for (int e = 0; e < 4; ++e) voff[e] = L::chunk_off(vkey(e), byte / 16) + byte % 16;
    }
    float *cw = comb + warp * C::kComb;
    // Unit pairs handed to each warp's stages so far, mod 256: one byte per
    // warp, kept exactly as the producer keeps it (with group items, whose
    // units every warp reads); without them a warp counts only its own.
    uint32_t handed = 0, taken = 0;
    uint32_t cpar = 0;
    bool ok = true;
    for (long long k = 0; ok; ++k) {
        long long i = blockIdx.x + k * gridDim.x;
        int members = 0;             // > 1: a shared-partition group item
        if (p.item_counter) {
            const int e = (int)(k % kQueue);
            if (!mbar_wait_warp(&qfull[e], (uint32_t)((k / kQueue) & 1))) {
                flag(p.status, PA_CHECK_TIMEOUT);
                ok = false;
                break;
            }
            const long long v = qitem[e];
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[e]);
            if (v < 0) break;
            i = v & ((1LL << kGroupShift) - 1);
            if constexpr (kGroups) members = (int)(v >> kGroupShift);
        }
        if (!walk.find(i, lane, it)) break;
        const bool grp = kGroups && members > 1;
        int k0, k1;
        item_keys<RPI>(p, it, part, k0, k1);
        const int npages = (k1 - k0 + kPage - 1) / kPage;
        const int qstart = p.qsl[it.r];
        const int nrows = it.n * p.G;
        const int pos0 = it.L - it.n;  // position of the request's first query token
        // last key each of this lane's two rows (2tq, 2tq + 1) may see; -1 for
        // rows past the item.  A group item's rows are 8 per warp (row 8 warp +
        // x is member (8 warp + x) / G's head (8 warp + x) % G) and see the
        // whole partition.
        int lim0 = -1, lim1 = -1;
        if (grp) {
            if (8 * warp + 2 * tq < members * p.G) lim0 = k1 - 1;
            if (8 * warp + 2 * tq + 1 < members * p.G) lim1 = k1 - 1;
        } else {
            const int r0 = it.chunk * RPI + 2 * tq, r1 = r0 + 1;
            if (2 * tq < RPI && r0 < nrows) lim0 = min(pos0 + r0 / p.G, k1 - 1);
            if (2 * tq + 1 < RPI && r1 < nrows) lim1 = min(pos0 + r1 / p.G, k1 - 1);
        }
        // Pages whose last key every row of the item sees need no mask (rows
        // past the item then pick up scores, but they are never written out).
        const int lim_all = grp ? k1 - 1 : min(pos0 + (it.chunk * RPI) / p.G, k1 - 1);

        // Q^T fragments (B operand): row gq of the item (of the warp's rows
        // for a group), this lane's dims.
        uint32_t qf[KS][2];
        {
            bool have;
            long long tok;
            int head;
            if (grp) {
                const int gr = 8 * warp + gq;
                have = gr < members * p.G;
                tok = qstart + (have ? gr / p.G : 0);   // members hold one token each, in order
                head = have ? gr % p.G : 0;
            } else {
                const int rr = it.chunk * RPI + gq;
                have = gq < RPI && rr < nrows;
                tok = qstart + (have ? rr / p.G : 0);
                head = have ? rr % p.G : 0;
            }
            const TQ *qrow = q + (tok * p.Hq + it.g * p.G + head) * D;
#pragma unroll
            for (int jj = 0; jj < NCH; ++jj) {
                const int d0 = (tq + 4 * jj) * (16 / L::E);   // first dim of the lane's chunk
#pragma unroll
                for (int h = 0; h < 16 / L::E / 8; ++h) {   // 8 dims (16 bytes of q) at a time
                    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
                    if (have) raw = *reinterpret_cast<const uint4 *>(qrow + d0 + 8 * h);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
                    // 4 dims per k-step: pairs (0,1) -> b0b1, (2,3) -> b2b3
                    qf[jj * KPC + 2 * h][0] = QConv<TQ, TM>::run(w4[0]);
                    qf[jj * KPC + 2 * h][1] = QConv<TQ, TM>::run(w4[1]);
                    qf[jj * KPC + 2 * h + 1][0] = QConv<TQ, TM>::run(w4[2]);
                    qf[jj * KPC + 2 * h + 1][1] = QConv<TQ, TM>::run(w4[3]);
                }
            }
        }
        float o[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY;   // reference max of rows 2tq, 2tq+1
        float l0 = 0.f, l1 = 0.f;               // this lane's share of the row sums

        constexpr int kSP = C::kSP;
        const int nunits = (npages + kSP - 1) / kSP;
        // One unit pair (K, V): QK of its pages and the release of K's stage,
        // one softmax update, PV and the release of V's stage (count: every
        // warp of a group item arrives; an ordinary item's owner arrives for
        // all).
        auto run_unit = [&](int pu, uint32_t stK, uint32_t phK, uint32_t release) -> bool {
            const uint32_t stV = stK + 1, phV = phK;
            if (!mbar_wait_warp(&full[stK], phK) || !mbar_wait_warp(&full[stV], phV)) {
                flag(p.status, PA_CHECK_TIMEOUT);
                return false;
            }
            // The unit's pages: QK of each (independent MMA chains), one
            // softmax update over all their keys, then PV of each.
            bool have[kSP];
            int keyb[kSP];                 // first key of each page
            float sv[kSP][4];              // (key_a, row 2tq), (key_a, 2tq+1), (key_b, 2tq), (key_b, 2tq+1)
#pragma unroll
            for (int sp = 0; sp < kSP; ++sp) {
                have[sp] = pu * kSP + sp < npages;
                keyb[sp] = k0 + (pu * kSP + sp) * kPage;
            }
            // ---- S^T = K Q^T for each page's 16 keys
#pragma unroll
            for (int sp = 0; sp < kSP; ++sp) {
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                if (have[sp]) {
                    const unsigned char *kpage = stages + stK * C::kUnitBytes + sp * L::kPageBytes;
#pragma unroll
                    for (int jj = 0; jj < NCH; ++jj) {
                        const uint4 ka = *reinterpret_cast<const uint4 *>(kpage + koff(koff_a, jj));
                        const uint4 kb = *reinterpret_cast<const uint4 *>(kpage + koff(koff_b, jj));
                        const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                        for (int sub = 0; sub < KPC; ++sub) {
                            const int s = jj * KPC + sub;
                            uint32_t a0, a1, a2, a3;
                            if constexpr (L::E == 2) {
                                a0 = wa[2 * sub];
                                a1 = wb[2 * sub];
                                a2 = wa[2 * sub + 1];
                                a3 = wb[2 * sub + 1];
                            } else {
                                e4m3x4_to_f16x4(wa[sub], a0, a2);
                                e4m3x4_to_f16x4(wb[sub], a1, a3);
                            }
                            if (s & 1) Mma<TM>::run(sb, a0, a1, a2, a3, qf[s][0], qf[s][1]);
                            else Mma<TM>::run(sa, a0, a1, a2, a3, qf[s][0], qf[s][1]);
                        }
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) sv[sp][e] = have[sp] ? (sa[e] + sb[e]) * qs : -INFINITY;
            }
            const bool unit_visible = keyb[kSP - 1] + kPage - 1 <= lim_all && have[kSP - 1];
            // K is in registers now: its stage goes back to the producer half a
            // unit before V's.
            __syncwarp();
            if (lane == 0) mbar_arrive_n(&empty[stK], release);

            // ---- online softmax with a lazily moved reference max: P stays
            //      below 2^8 (inside the 16-bit types' range; bf16 P enters
            //      the PV product as a hi + lo pair), the sums stay in f32,
            //      and O is rescaled only when a row's max grows by more than 8
            //      (in log2 units).
            if (!unit_visible) {
#pragma unroll
                for (int sp = 0; sp < kSP; ++sp) {
                    const int pa = keyb[sp] + perm16(gq), pb = keyb[sp] + perm16(gq + 8);
                    sv[sp][0] = pa <= lim0 ? sv[sp][0] : -INFINITY;
                    sv[sp][1] = pa <= lim1 ? sv[sp][1] : -INFINITY;
                    sv[sp][2] = pb <= lim0 ? sv[sp][2] : -INFINITY;
                    sv[sp][3] = pb <= lim1 ? sv[sp][3] : -INFINITY;
                }
            }
            float mx0 = fmaxf(sv[0][0], sv[0][2]), mx1 = fmaxf(sv[0][1], sv[0][3]);
#pragma unroll
            for (int sp = 1; sp < kSP; ++sp) {
                mx0 = fmaxf(mx0, fmaxf(sv[sp][0], sv[sp][2]));
                mx1 = fmaxf(mx1, fmaxf(sv[sp][1], sv[sp][3]));
            }
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
            }
            const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;
            if (up0 || up1) {
                const float al0 = up0 ? fast_exp2(m0 - mx0) : 1.f;
                const float al1 = up1 ? fast_exp2(m1 - mx1) : 1.f;
                if (up0) m0 = mx0;
                if (up1) m1 = mx1;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    o[mt][0] *= al0;
                    o[mt][1] *= al1;
                    o[mt][2] *= al0;
                    o[mt][3] *= al1;
                }
                l0 *= al0;
                l1 *= al1;
            }
            constexpr bool kSplit = Mma<TM>::kSplitP;
            uint32_t pb[kSP][2], pl[kSP][2];
#pragma unroll
            for (int sp = 0; sp < kSP; ++sp) {
                float pv[4];
                if (unit_visible) {
                    pv[0] = fast_exp2(sv[sp][0] - m0);
                    pv[1] = fast_exp2(sv[sp][1] - m1);
                    pv[2] = fast_exp2(sv[sp][2] - m0);
                    pv[3] = fast_exp2(sv[sp][3] - m1);
                } else {
                    pv[0] = m0 == -INFINITY ? 0.f : fast_exp2(sv[sp][0] - m0);
                    pv[1] = m1 == -INFINITY ? 0.f : fast_exp2(sv[sp][1] - m1);
                    pv[2] = m0 == -INFINITY ? 0.f : fast_exp2(sv[sp][2] - m0);
                    pv[3] = m1 == -INFINITY ? 0.f : fast_exp2(sv[sp][3] - m1);
                }
                l0 += pv[0] + pv[2];
                l1 += pv[1] + pv[3];
                const uint32_t h0 = Mma<TM>::pack(pv[0], pv[1]), h1 = Mma<TM>::pack(pv[2], pv[3]);
                pb[sp][0] = movmatrix_trans(h0);
                pb[sp][1] = movmatrix_trans(h1);
                if constexpr (kSplit) {
                    pl[sp][0] = movmatrix_trans(Mma<TM>::residual(pv[0], pv[1], h0));
                    pl[sp][1] = movmatrix_trans(Mma<TM>::residual(pv[2], pv[3], h1));
                }
            }

            // ---- O^T += V^T P^T, page by page
#pragma unroll
            for (int sp = 0; sp < kSP; ++sp) {
            if (!have[sp]) break;
            const int key0 = keyb[sp];
            const uint32_t pb0 = pb[sp][0], pb1 = pb[sp][1];
            const uint32_t pl0 = kSplit ? pl[sp][0] : 0u, pl1 = kSplit ? pl[sp][1] : 0u;
            const unsigned char *vpage = stages + stV * C::kUnitBytes + sp * L::kPageBytes;
            // Slots past the context hold stale data (maybe NaN): on a partial
            // page their V is zeroed in registers (their P is already 0).
            auto pv_page = [&](auto full_page) {
                constexpr bool kFull = decltype(full_page)::value;
                const int nvalid = min(kPage, k1 - key0);
                if constexpr (L::E == 2) {
                    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;  // keys (2tq, 2tq+1), (+8, +9)
                    if constexpr (!kFull) {
                        mlo = (vkey(0) < nvalid ? 0x0000ffffu : 0u) | (vkey(1) < nvalid ? 0xffff0000u : 0u);
                        mhi = (vkey(2) < nvalid ? 0x0000ffffu : 0u) | (vkey(3) < nvalid ? 0xffff0000u : 0u);
                    }
                    const uint32_t vbase = smem_u32(vpage);
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        uint32_t a[4];
                        // chunk 2 mt + (matrix & 1): flip bits 5-6 by 2 mt mod 8, add boxes
                        ldmatrix_x4_trans(a, vbase + ((voff[0] ^ (((2 * mt) & 7) << 4)) +
                                                      (mt >> 2) * L::kSubBytes));
                        if constexpr (!kFull) {
                            a[0] &= mlo;
                            a[1] &= mlo;
                            a[2] &= mhi;
                            a[3] &= mhi;
                        }
                        Mma<TM>::run(o[mt], a[0], a[1], a[2], a[3], pb0, pb1);
                        if constexpr (kSplit) Mma<TM>::run(o[mt], a[0], a[1], a[2], a[3], pl0, pl1);
                    }
                } else {
                    // D/32 words per key: dims gq*D/8 + 4 tp .. + 3; byte-interleave
                    // the key pairs, widen to f16, two m-tiles per word
                    constexpr int NW = D / 32;
                    uint32_t w[4][NW];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if constexpr (NW == 4) {
                            const uint4 v4 = *reinterpret_cast<const uint4 *>(vpage + voff[e]);
                            w[e][0] = v4.x;
                            w[e][1] = v4.y;
                            w[e][2] = v4.z;
                            w[e][3] = v4.w;
                        } else {
                            const uint2 v2 = *reinterpret_cast<const uint2 *>(vpage + voff[e]);
                            w[e][0] = v2.x;
                            w[e][1] = v2.y;
                        }
                        if constexpr (!kFull) {
                            const uint32_t keep = vkey(e) < nvalid ? 0xffffffffu : 0u;
#pragma unroll
                            for (int tp = 0; tp < NW; ++tp) w[e][tp] &= keep;
                        }
                    }
#pragma unroll
                    for (int tp = 0; tp < NW; ++tp) {
                        uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
                        e4m3x4_to_f16x4(__byte_perm(w[0][tp], w[1][tp], 0x5140), a0, a1);
                        e4m3x4_to_f16x4(__byte_perm(w[2][tp], w[3][tp], 0x5140), a2, a3);
                        e4m3x4_to_f16x4(__byte_perm(w[0][tp], w[1][tp], 0x7362), c0, c1);
                        e4m3x4_to_f16x4(__byte_perm(w[2][tp], w[3][tp], 0x7362), c2, c3);
                        Mma<TM>::run(o[2 * tp], a0, a1, a2, a3, pb0, pb1);
                        Mma<TM>::run(o[2 * tp + 1], c0, c1, c2, c3, pb0, pb1);
                    }
                }
            };
            if (key0 + kPage <= k1) pv_page(std::true_type{});
            else pv_page(std::false_type{});
          }
            __syncwarp();
            if (lane == 0) mbar_arrive_n(&empty[stV], release);
            return true;
        };
        // Unit j sits in the next stage pair of warp j mod 4.  A warp takes
        // its own units of an ordinary item, every unit of a group item.
        if (!grp) {
            uint32_t c = kGroups ? (handed >> (8 * warp)) & 0xffu : taken;
            for (int pu = warp; ok && pu < nunits; pu += kConsumerWarps, ++c)
                ok = run_unit(pu, pair_stage<C::kPairsPerWarp>(warp, c), (c / C::kPairsPerWarp) & 1u,
                              kRelease);
            if constexpr (!kGroups) taken = c;
        } else {
            for (int pu = 0; ok && pu < nunits; ++pu) {
                const int ow = pu % kConsumerWarps;
                const uint32_t c = ((handed >> (8 * ow)) & 0xffu) + (uint32_t)(pu / kConsumerWarps);
                ok = run_unit(pu, pair_stage<C::kPairsPerWarp>(ow, c), (c / C::kPairsPerWarp) & 1u, 1u);
            }
        }
        if (!ok) break;
        if constexpr (kGroups) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const uint32_t units = nunits > w ? (uint32_t)((nunits - w + kConsumerWarps - 1) / kConsumerWarps) : 0u;
                const uint32_t c = (((handed >> (8 * w)) & 0xffu) + units) & 0xffu;
                handed = (handed & ~(0xffu << (8 * w))) | (c << (8 * w));
            }
        }

        if (grp) {
            // ---- each warp's rows are complete: write them to their members'
            //      partial slots (the merge pass combines the partitions)
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, x);
                l1 += __shfl_xor_sync(0xffffffffu, l1, x);
            }
            // partial slot of the member holding row 8 warp + x, from the
            // walker's window (a group never crosses a 32-request window)
            auto slot_of = [&](int x) -> long long {
                const int gr = 8 * warp + x;
                const int rl = it.r - walk.rb + min(gr / p.G, members - 1);
                const int items = __shfl_sync(0xffffffffu, walk.items, rl);
                const int pincl = __shfl_sync(0xffffffffu, walk.pincl, rl);
                const int nsp = __shfl_sync(0xffffffffu, walk.nsplit, rl);
                return walk.pslot_base + (pincl - items) + (long long)it.g * nsp + it.split;
            };
            const long long ps0 = slot_of(2 * tq), ps1 = slot_of(2 * tq + 1);
            const int h0 = (8 * warp + 2 * tq) % p.G, h1 = (8 * warp + 2 * tq + 1) % p.G;
            const bool v0 = lim0 >= 0, v1 = lim1 >= 0;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                int dlo, dhi;
                if constexpr (L::E == 2) {
                    dlo = 16 * mt + gq;
                    dhi = dlo + 8;
                } else {
                    dlo = gq * (D / 8) + 4 * (mt >> 1) + 2 * (mt & 1);
                    dhi = dlo + 1;
                }
                if (v0) {
                    float *po = p.part_o + (ps0 * RPI + h0) * D;
                    po[dlo] = o[mt][0] * vs;
                    po[dhi] = o[mt][2] * vs;
                }
                if (v1) {
                    float *po = p.part_o + (ps1 * RPI + h1) * D;
                    po[dlo] = o[mt][1] * vs;
                    po[dhi] = o[mt][3] * vs;
                }
            }
            if (gq == 0) {
                if (v0) *reinterpret_cast<float2 *>(p.part_ml + (ps0 * RPI + h0) * 2) = make_float2(m0, l0);
                if (v1) *reinterpret_cast<float2 *>(p.part_ml + (ps1 * RPI + h1) * 2) = make_float2(m1, l1);
            }
            continue;
        }

        // ---- combine the four warps' states and write the item out
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, x);
            l1 += __shfl_xor_sync(0xffffffffu, l1, x);
        }
        constexpr int DC = C::kDC;
        if (gq == 0) {   // (m, l) once: the passes leave them in place
            if (2 * tq < RPI) {
                cw[RPI * DC + 2 * tq] = m0;
                cw[RPI * DC + RPI + 2 * tq] = l0;
            }
            if (2 * tq + 1 < RPI) {
                cw[RPI * DC + 2 * tq + 1] = m1;
                cw[RPI * DC + RPI + 2 * tq + 1] = l1;
            }
        }
#pragma unroll
        for (int hp = 0; hp < C::kCombPasses; ++hp) {
            // O^T element (dim row, item row): rows 2tq, 2tq+1 of this lane;
            // an m-tile's two dims of a lane lie in the same pass
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                int dlo, dhi;   // dims of the m-tile's rows gq and gq + 8
                if constexpr (L::E == 2) {
                    dlo = 16 * mt + gq;
                    dhi = dlo + 8;
                } else {
                    dlo = gq * (D / 8) + 4 * (mt >> 1) + 2 * (mt & 1);
                    dhi = dlo + 1;
                }
                const bool mine = L::E == 2 ? (16 * mt) / DC == hp : dlo / DC == hp;
                if (!mine) continue;
                dlo -= hp * DC;
                dhi -= hp * DC;
                if (2 * tq < RPI) {
                    cw[(2 * tq) * DC + dlo] = o[mt][0];
                    cw[(2 * tq) * DC + dhi] = o[mt][2];
                }
                if (2 * tq + 1 < RPI) {
                    cw[(2 * tq + 1) * DC + dlo] = o[mt][1];
                    cw[(2 * tq + 1) * DC + dhi] = o[mt][3];
                }
            }
            if (!consumer_sync(cbar, cpar, lane)) {
                flag(p.status, PA_CHECK_TIMEOUT);
                ok = false;
                break;
            }
            for (int o2 = tid; o2 < RPI * DC / 2; o2 += kConsumers) {
                const int r = o2 / (DC / 2);
                const int dl = (o2 % (DC / 2)) * 2, d = hp * DC + dl;
                const int rr = it.chunk * RPI + r;
                if (rr >= nrows) continue;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb[w * C::kComb + RPI * DC + r]);
                float Ls = 0.f, s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float *c = comb + w * C::kComb;
                    const float mw = c[RPI * DC + r];
                    const float sw = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                    Ls += sw * c[RPI * DC + RPI + r];
                    const float2 a = *reinterpret_cast<const float2 *>(c + r * DC + dl);
                    s0 += sw * a.x;
                    s1 += sw * a.y;
                }
                s0 *= vs;   // an FP8 pool's V scale; 1 otherwise
                s1 *= vs;
                if (it.pslot < 0) {
                    const float inv = 1.f / Ls;
                    const int h = it.g * p.G + rr % p.G;
                    TQ *dst = reinterpret_cast<TQ *>(p.out) +
                              ((long long)(qstart + rr / p.G) * p.Hq + h) * D + d;
                    *reinterpret_cast<uint32_t *>(dst) = Elt<TQ>::pack2(s0 * inv, s1 * inv);
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
        if (!ok) break;
    }
    // A consumer that stops early (a timed-out wait) releases every stage,
    // every queue entry and the item barrier once, so the others' bounded
    // waits and the producer's drain can finish.
    if (!ok && lane == 0) {
        for (int s = 0; s < kSt; ++s) mbar_arrive_n(&empty[s], kRelease);
        for (int e = 0; e < kQueue; ++e) mbar_arrive(&qempty[e]);
        mbar_arrive(cbar);
    }
}

// Second pass: for each (token, q head) of a request whose context was split,
// combine the partitions' (m, l, o): M = max m_s, o = sum 2^(m_s-M) o_s /
// sum 2^(m_s-M) l_s.  One CTA of 8 warps per (request, group of 8 / WPH q
// heads), looping over the request's few query tokens; WPH warps share a
// head, warp k of them taking partitions k, k + WPH, ...  Latency, not
// bytes, bounds it, so a warp issues its first kMergeBatch partial rows
// (lanes over dims) before anything that depends on the (m, l) values and
// loads each partition's (m, l) once (lanes over partitions); the WPH
// partial merges then combine the same way through shared memory.
// Launched as a programmatic dependent of the split-K kernel: its CTAs can
// become resident while that kernel's last items finish, and wait for all
// of its writes before reading.
constexpr int kMergeWarps = 8;
constexpr int kMergeBatch = 16;   // partial rows in flight per warp

template <int DPL> struct MergeVec;
template <> struct MergeVec<4> { using type = float4; };
template <> struct MergeVec<2> { using type = float2; };

template <typename V> __device__ __forceinline__ void fma_vec(float *o, float w, const V &v);
template <> __device__ __forceinline__ void fma_vec<float4>(float *o, float w, const float4 &v) {
    o[0] = fmaf(w, v.x, o[0]);
    o[1] = fmaf(w, v.y, o[1]);
    o[2] = fmaf(w, v.z, o[2]);
    o[3] = fmaf(w, v.w, o[3]);
}
template <> __device__ __forceinline__ void fma_vec<float2>(float *o, float w, const float2 &v) {
    o[0] = fmaf(w, v.x, o[0]);
    o[1] = fmaf(w, v.y, o[1]);
}

// B: partial rows in flight per warp (fewer registers for short contexts)
template <typename T, int D, int RPI, int WPH, int B>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const __grid_constant__ Params p) {
    constexpr int DPL = D / 32;
    constexpr int kHeads = kMergeWarps / WPH;   // heads per CTA
    using V = typename MergeVec<DPL>::type;
    __shared__ __align__(16) float sh_o[WPH > 1 ? kMergeWarps : 1][D];
    __shared__ float2 sh_ml[kMergeWarps];
    const int groups = (p.Hq + kHeads - 1) / kHeads;
    const int r = blockIdx.x / groups;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = (blockIdx.x % groups) * kHeads + warp / WPH;
    const int sub = warp % WPH;
    // A grid launched after this one as a programmatic dependent (the rest of
    // the tensor-core kernel's items) may be scheduled now: it reads nothing
    // this pass writes.
    if (threadIdx.x == 0) grid_launch_dependents();
    grid_dependency_wait();   // every write of the split-K kernel is visible past here
    if (r >= p.R) return;
    const int4 meta = reinterpret_cast<const int4 *>(p.req_meta)[r];
    const int nsplit = meta.z, nchunks = meta.w;
    if (nsplit <= 1) return;                    // the same for the whole CTA
    const bool active = h < p.Hq;               // a CTA's last heads may be past Hq
    const int t0 = p.qsl[r], n = p.qsl[r + 1] - t0;
    const long long pbase = (long long)(unsigned)meta.x | ((long long)meta.y << 32);
    const int g = h / p.G;
    const int cnt_w = nsplit > sub ? (nsplit - sub + WPH - 1) / WPH : 0;   // this warp's partitions
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
    for (int tl = 0; tl < n; ++tl) {
        const int rr = tl * p.G + h % p.G;
        const int chunk = rr / RPI, j = rr % RPI;
        const long long first = pbase + ((long long)g * nchunks + chunk) * nsplit;
        // this warp's i-th partition
        auto split = [&](int i) { return first + sub + (long long)i * WPH; };
        auto row = [&](int i) {
            return reinterpret_cast<const V *>(p.part_o + (split(i) * RPI + j) * D) + lane;
        };
        float o[DPL];
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[d] = 0.f;
        float M = -INFINITY, Lsum = 0.f;
        if (active && cnt_w > 0) {
            // the first batch of partial rows, and (m, l) of partitions lane, lane + 32, ...
            V v[B];
#pragma unroll
            for (int k = 0; k < B; ++k)
                if (k < cnt_w) v[k] = *row(k);
            const float2 ml0 = lane < cnt_w ? ml[split(lane) * RPI + j] : make_float2(-INFINITY, 0.f);
            M = ml0.x;
            for (int i = lane + 32; i < cnt_w; i += 32) M = fmaxf(M, ml[split(i) * RPI + j].x);
#pragma unroll
            for (int x = 16; x >= 1; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
            for (int i0 = 0; i0 < cnt_w; i0 += 32) {
                // weight of partition i0 + lane
                float2 mv = ml0;
                if (i0 > 0) mv = i0 + lane < cnt_w ? ml[split(i0 + lane) * RPI + j] : make_float2(-INFINITY, 0.f);
                const float w = mv.x == -INFINITY ? 0.f : fast_exp2(mv.x - M);
                Lsum += w * mv.y;
                const int cnt = min(32, cnt_w - i0);
                for (int k0 = 0; k0 < cnt; k0 += B) {
                    if (i0 + k0 > 0) {   // later batches (the first was issued above)
#pragma unroll
                        for (int k = 0; k < B; ++k)
                            if (k0 + k < cnt) v[k] = *row(i0 + k0 + k);
                    }
#pragma unroll
                    for (int k = 0; k < B; ++k) {
                        const float wk = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);
                        if (k0 + k < cnt) fma_vec(o, wk, v[k]);
                    }
                }
            }
#pragma unroll
            for (int x = 16; x >= 1; x >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, x);
        }
        if constexpr (WPH > 1) {
            // combine the WPH warps of each head: M = max M_k, o = sum 2^(M_k - M) o_k
#pragma unroll
            for (int d = 0; d < DPL; ++d) sh_o[warp][lane * DPL + d] = o[d];
            if (lane == 0) sh_ml[warp] = make_float2(M, Lsum);
            __syncthreads();
            if (sub == 0 && active) {
                float Mh = -INFINITY;
#pragma unroll
                for (int k = 0; k < WPH; ++k) Mh = fmaxf(Mh, sh_ml[warp + k].x);
                float acc[DPL], Lh = 0.f;
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
                for (int k = 0; k < WPH; ++k) {
                    const float2 mk = sh_ml[warp + k];
                    const float wk = mk.x == -INFINITY ? 0.f : fast_exp2(mk.x - Mh);
                    Lh += wk * mk.y;
                    fma_vec(acc, wk, reinterpret_cast<const V *>(sh_o[warp + k])[lane]);
                }
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[d] = acc[d];
                Lsum = Lh;
            }
            __syncthreads();   // shared memory is free for the next token
        }
        if (sub == 0 && active) {
            const float inv = 1.f / Lsum;
            T *dst = reinterpret_cast<T *>(p.out) + ((long long)(t0 + tl) * p.Hq + h) * D + lane * DPL;
#pragma unroll
            for (int d = 0; d < DPL; d += 2)
                *reinterpret_cast<uint32_t *>(dst + d) = Elt<T>::pack2(o[d] * inv, o[d + 1] * inv);
        }
    }
}

// Warps per head of the merge pass: enough that each warp's share of the
// longest context's partitions fits one batch of in-flight rows, but no more
// CTAs than about two waves (many short requests beside one long one keep
// the grid small instead).
static int merge_warps_per_head(long long max_splits, long long R, long long Hq) {
    int wph = 1;
    while (wph < kMergeWarps && max_splits > (long long)wph * kMergeBatch) wph *= 2;
    while (wph > 1 && R * ((Hq * wph + kMergeWarps - 1) / kMergeWarps) > 4LL * num_sms()) wph /= 2;
    return wph;
}

template <typename T, int D, int RPI, int WPH, int B = kMergeBatch>
static pa_status launch_merge(const Params &prm, cudaStream_t stream) {
    constexpr int kHeads = kMergeWarps / WPH;
    const long long groups = (prm.Hq + kHeads - 1) / kHeads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(prm.R * groups));
    cfg.blockDim = dim3(32 * kMergeWarps);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // Right behind the split-K grid: a programmatic dependent (its CTAs wait
    // in griddepcontrol.wait for that grid).  Launched later on its own (the
    // merge-only part), an ordinary launch: it starts once everything before
    // it in the stream has finished.
    cfg.numAttrs = prm.launch_part == 2 ? 0 : 1;
    PA_TRY_CUDA(cudaLaunchKernelEx(&cfg, merge_kernel<T, D, RPI, WPH, B>, prm));
    note_launch();
    return PA_OK;
}

template <typename TQ, typename TC, int D, int RPI, bool kGroups>
pa_status launch_split_k(Params &prm, long long max_items, cudaStream_t stream) {
    using S = Cfg<TC, D, RPI>;
    static int resident[64] = {};  // CTAs per SM, per device
    int dev = 0;
    PA_TRY_CUDA(cudaGetDevice(&dev));
    int per_sm = dev < 64 ? resident[dev] : 0;
    if (per_sm == 0) {
        PA_TRY_CUDA(cudaFuncSetAttribute(paged_decode_kernel<TQ, TC, D, RPI, kGroups>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes));
        PA_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, paged_decode_kernel<TQ, TC, D, RPI, kGroups>, kThreads, S::kBytes));
        if (per_sm < 1) return PA_ERR_UNSUPPORTED;
        if (dev < 64) resident[dev] = per_sm;
    }
    // Persistent grid: every resident slot once, no more CTAs than items.
    long long grid = (long long)per_sm * num_sms();
    if (max_items < grid) grid = max_items;
    if (grid < 1) grid = 1;
    if (prm.launch_pdl) {
        // Beside the tensor-core kernel's first grid: this grid may start
        // while it runs (it reads nothing that grid writes), its CTAs taking
        // the SMs that grid leaves free, then the rest as its CTAs exit.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = S::kBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        PA_TRY_CUDA(cudaLaunchKernelEx(&cfg, paged_decode_kernel<TQ, TC, D, RPI, kGroups>, prm));
    } else {
        paged_decode_kernel<TQ, TC, D, RPI, kGroups><<<(int)grid, kThreads, S::kBytes, stream>>>(prm);
        PA_TRY_CUDA(cudaGetLastError());
    }
    note_launch();
    return PA_OK;
}

template <typename TQ, typename TC, int D, int RPI>
pa_status launch_typed(Params &prm, long long max_items, long long merge_splits, bool groups,
                       cudaStream_t stream) {
    if (prm.launch_part != 2) {
        const pa_status st = groups ? launch_split_k<TQ, TC, D, RPI, true>(prm, max_items, stream)
                                    : launch_split_k<TQ, TC, D, RPI, false>(prm, max_items, stream);
        if (st != PA_OK) return st;
    }
    if (merge_splits > 0 && prm.R > 0 && prm.launch_part != 1) {
        switch (merge_warps_per_head(merge_splits, prm.R, prm.Hq)) {
            case 1:   // at most 8 partitions: a batch of 8 rows, more warps resident
                return merge_splits <= 8 ? launch_merge<TQ, D, RPI, 1, 8>(prm, stream)
                                         : launch_merge<TQ, D, RPI, 1>(prm, stream);
            case 2: return launch_merge<TQ, D, RPI, 2>(prm, stream);
            case 4: return launch_merge<TQ, D, RPI, 4>(prm, stream);
            default: return launch_merge<TQ, D, RPI, 8>(prm, stream);
        }
    }
    return PA_OK;
}

template <typename TQ, typename TC, int D>
pa_status dispatch_rpi(int rpi, Params &prm, long long grid, long long merge, bool groups,
                       cudaStream_t stream) {
    switch (rpi) {
        case 1: return launch_typed<TQ, TC, D, 1>(prm, grid, merge, groups, stream);
        case 2: return launch_typed<TQ, TC, D, 2>(prm, grid, merge, groups, stream);
        case 4: return launch_typed<TQ, TC, D, 4>(prm, grid, merge, groups, stream);
        default: return launch_typed<TQ, TC, D, 8>(prm, grid, merge, groups, stream);
    }
}

template <typename TQ>
pa_status dispatch_cache(bool fp8, int D, int rpi, Params &prm, long long grid, long long merge,
                         bool groups, cudaStream_t stream) {
    if (fp8)
        return D == 128 ? dispatch_rpi<TQ, Fp8E4M3, 128>(rpi, prm, grid, merge, groups, stream)
                        : dispatch_rpi<TQ, Fp8E4M3, 64>(rpi, prm, grid, merge, groups, stream);
    return D == 128 ? dispatch_rpi<TQ, TQ, 128>(rpi, prm, grid, merge, groups, stream)
                    : dispatch_rpi<TQ, TQ, 64>(rpi, prm, grid, merge, groups, stream);
}

// The fp16 instantiations compile in a translation unit of their own
// (decode_fp16.cu includes this file with PA_DECODE_FP16_UNIT defined), in
// parallel with the bf16 ones here.
pa_status dispatch_fp16(bool fp8, int D, int rpi, Params &prm, long long grid, long long merge,
                        bool groups, cudaStream_t stream);
#ifdef PA_DECODE_FP16_UNIT
pa_status dispatch_fp16(bool fp8, int D, int rpi, Params &prm, long long grid, long long merge,
                        bool groups, cudaStream_t stream) {
    return dispatch_cache<__half>(fp8, D, rpi, prm, grid, merge, groups, stream);
}
#endif

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
// A whole partition holds at least 32 pages: the split-K kernel's group check
// reads a partition's first 32 block ids at once.
static_assert(kPreferredPartition % (32 * kPage) == 0, "partitions of whole 32-page groups");
constexpr size_t kAlign = 256;

inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace decode

#ifndef PA_DECODE_FP16_UNIT
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
    const bool fp8 = a.cache_dtype == PA_FP8_E4M3;
    const int elt = fp8 ? 1 : 2;
    if (!encode_pool_map_swizzled(&prm.tmK, a.kc, slots, a.Hkv, a.D, elt, kPage) ||
        !encode_pool_map_swizzled(&prm.tmV, a.vc, slots, a.Hkv, a.D, elt, kPage))
        return PA_ERR_CUDA;
    prm.k_scale = a.k_scale;
    prm.v_scale = a.v_scale;
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
    prm.max_seq = a.max_seq;
    prm.qscale = a.scale * 1.4426950408889634f;
    prm.status = status_word();
    if (!prm.status) return PA_ERR_CUDA;
    prm.launch_pdl = a.pdl ? 1 : 0;
    prm.launch_part = a.decode_part;
    prm.item_counter = a.ctrl ? a.ctrl + kCtrlDecodeCounter : nullptr;
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
            // the same bytes per partition in every layout: 512 keys of a
            // 16-bit pool at head_dim 128 (256 KiB of K and V per kv head),
            // 1024 at head_dim 64 or over FP8 pools, 2048 for both.  FP8
            // decode at 1024 keys: 220.6 -> 211.6 us on the decode batch.
            prm.p_min = kPreferredPartition * (256 / (a.D * elt));
            merge = true;
            // Every request is at most max_seq long (longer ones are flagged
            // and skipped), so when the workspace holds the partials of this
            // bound at p_min the kernel needs no pass over the requests to
            // choose a partition length.
            const long long bound = (long long)a.Hkv *
                                    ((long long)a.R + ((long long)a.T * prm.G + rpi - 1) / rpi) *
                                    ((a.max_seq + prm.p_min - 1) / prm.p_min);
            prm.part_fixed = cap >= bound ? 1 : 0;
        }
    }

    // Upper bound on the work items (the grid never exceeds it).
    const long long splits = prm.p_min >= kSingle ? 1 : (a.max_seq + prm.p_min - 1) / prm.p_min;
    const long long chunks = (long long)a.R + ((long long)a.T * prm.G + rpi - 1) / rpi;
    const long long grid = (long long)a.Hkv * chunks * splits;

    // the merge pass (when partitions exist) sizes itself by the most partitions a request can have
    const long long merge_splits = merge ? splits : 0;
    // group items need the partial slots (a merge pass) and the item queue
    const bool groups = (a.flags & PA_ATTN_SHARED_BLOCKS) && merge && a.ctrl;
    return a.dtype == PA_BF16
               ? dispatch_cache<__nv_bfloat16>(fp8, a.D, rpi, prm, grid, merge_splits, groups, stream)
               : dispatch_fp16(fp8, a.D, rpi, prm, grid, merge_splits, groups, stream);
}
#endif  // PA_DECODE_FP16_UNIT

}  // namespace pa
