// Paged attention for long query chunks (prompt prefill) on the 5th-generation
// tensor cores: tcgen05.mma with operands staged by TMA, accumulators in TMEM.
//
// "How vLLM Works Internally", sections "How the Kernel Works" and the
// prefill/decode split (prefill is compute-bound); "Inside vLLM", the read
// path (cu_seqlens_q, seqused_k, block_table).  Same maths as the split-K
// kernel: out = softmax(scale * q K^T, causal) V per request and kv head.
//
// Work item = (request, kv head g, pair of row tiles).  A row is one
// (query token, q head of group g) pair, so a K/V tile serves all G = Hq/Hkv
// heads of the group and both 128-row tiles ("slots" A and B) of the pair.
// A tile holds TT = floor(128/G) whole tokens (TT*G rows, token-major); each
// Q tile is one 3-D TMA box {64 dims, G heads, TT tokens} per 64-dim half.
// When G does not divide 128 the last 128 - TT*G rows of every Q buffer are
// zeroed once and never loaded or written out.  Items run on persistent
// CTAs (one per SM), heaviest first.
//
// Per 128-key KV tile j (8 pages of 16 tokens, each page one TMA box per
// 64-dim half, 128-byte swizzle, addressed through the block table), for
// each slot X in {A, B}:
//   S_X = Q_X K_j^T       tcgen05.mma, A = Q (smem, K-major), B = K (smem,
//                         K-major), fp32 accumulator in TMEM
//   P_X = exp2(S_X*c - m) the slot's softmax warps, one row per thread
//                         (tcgen05.ld), written back over S_X in TMEM
//   O_X += P_X V_j        tcgen05.mma, A = P (TMEM), B = V (smem, MN-major)
// The MMA warp issues PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1): while one
// slot's softmax runs, the tensor core works for the other slot.  The
// running max only moves (and O is rescaled in TMEM) when a tile's max
// exceeds it by more than 2^8; otherwise P keeps the old reference, which
// bounds every P by 256 and leaves the result exact.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (+ TMEM allocation), 2..5 = slot A
// softmax and epilogue, 6..9 = slot B; warp w reads TMEM lanes 32*(w%4)..+31.
// Every mbarrier wait is bounded.
//
// FP8 (E4M3) pools: the MMAs run in f16 (E4M3 widens to f16 exactly; a bf16
// q is rounded to f16).  At head_dim 128 each FP8 page lands (one 128-byte
// row per slot, swizzled) in the upper half of its f16 tile buffer, where an
// FP8 row takes exactly the bytes of its own upper-half f16 row; at head_dim
// 64 it lands (64-byte rows, unswizzled) in a staging area of its own.  Two
// more warps (10, 11) widen the tile into the f16 layout, row by row, and
// only then signal the tile full.  K's scale joins the softmax scale, V's
// scales the output.
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>
#include <type_traits>

#include "pa_internal.cuh"

namespace pa {
namespace prefill {

constexpr int kBM = 128;          // rows per tile
constexpr int kBN = 128;          // keys per KV tile
constexpr int kPage = 16;
constexpr int kPagesPerTile = kBN / kPage;
constexpr int kSoftmaxWarps = 8;   // four per slot
constexpr int kConvWarps = 2;      // FP8 pools: E4M3 -> f16; bf16 pools: V tiles bf16 -> f16
__host__ __device__ constexpr int threads_for(bool conv) {
    return (2 + kSoftmaxWarps + (conv ? kConvWarps : 0)) * 32;
}
// Which tiles the two converter warps rewrite in shared memory before the
// tensor core reads them.  FP8 pools: Q (bf16 -> f16), K and V (E4M3 -> f16).
// bf16 pools: V only, so that P enters PV as f16 (11 significant bits; a
// bf16 P would add up to 2^-9 of |v| to the error).  fp16 pools: none.
template <typename T, bool F8>
struct Conv {
    static constexpr bool kV = !F8 && std::is_same<T, __nv_bfloat16>::value;
    static constexpr bool kAny = F8 || kV;
};
// Largest magnitude (bits without the sign) of a bf16 value that f16
// represents: 65280; the next bf16 value, 65536, is past f16's 65504.
constexpr uint32_t kBf16F16Max = 0x477Fu;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kTauDefault = 16;           // longer query chunks take this kernel

struct Params {
    CUtensorMap tmQ;
    CUtensorMap tmK;
    CUtensorMap tmV;
    CUtensorMap tmVw;   // bf16 pools: the prefill requests' V widened to f16 (below)
    void *out;
    const int32_t *bt;
    const int32_t *qsl;
    const int32_t *seq_lens;
    int R, T, MB, NB, Hq, Hkv, G;
    int TT;         // query tokens per 128-row tile: floor(128 / G)
    int tau;        // requests with more than tau query tokens are handled here
    float qscale;   // softmax scale * log2(e)
    const float *k_scale, *v_scale;   // FP8 pools (device scalars; NULL = 1)
    unsigned int *item_counter;       // zeroed before launch: items are taken in order
                                      // as CTAs free up (NULL: fixed snake order)
    // bf16 pools: V of the prefill requests widened to f16 once per call by
    // widen_v_kernel, token-major like a pool (NULL: not widened).  w_off[r]
    // is request r's first token there, or -1; w_flag[page * Hkv + head] is
    // 1 where a value of that page f16 cannot hold (the tile then comes from
    // the pool and is converted in the kernel, with the bf16 route).
    const int32_t *w_off;
    const uint8_t *w_flag;
    unsigned int *status;
};

template <int D>
struct Cfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kQBytes = kBM * D * 2;          // one 128-row Q tile
    static constexpr int kTileBytes = kBN * D * 2;
    static constexpr int kHalfBytes = kBN * 128;         // one 64-dim half of a K/V tile
    static constexpr int kPageHalfBytes = kPage * 128;
    // Q (2 tiles), K (2 stages), V (vst stages), barriers and slack to align
    static constexpr int smem(int vst) { return 2 * kQBytes + (2 + vst) * kTileBytes + 512 + 1024; }
    // FP8 pools at head_dim 64: 64-byte rows of K and V, two stages each,
    // staged after the barriers (1024-byte aligned) before widening
    static constexpr int kLandBytes = kBN * 64;
    static constexpr int kLandOffset = 2 * kQBytes + 4 * kTileBytes + 1024;
    static constexpr int kSmemF8Land = kLandOffset + 4 * kLandBytes + 1024;
    // TMEM columns: S_A 0, O_A 128, S_B 256, O_B 384
    __device__ static constexpr uint32_t col_s(int slot) { return (uint32_t)slot * 256; }
    __device__ static constexpr uint32_t col_o(int slot) { return (uint32_t)slot * 256 + 128; }
};

// Barrier slots (uint64) in shared memory.
enum {
    B_QFULL = 0, B_QEMPTY, B_KFULL, B_KFULL1, B_KEMPTY, B_KEMPTY1,
    B_VFULL,                 // [3] per V stage (two or three in use)
    B_VEMPTY = B_VFULL + 3,  // [3]
    B_SFULL = B_VEMPTY + 3,  // [2] per slot: S_X ready
    B_PFULL = B_SFULL + 2,   // [2] per slot: P_X written (one arrive per softmax warp)
    B_ODONE = B_PFULL + 2,   // [2] per slot: the item's last PV_X done
    B_OFREE = B_ODONE + 2,   // [2] per slot: O_X read out by the epilogue
    B_DRAIN = B_OFREE + 2,
    B_QLAND,      // FP8 pools: TMA bytes landed, before widening
    B_KLAND, B_KLAND1,
    B_VLAND,                      // [3]
    B_IFULL = B_VLAND + 3,        // [kQueue] item queue entry written by the producer
    B_IEMPTY = B_IFULL + 4,       // [kQueue] entry read by every other warp
    B_SPLITREQ = B_IEMPTY + 4,    // [2] per slot: the MMA warp asks for P as bf16 pairs
    B_SPLITDONE = B_SPLITREQ + 2, // [2] per slot: P rewritten (one arrive per softmax warp)
    B_COUNT = B_SPLITDONE + 2
};
constexpr int kQueue = 4;         // items the producer may run ahead

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3fff);
    d |= (uint64_t)((lbo >> 4) & 0x3fff) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3fff) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for this architecture
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

template <typename T>
__device__ __forceinline__ uint32_t instr_desc(int M, int N, int b_mn_major) {
    constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    uint32_t d = 1u << 4;  // fp32 accumulator
    d |= fmt << 7;         // A type
    d |= fmt << 10;        // B type
    d |= (uint32_t)b_mn_major << 16;
    d |= (uint32_t)(N >> 3) << 17;
    d |= (uint32_t)(M >> 4) << 24;
    return d;
}

// The MMA and commit wrappers are executed by the whole (converged) MMA warp
// with warp-uniform operands; one lane, chosen by elect.sync, issues.
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p, e;\nelect.sync _|e, 0xffffffff;\nsetp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p, e;\nelect.sync _|e, 0xffffffff;\nsetp.ne.b32 p, %4, 0;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM words: each thread gets its lane's 32.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Whether the phase with the given parity has completed (never blocks).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------------------
// Work items: per request with more than tau tokens, Hkv x ceil(n/(2 TT))
// tile pairs, ordered last pair first (the tile with the most keys), kv heads
// interleaved.  Every warp walks the request list itself.
// ---------------------------------------------------------------------------

struct Item {
    int r, g, mt, n, L, qstart;
};

struct Walker {
    const Params *p;
    int rb;
    long long base;  // items before the window
    int n, L, a, items, incl, total;

    __device__ void load(int lane) {
        const int r = rb + lane;
        n = 0;
        L = 0;
        a = 0;
        items = 0;
        if (r < p->R) {
            a = p->qsl[r];
            const int b = p->qsl[r + 1];
            n = b - a;
            L = p->seq_lens[r];
            const bool sane = a >= 0 && b <= p->T && n >= 0 && L >= n &&
                              (L + kPage - 1) / kPage <= p->MB;
            if (sane && n > p->tau) items = p->Hkv * ((n + 2 * p->TT - 1) / (2 * p->TT));
        }
        incl = items;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        total = __shfl_sync(0xffffffffu, incl, 31);
    }
    __device__ void begin(const Params *params, int lane) {
        p = params;
        rb = 0;
        base = 0;
        load(lane);
    }
    __device__ bool find(long long i, int lane, Item &it) {
        while (i >= base + total) {
            base += total;
            rb += 32;
            if (rb >= p->R) return false;
            load(lane);
        }
        const int li = (int)(i - base);
        const int src = __ffs(__ballot_sync(0xffffffffu, incl > li)) - 1;
        const int excl = __shfl_sync(0xffffffffu, incl - items, src);
        it.n = __shfl_sync(0xffffffffu, n, src);
        it.L = __shfl_sync(0xffffffffu, L, src);
        it.qstart = __shfl_sync(0xffffffffu, a, src);
        it.r = rb + src;
        const int local = li - excl;
        const int nm = (it.n + 2 * p->TT - 1) / (2 * p->TT);
        it.g = local % p->Hkv;
        it.mt = nm - 1 - local / p->Hkv;  // index of the tile pair
        return true;
    }
};

// The k-th item of CTA b: rounds of gridDim items, dealt left to right in
// even rounds and right to left in odd ones, so the heavy items at the front
// of the list spread evenly over the CTAs.
__device__ __forceinline__ long long snake_item(int k) {
    const long long round = (long long)k * gridDim.x;
    return (k & 1) ? round + (gridDim.x - 1 - blockIdx.x) : round + blockIdx.x;
}

// KV tiles slot `slot` of an item needs: keys 0 .. (last position any of its
// rows sees); 0 when the slot has no rows.
__device__ __forceinline__ int slot_tiles(const Params &p, const Item &it, int slot) {
    const int first_tok = (it.mt * 2 + slot) * p.TT;
    if (first_tok >= it.n) return 0;
    const int last_tok = min(first_tok + p.TT, it.n) - 1;
    const int max_pos = it.L - it.n + last_tok;
    return (max_pos + kBN) / kBN;
}

// Widen the E4M3 rows [r0, r1) of a 128-row tile in place: the FP8 tile sits
// in the upper 64-dim half (row r at half1 + 128 r, 128-byte swizzle); each
// row becomes two f16 rows (dims 0-63 in the lower half, 64-127 in the upper),
// same swizzle.  A warp reads 16 rows whole (four 16-byte loads in flight per
// lane) before it writes them; r1 - r0 is a multiple of 16.
__device__ __forceinline__ void widen_e4m3_tile(unsigned char *tile, int half_bytes, int r0, int r1,
                                                int lane) {
    const int c = lane & 7;                 // 16 dims 16c .. 16c+15 of the row
    const int fc = 2 * (c & 3);             // f16 chunks fc, fc+1 of a half row
    for (int rb = r0; rb < r1; rb += 16) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = rb + 4 * u + (lane >> 3);
            v[u] = *reinterpret_cast<const uint4 *>(tile + half_bytes + r * 128 + ((c ^ (r & 7)) << 4));
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = rb + 4 * u + (lane >> 3), x = r & 7;
            uint32_t h[8];
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                asm("{\n.reg .b16 l, hh;\nmov.b32 {l, hh}, %2;\n"
                    "cvt.rn.f16x2.e4m3x2 %0, l;\ncvt.rn.f16x2.e4m3x2 %1, hh;\n}"
                    : "=r"(h[2 * e]), "=r"(h[2 * e + 1])
                    : "r"(w[e]));
            }
            unsigned char *dst_row = tile + (c >> 2) * half_bytes + r * 128;
            *reinterpret_cast<uint4 *>(dst_row + ((fc ^ x) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(dst_row + (((fc + 1) ^ x) << 4)) =
                make_uint4(h[4], h[5], h[6], h[7]);
        }
        __syncwarp();
    }
}

// Round a bf16 tile to f16 in place (same positions, same swizzle).
__device__ __forceinline__ void bf16_tile_to_f16(unsigned char *tile, int bytes, int t, int nt) {
    for (int o = t * 16; o < bytes; o += nt * 16) {
        uint4 v = *reinterpret_cast<const uint4 *>(tile + o);
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[e] << 16),
                                                __uint_as_float(w[e] & 0xffff0000u));
            w[e] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(tile + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Widen the E4M3 rows [r0, r1) of a 64-dim tile: row r's 64 bytes sit
// unswizzled at land + 64 r; its 64 f16 values become row r of the f16 tile
// (128 bytes, 128-byte swizzle).  Lane: row r0 + 8u + lane/4, 16 dims
// 16 (lane%4) .. +15 (two f16 chunks).  r1 - r0 is a multiple of 32.
__device__ __forceinline__ void widen_e4m3_rows64(const unsigned char *land, unsigned char *tile,
                                                  int r0, int r1, int lane) {
    const int c = lane & 3;
    for (int rb = r0; rb < r1; rb += 32) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = rb + 8 * u + (lane >> 2);
            v[u] = *reinterpret_cast<const uint4 *>(land + r * 64 + (c << 4));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = rb + 8 * u + (lane >> 2), x = r & 7;
            uint32_t h[8];
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                asm("{\n.reg .b16 l, hh;\nmov.b32 {l, hh}, %2;\n"
                    "cvt.rn.f16x2.e4m3x2 %0, l;\ncvt.rn.f16x2.e4m3x2 %1, hh;\n}"
                    : "=r"(h[2 * e]), "=r"(h[2 * e + 1])
                    : "r"(w[e]));
            }
            unsigned char *dst_row = tile + r * 128;
            *reinterpret_cast<uint4 *>(dst_row + (((2 * c) ^ x) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(dst_row + (((2 * c + 1) ^ x) << 4)) =
                make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

// One 64-key half of a bf16 V tile (keys 64 h .. 64 h + 63: 8 KiB of
// 128-byte rows in each 64-dim half of the tile, at v0 + dh * half_bytes)
// to f16 in place, when f16 holds every value of its first `valid` keys
// (the keys inside the context; the rest is zeroed before the tensor core
// reads the tile).  Elementwise, so the swizzle does not matter.  Values
// below f16's normal range round to its subnormals (an absolute error of
// 2^-25 at most).  Returns 0 when converted; 1 when some value is past
// 65280 in magnitude, infinite or NaN: the half stays bf16 (its P is then
// written as a bf16 pair).
template <int kHalves>
__device__ __forceinline__ int v_half_to_f16(unsigned char *v0, int half_bytes, int valid, int lane) {
    uint32_t mx = 0;
#pragma unroll
    for (int dh = 0; dh < kHalves; ++dh)
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            const int c = lane + 32 * i;   // 16-byte chunk; row c / 8
            if (c / 8 < valid) {
                const uint4 x = *reinterpret_cast<const uint4 *>(v0 + dh * half_bytes + c * 16);
                mx = __vmaxu2(mx, x.x & 0x7fff7fffu);
                mx = __vmaxu2(mx, x.y & 0x7fff7fffu);
                mx = __vmaxu2(mx, x.z & 0x7fff7fffu);
                mx = __vmaxu2(mx, x.w & 0x7fff7fffu);
            }
        }
    mx = __reduce_max_sync(0xffffffffu, max(mx & 0xffffu, mx >> 16));
    if (mx > kBf16F16Max) return 1;
#pragma unroll
    for (int dh = 0; dh < kHalves; ++dh)
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
            uint4 *ptr = reinterpret_cast<uint4 *>(v0 + dh * half_bytes + (lane + 32 * i) * 16);
            uint4 x = *ptr;
            uint32_t *w = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __half2 h = __floats2half2_rn(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
                w[e] = *reinterpret_cast<uint32_t *>(&h);
            }
            *ptr = x;
        }
    return 0;
}

// Rewrite the f16 P of the key halves set in `halves` (bit h: keys 64h ..
// 64h+63, columns 64h .. 64h+31 of this warp's TMEM lanes) as bf16 pairs:
// hi = bf16(p) in the same columns, lo = bf16(p - hi) in 64h+32 .. 64h+63.
// Both are exact: an f16 value's 11 significant bits are hi's 8 and lo's 3.
__device__ __noinline__ void split_p_halves(uint32_t colS, int halves) {
    for (int h = 0; h < 2; ++h) {
        if (!((halves >> h) & 1)) continue;
        for (int c0 = 0; c0 < 32; c0 += 16) {
            uint32_t w[16], wl[16];
            tmem_ld16(colS + 64 * h + c0, w);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                float a, b, ha, hb;
                Elt<__half>::unpack2(w[e], a, b);
                w[e] = Elt<__nv_bfloat16>::pack2(a, b);
                Elt<__nv_bfloat16>::unpack2(w[e], ha, hb);
                wl[e] = Elt<__nv_bfloat16>::pack2(a - ha, b - hb);
            }
            tmem_st16(colS + 64 * h + c0, w);
            tmem_st16(colS + 64 * h + 32 + c0, wl);
        }
    }
    tmem_wait_st();
}

// The MMA warp's PV of one tile when some key half of its V stayed bf16
// (bits of `bfh`): ask the slot's softmax warps to rewrite those halves' f16
// P as bf16 pairs and wait for them, then issue PV with one f16 MMA per 16
// keys of an f16 half and two bf16 MMAs (hi, lo) per 16 keys of a bf16 half.
// Called by the whole MMA warp; false when the wait ran out.
__device__ __noinline__ bool pv_with_bf16_halves(uint64_t *req, uint64_t *done, volatile int *fmt,
                                                 int bfh, uint32_t *nsplit, uint32_t col_o,
                                                 uint32_t col_s, uint64_t dv0, uint32_t idPV,
                                                 uint32_t idPVb, bool accumulate) {
    if ((threadIdx.x & 31) == 0) {
        *fmt = bfh;
        mbar_arrive(req);
    }
    if (!mbar_wait_warp(done, *nsplit & 1u)) return false;
    ++*nsplit;
    tc_fence_after();
    for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint32_t pa = col_s + (kk >> 2) * 64 + (kk & 3) * 8;
        const uint64_t dv = dv0 + (uint64_t)(kk * 2048 >> 4);
        const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
        if ((bfh >> (kk >> 2)) & 1) {
            mma_ts(col_o, pa, dv, idPVb, acc);
            mma_ts(col_o, pa + 32, dv, idPVb, 1u);
        } else {
            mma_ts(col_o, pa, dv, idPV, acc);
        }
    }
    return true;
}

template <typename T, int D, bool F8>
__global__ void __launch_bounds__(threads_for(Conv<T, F8>::kAny), 1)
paged_prefill_kernel(const __grid_constant__ Params p) {
    using C = Cfg<D>;
    // QK runs in q's type (f16 over FP8 pools); PV runs in f16: P as f16
    // and V as f16 (bf16 pools: converted in shared memory first).  A bf16
    // V half that f16 cannot hold stays bf16, and its f16 P is rewritten as
    // two bf16 terms (split_p_halves) for two PV MMAs: the same P, exactly.
    // P of keys 64h .. 64h+63 of a tile: f16 (or hi) in S columns 64h ..
    // 64h+31, lo in 64h+32 .. 64h+63.
    using TQK = typename std::conditional<F8, __half, T>::type;
    constexpr bool kConvV = Conv<T, F8>::kV;
    constexpr bool kConv = Conv<T, F8>::kAny;
    // V ring stages.  bf16 pools take three: a V tile must land and then be
    // converted by the converter warps before the MMA warp takes the tile,
    // and with two stages its copy could only start once the PV two tiles
    // back had released the stage (measured slower: 410 against 366 us on a
    // 5000-token chunk, before V was widened once per call).
    constexpr int kVSt = kConvV ? 3 : 2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sQ = base;                       // 2 tiles: slot A, slot B
    unsigned char *sK = sQ + 2 * C::kQBytes;        // 2 stages
    unsigned char *sV = sK + 2 * C::kTileBytes;     // kVSt stages
    uint64_t *bar = reinterpret_cast<uint64_t *>(sV + kVSt * C::kTileBytes);
    unsigned char *sL = base + C::kLandOffset;      // FP8 at head_dim 64: [K st0, K st1, V st0, V st1]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *q_items = reinterpret_cast<volatile int *>(tmem_slot + 2);   // [kQueue]
    // bf16 pools: per V stage and key half, 1 when the half stayed bf16
    volatile int *v_fmt = reinterpret_cast<volatile int *>(tmem_slot + 2 + kQueue);   // [kVSt][2]
    volatile int *split_fmt = v_fmt + 2 * 3;   // [2]: halves of the requested P rewrite
    // bf16 pools: per V stage, 1 when the tile came widened (no conversion)
    volatile int *v_src = split_fmt + 2;        // [3]
    static_assert(B_COUNT * 8 + (2 + kQueue + 2 * 3 + 2 + 3) * 4 <= 512, "control block");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // A grid launched after this one as a programmatic dependent (the
    // split-K kernel beside this grid) may be scheduled at once: it reads
    // nothing this kernel writes.
    if (tid == 0) grid_launch_dependents();

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            const bool per_warp = (i >= B_PFULL && i < B_PFULL + 2) || (i >= B_OFREE && i < B_OFREE + 2) ||
                                  (i >= B_SPLITDONE && i < B_SPLITDONE + 2);
            // FP8: Q/K/V full are signalled by the widening warps; bf16: V full
            const bool widened = (F8 && (i == B_QFULL || (i >= B_KFULL && i <= B_KFULL1))) ||
                                 (kConv && i >= B_VFULL && i < B_VFULL + 3);
            const bool readers = i >= B_IEMPTY && i < B_IEMPTY + kQueue;   // every warp but 0
            mbar_init(&bar[i], readers ? 1 + kSoftmaxWarps + (kConv ? kConvWarps : 0)
                                       : per_warp ? kSoftmaxWarps / 2 : (widened ? kConvWarps : 1));
        }
        fence_mbar_init();
        prefetch_tensor_map(&p.tmQ);
        prefetch_tensor_map(&p.tmK);
        prefetch_tensor_map(&p.tmV);
    }
    {
        // Rows TT*G .. 127 of both Q tiles (G does not divide 128): no box
        // lands there, so zero them once and their scores stay finite.  With
        // the 128-byte swizzle a row keeps its own 128 bytes of each half.
        const int pad0 = p.TT * p.G, per = (kBM - pad0) * 8;   // 16-byte chunks per half
        for (int i = tid; i < 2 * C::kHalves * per; i += blockDim.x)
            *reinterpret_cast<uint4 *>(sQ + (i / per) * (kBM * 128) + (pad0 + (i % per) / 8) * 128 +
                                       (i % 8) * 16) = make_uint4(0, 0, 0, 0);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    Walker walk;
    walk.begin(&p, lane);
    Item it;

    auto fail = [&](void) {
        flag(p.status, PA_CHECK_TIMEOUT);
        *abort_flag = 1;
    };
    // The k-th item of this CTA, as every warp but the producer sees it:
    // with an item counter, the index the producer published in queue entry
    // k % kQueue (-1: no more items); otherwise the fixed snake order.
    auto item_at = [&](int k) -> long long {
        if (!p.item_counter) return snake_item(k);
        const int e = k % kQueue;
        if (!mbar_wait_warp(&bar[B_IFULL + e], (uint32_t)((k / kQueue) & 1))) {
            if (lane == 0) fail();
            return -1;
        }
        const long long v = q_items[e];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_IEMPTY + e]);
        return v;
    };
    // The producer's k-th item: the next index from the counter (the list is
    // heaviest first, so CTAs that free up early take the next heaviest),
    // published for the other warps.  False when the list is done (or a wait
    // timed out; *timed_out tells which).
    auto next_item = [&](int k, bool *timed_out) -> bool {
        *timed_out = false;
        if (!p.item_counter) return walk.find(snake_item(k), lane, it);
        unsigned int cand = 0;
        if (lane == 0) cand = atomicAdd(p.item_counter, 1u);
        cand = __shfl_sync(0xffffffffu, cand, 0);
        const bool valid = walk.find((long long)cand, lane, it);
        const int e = k % kQueue;
        if (!mbar_wait_warp(&bar[B_IEMPTY + e], (uint32_t)(((k / kQueue) & 1) ^ 1))) {
            *timed_out = true;
            return false;
        }
        if (lane == 0) {
            q_items[e] = valid ? (int)cand : -1;
            mbar_arrive(&bar[B_IFULL + e]);
        }
        __syncwarp();
        return valid;
    };

    if (warp == 0) {
        // =================== TMA producer ===================
        long long t = 0;  // KV tiles issued so far (both rings advance per tile)
        int items = 0;
        bool ok = true;
        long long lastK = -1, lastV = -1;
        for (int k = 0; ok; ++k, ++items) {
            bool timed_out = false;
            if (!next_item(k, &timed_out)) {
                if (timed_out) ok = false;
                break;
            }
            const int ntB = slot_tiles(p, it, 1);
            const int nt = max(slot_tiles(p, it, 0), ntB);
            const int32_t *row = p.bt + (long long)it.r * p.MB;
            const int ctx_pages = (it.L + kPage - 1) / kPage;
            // bf16 pools: the request's first token in the widened V, or -1
            int woff = -1;
            if constexpr (kConvV) {
                if (p.w_off && lane == 0) woff = p.w_off[it.r];
                woff = __shfl_sync(0xffffffffu, woff, 0);
            }
            if (lane == 0) {
                if (!mbar_wait(&bar[B_QEMPTY], (items & 1) ^ 1)) ok = false;
                else {
                    const int nslots = ntB > 0 ? 2 : 1;
                    uint64_t *qb = &bar[F8 ? B_QLAND : B_QFULL];
                    // a box counts in full, zero-filled rows past T included
                    mbar_arrive_expect_tx(qb, nslots * p.TT * p.G * (D * 2));
                    for (int sl = 0; sl < nslots; ++sl) {
                        const int tok0 = it.qstart + (it.mt * 2 + sl) * p.TT;
#pragma unroll
                        for (int h = 0; h < C::kHalves; ++h)
                            tma_load_3d(sQ + sl * C::kQBytes + h * (kBM * 128), &p.tmQ, qb, h * 64,
                                        it.g * p.G, tok0);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            for (int j = 0; ok && j < nt; ++j, ++t) {
                const int pg0 = j * kPagesPerTile;
                const int npg = min(kPagesPerTile, ctx_pages - pg0);
                int blk = 0;
                uint32_t wfl = 0;
                if (lane < npg) {
                    blk = row[pg0 + lane];
                    if (kConvV && woff >= 0)
                        wfl = p.w_flag[((long long)(woff / kPage) + pg0 + lane) * p.Hkv + it.g];
                    if (blk < 0 || blk >= p.NB) {
                        flag(p.status, PA_CHECK_BLOCK_ID);
                        blk = 0;
                    }
                }
                // V of this tile from the widened copy: one 128-token box
                // per 64-dim half (counted in full, rows past the request
                // included: the softmax zeroes keys past the context)
                const bool vw = kConvV && woff >= 0 && !__any_sync(0xffffffffu, wfl != 0);
                // K ring: two stages; V ring: kVSt
                const int kst = (int)(t & 1), vst = (int)(t % kVSt);
                const uint32_t kph = (uint32_t)((t >> 1) & 1), vph = (uint32_t)((t / kVSt) & 1);
                // FP8: one D-byte row per slot (head_dim 128: into the tile's
                // upper half; 64: into the staging area)
                const uint32_t bytes = F8 ? (uint32_t)npg * kPage * D
                                          : (uint32_t)npg * C::kHalves * C::kPageHalfBytes;
                const uint32_t vbytes = vw ? (uint32_t)C::kTileBytes : bytes;
#pragma unroll
                for (int kv = 0; kv < 2; ++kv) {
                    const int st = kv ? vst : kst;
                    uint64_t *fullb = &bar[(F8 ? (kv ? B_VLAND : B_KLAND)
                                               : (kv ? (kConvV ? B_VLAND : B_VFULL) : B_KFULL)) + st];
                    uint64_t *emptyb = &bar[(kv ? B_VEMPTY : B_KEMPTY) + st];
                    unsigned char *dst = (kv ? sV : sK) + st * C::kTileBytes;
                    if (lane == 0) {
                        if (!mbar_wait(emptyb, (kv ? vph : kph) ^ 1)) {
                            ok = false;
                        } else {
                            if (kConvV && kv) v_src[st] = vw ? 1 : 0;
                            mbar_arrive_expect_tx(fullb, kv ? vbytes : bytes);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (kConvV && kv && vw) {
                        if (lane == 0) {
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_load_3d(dst + h * C::kHalfBytes, &p.tmVw, fullb, h * 64, it.g,
                                            woff + pg0 * kPage);
                        }
                    } else if (lane < npg) {
                        if constexpr (F8) {
                            unsigned char *fdst =
                                D == 128 ? dst + C::kHalfBytes + lane * kPage * 128
                                         : sL + (kv * 2 + st) * C::kLandBytes + lane * kPage * 64;
                            tma_load_3d(fdst, kv ? &p.tmV : &p.tmK, fullb, 0, it.g, blk * kPage);
                        } else {
#pragma unroll
                            for (int h = 0; h < C::kHalves; ++h)
                                tma_load_3d(dst + h * C::kHalfBytes + lane * C::kPageHalfBytes,
                                            kv ? &p.tmV : &p.tmK, fullb, h * 64, it.g, blk * kPage);
                        }
                    }
                    if (kv) lastV = t; else lastK = t;
                }
            }
            if (*abort_flag) ok = false;
        }
        if (!ok) fail();
        // Drain: the last copies issued into each ring must have landed.
        if (lane == 0) {
            const int kf = F8 ? B_KLAND : B_KFULL, vf = kConv ? B_VLAND : B_VFULL;
            if (lastK >= 0) mbar_wait(&bar[kf + (int)(lastK & 1)], (uint32_t)((lastK >> 1) & 1));
            if (lastV >= 0) mbar_wait(&bar[vf + (int)(lastV % kVSt)], (uint32_t)((lastV / kVSt) & 1));
        }
    } else if (warp == 1) {
        // =================== MMA issuer ===================
        const uint32_t idQK = instr_desc<TQK>(kBM, kBN, 0);
        const uint32_t idPV = instr_desc<__half>(kBM, D, 1);
        const uint32_t idPVb = instr_desc<__nv_bfloat16>(kBM, D, 1);   // bf16 V halves
        long long t0 = 0;           // KV tiles of earlier items
        long long cnt[2] = {0, 0};  // tiles processed per slot (barrier phases)
        int its[2] = {0, 0};        // items processed per slot
        uint32_t nsplit[2] = {0, 0};   // P rewrites requested per slot
        int vst = 0;                   // V stage of the next tile (0 .. kVSt-1) and
        uint32_t vph = 0;              // its mbarrier phase, advanced per tile
        int items = 0;
        bool ok = true;
        for (int k = 0; ok; ++k, ++items) {
            const long long ik = item_at(k);
            if (ik < 0 || !walk.find(ik, lane, it)) break;
            int ns[2] = {slot_tiles(p, it, 0), slot_tiles(p, it, 1)};
            const int nt = max(ns[0], ns[1]);
            {
                // The whole warp runs this loop, converged, on warp-uniform
                // values; the MMA and commit wrappers issue from one lane.
                const uint32_t q0 = smem_u32(sQ);
                auto wait_or_fail = [&](uint64_t *b, uint32_t par) {
                    if (ok && !mbar_wait_warp(b, par)) ok = false;
                    return ok;
                };
                auto issue_qk = [&](int slot, int kst) {
                    const uint32_t qa = q0 + slot * C::kQBytes;
                    const uint32_t ka = smem_u32(sK + kst * C::kTileBytes);
                    const uint64_t dq0 = smem_desc_sw128(qa, 16, 1024);
                    const uint64_t dk0 = smem_desc_sw128(ka, 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                        const uint32_t koff = (kk >> 2) * C::kHalfBytes + (kk & 3) * 32;
                        // descriptors differ only in the start address (16-byte
                        // units, a 14-bit field that never carries here)
                        mma_ss(tmem + C::col_s(slot), dq0 + (off >> 4), dk0 + (koff >> 4), idQK,
                               kk > 0);
                    }
                    mma_commit(&bar[B_SFULL + slot]);
                };
                wait_or_fail(&bar[B_QFULL], items & 1);
                // tile 0: both slots' scores
                if (ok && wait_or_fail(&bar[B_KFULL + (int)(t0 & 1)], (uint32_t)((t0 >> 1) & 1))) {
                    tc_fence_after();
                    for (int sl = 0; sl < 2; ++sl)
                        if (ns[sl] > 0) issue_qk(sl, (int)(t0 & 1));
                    mma_commit(&bar[B_KEMPTY + (int)(t0 & 1)]);
                    if (nt == 1) mma_commit(&bar[B_QEMPTY]);
                }
                for (int j = 0; ok && j < nt; ++j) {
                    const long long t = t0 + j;
                    const int st = vst;            // V stage of tile t (t % kVSt)
                    const uint32_t ph = vph;       // (t / kVSt) & 1
                    if (++vst == kVSt) {
                        vst = 0;
                        vph ^= 1u;
                    }
                    const long long t1 = t + 1;
                    // This tile's V is waited for before the tile's first P (it
                    // is normally in long before it), so the PV issues as soon
                    // as P is; the next tile's K only before the first QK that
                    // reads it (over FP8 pools it may still be being widened).
                    if (!wait_or_fail(&bar[B_VFULL + st], ph)) break;
                    int bfh = 0;   // bf16 pools: key halves of this V tile that stayed bf16
                    if constexpr (kConvV) bfh = v_fmt[2 * st] | (v_fmt[2 * st + 1] << 1);
                    bool k_next_ready = false;
                    for (int sl = 0; ok && sl < 2; ++sl) {
                        if (j >= ns[sl]) continue;
                        if (!wait_or_fail(&bar[B_PFULL + sl], (uint32_t)(cnt[sl] & 1))) break;
                        if (j == 0 && !wait_or_fail(&bar[B_OFREE + sl], (uint32_t)((its[sl] & 1) ^ 1)))
                            break;
                        tc_fence_after();
                        const uint64_t dv0 = smem_desc_sw128(smem_u32(sV + st * C::kTileBytes),
                                                             C::kHalfBytes, 1024);
                        if (kConvV && bfh) {
                            // rare: a key half stayed bf16 (out of line)
                            if (!pv_with_bf16_halves(bar + B_SPLITREQ + sl, bar + B_SPLITDONE + sl,
                                                     split_fmt + sl, bfh, &nsplit[sl],
                                                     tmem + C::col_o(sl), tmem + C::col_s(sl), dv0,
                                                     idPV, idPVb, j > 0)) {
                                ok = false;
                                break;
                            }
                        } else {
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; ++kk)
                                mma_ts(tmem + C::col_o(sl),
                                       tmem + C::col_s(sl) + (kk >> 2) * 64 + (kk & 3) * 8,
                                       dv0 + (uint64_t)(kk * 2048 >> 4), idPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        // O_X is read only by the epilogue, after the item's last
                        // PV; a rescale before that is ordered by S_FULL, whose
                        // commit covers every earlier MMA of this thread.
                        if (j + 1 == ns[sl]) mma_commit(&bar[B_ODONE + sl]);
                        ++cnt[sl];
                        if (j + 1 < ns[sl]) {
                            if (!k_next_ready &&
                                !wait_or_fail(&bar[B_KFULL + (int)(t1 & 1)], (uint32_t)((t1 >> 1) & 1)))
                                break;
                            k_next_ready = true;
                            tc_fence_after();
                            issue_qk(sl, (int)(t1 & 1));
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bar[B_VEMPTY + st]);
                    if (k_next_ready) {
                        mma_commit(&bar[B_KEMPTY + (int)(t1 & 1)]);
                        if (j + 1 == nt - 1) mma_commit(&bar[B_QEMPTY]);
                    }
                    if (*abort_flag) ok = false;
                }
            }
            for (int sl = 0; sl < 2; ++sl)
                if (ns[sl] > 0) ++its[sl];
            t0 += nt;
        }
        if (!ok && lane == 0) fail();
        // Every MMA issued must be complete before TMEM is released.
        mma_commit(&bar[B_DRAIN]);
        mbar_wait_warp(&bar[B_DRAIN], 0);
    } else if (warp >= 2 + kSoftmaxWarps) {
        // =================== converters (warps 10, 11) ===================
        if constexpr (kConvV) {
            // bf16 pools: each landed V tile to f16, warp cw taking keys
            // 64 cw .. 64 cw + 63; the format of each half for the softmax
            // and MMA warps, then V full.
            const int cw = warp - (2 + kSoftmaxWarps);
            long long t = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const long long ik = item_at(k);
                if (ik < 0 || !walk.find(ik, lane, it)) break;
                const int nt = max(slot_tiles(p, it, 0), slot_tiles(p, it, 1));
                for (int j = 0; ok && j < nt; ++j, ++t) {
                    const int st = (int)(t % kVSt);
                    if (!mbar_wait_warp(&bar[B_VLAND + st], (uint32_t)((t / kVSt) & 1))) {
                        ok = false;
                        break;
                    }
                    const int valid = min(kBN, it.L - j * kBN) - 64 * cw;   // keys inside the context
                    const int f = v_src[st] ? 0
                                            : v_half_to_f16<C::kHalves>(sV + st * C::kTileBytes + cw * 64 * 128,
                                                                        C::kHalfBytes, valid, lane);
                    if (lane == 0) v_fmt[2 * st + cw] = f;
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[B_VFULL + st]);
                }
                if (*abort_flag) ok = false;
            }
            if (!ok) fail();
        }
        // FP8 pools: widen landed Q, K and V tiles to f16 (K and V rings of
        // two stages each, same index)
        static_assert(!F8 || kVSt == 2, "FP8 pools use a two-stage V ring");
        if constexpr (F8) {
            const int cw = warp - (2 + kSoftmaxWarps);   // rows 64 cw .. 64 cw + 63 of each tile
            long long t = 0;
            int items = 0;
            bool ok = true;
            for (int k = 0; ok; ++k, ++items) {
                const long long ik = item_at(k);
                if (ik < 0 || !walk.find(ik, lane, it)) break;
                const int ntB = slot_tiles(p, it, 1);
                const int nt = max(slot_tiles(p, it, 0), ntB);
                if (!mbar_wait_warp(&bar[B_QLAND], items & 1)) {
                    ok = false;
                    break;
                }
                if constexpr (std::is_same<T, __nv_bfloat16>::value) {
                    const int nslots = ntB > 0 ? 2 : 1;
                    bf16_tile_to_f16(sQ, nslots * C::kQBytes, cw * 32 + lane, kConvWarps * 32);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_QFULL]);
                for (int j = 0; ok && j < nt; ++j, ++t) {
                    const int st = (int)(t & 1);
                    const uint32_t ph = (uint32_t)((t >> 1) & 1);
#pragma unroll
                    for (int kv = 0; kv < 2; ++kv) {
                        if (!mbar_wait_warp(&bar[(kv ? B_VLAND : B_KLAND) + st], ph)) {
                            ok = false;
                            break;
                        }
                        if constexpr (D == 128)
                            widen_e4m3_tile((kv ? sV : sK) + st * C::kTileBytes, C::kHalfBytes, cw * 64,
                                            cw * 64 + 64, lane);
                        else
                            widen_e4m3_rows64(sL + (kv * 2 + st) * C::kLandBytes,
                                              (kv ? sV : sK) + st * C::kTileBytes, cw * 64, cw * 64 + 64,
                                              lane);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[(kv ? B_VFULL : B_KFULL) + st]);
                    }
                }
                if (*abort_flag) ok = false;
            }
            if (!ok) fail();
        }
    } else {
        // =================== softmax + epilogue (warps 2..9) ===================
        const int slot = (warp - 2) >> 2;          // 0 = A, 1 = B
        const int sub = warp & 3;                  // TMEM sub-partition of this warp
        const int row = sub * 32 + lane;           // tile row = TMEM lane
        const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
        const uint32_t colS = tmem + lane_addr + C::col_s(slot);
        const uint32_t colO = tmem + lane_addr + C::col_o(slot);
        const float ks = (F8 && p.k_scale) ? *p.k_scale : 1.f;
        const float vs = (F8 && p.v_scale) ? *p.v_scale : 1.f;
        const float2 c2 = make_float2(p.qscale * ks, p.qscale * ks);
        long long cnt = 0;   // tiles this slot processed (barrier phases)
        long long t0 = 0;    // KV tiles of earlier items (V ring phases)
        int items_done = 0;  // items this slot finished (O_DONE phases)
        // Wait for a phase of `b`, meanwhile serving the MMA warp's requests
        // (bf16 pools, rare): a key half whose V stayed bf16 (it holds a value
        // f16 cannot) needs the last tile's f16 P rewritten as two bf16 terms
        // hi and lo (an f16 value's 11 significant bits split exactly into
        // 8 + 3).  The request comes after this slot's P full and before the
        // MMA warp issues that tile's PV and the next QK, which is when these
        // warps wait here.  Bounded like every wait.
        uint32_t split_ph = 0;
        auto wait_serving = [&](uint64_t *b, uint32_t par) -> bool {
            if constexpr (!kConvV) {
                return mbar_wait_warp(b, par);
            } else {
                uint64_t start = 0;
                for (;;) {
                    // a suspending wait: the warp takes no issue slots while
                    // it waits (a pending request shows when it returns
                    // without the phase)
                    if (__all_sync(0xffffffffu, mbar_try_wait(b, par))) return true;
                    if (__all_sync(0xffffffffu, mbar_test(&bar[B_SPLITREQ + slot], split_ph))) {
                        tc_fence_after();
                        split_p_halves(colS, split_fmt[slot]);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[B_SPLITDONE + slot]);
                        split_ph ^= 1;
                        continue;
                    }
                    const uint64_t now = globaltimer_ns();
                    if (!start) start = now;
                    else if (now - start > kWaitLimitNs) return false;
                }
            }
        };
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const long long ik = item_at(k);
            if (ik < 0 || !walk.find(ik, lane, it)) break;
            const int ntS = slot_tiles(p, it, slot);
            const int nt = max(slot_tiles(p, it, 0), slot_tiles(p, it, 1));
            if (ntS == 0) {
                t0 += nt;
                continue;
            }
            const int tl = (it.mt * 2 + slot) * p.TT + row / p.G;   // token in the request
            const bool valid = row < p.TT * p.G && tl < it.n;
            // The last key this row sees.  A row that is never written out (the
            // empty rows of a tile whose G does not divide 128, or tokens past
            // the request) sees every key: with -1 it would take the masking
            // path on every tile and hold the slot's P back (28/4 heads:
            // 345 -> 275 us on a 5000-token chunk).  Its values stay in its own row.
            const int pos = valid ? it.L - it.n + tl : INT_MAX / 2;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < ntS; ++j, ++cnt) {
                if (!wait_serving(&bar[B_SFULL + slot], (uint32_t)(cnt & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int key0 = j * kBN;
                const bool full_tile = key0 + kBN - 1 <= pos;
                if constexpr (!F8) {
                    // One TMEM pass, 64 columns at a time: the half's row max (scale
                    // > 0 keeps the argmax), then P = exp2(s*c - m_ref) in packed
                    // f16 pairs written over the scores already read (64 keys ->
                    // columns 64hh..64hh+31).  The reference max moves lazily:
                    // only when a half's max passes it by more than 2^8, so P stays
                    // below 256.  Sums and O accumulated against an older reference
                    // are scaled down when it moves: the tile's first half in
                    // TMEM (rare: only when the second half moves it again), the
                    // tile's partial sum, and O and l of earlier tiles once per
                    // tile.  A row with no visible key is never written out, so
                    // any NaN stays in its own row.
                    const float m_prev = m_ref;
                    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[64];
                        tmem_ld32(colS + hh * 64, *reinterpret_cast<uint32_t (*)[32]>(r));
                        tmem_ld32(colS + hh * 64 + 32, *reinterpret_cast<uint32_t (*)[32]>(r + 32));
                        tmem_wait_ld();
                        if (!full_tile) {
    #pragma unroll
                            for (int k = 0; k < 64; ++k)
                                if (key0 + hh * 64 + k > pos) r[k] = 0xff800000u;
                        }
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    #pragma unroll
                        for (int k = 0; k < 64; k += 2)
                            m4[(k >> 1) & 3] = fmaxf(m4[(k >> 1) & 3],
                                                     fmaxf(__uint_as_float(r[k]), __uint_as_float(r[k + 1])));
                        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2.x;
                        const bool need = mx > m_ref + kRescaleThreshold;
                        if (need) {
                            const float alpha = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - mx);
                            acc[0].x *= alpha;
                            acc[0].y *= alpha;
                            acc[1].x *= alpha;
                            acc[1].y *= alpha;
                        }
                        if (hh == 1 && __any_sync(0xffffffffu, need)) {
                            // the first half's P was written against the old reference
                            // (its store completes first)
                            const float alpha = need ? fast_exp2(m_ref - mx) : 1.f;
                            tmem_wait_st();
                            uint32_t w[32];
                            tmem_ld32(colS, w);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                float a, b;
                                Elt<__half>::unpack2(w[e], a, b);
                                w[e] = Elt<__half>::pack2(a * alpha, b * alpha);
                            }
                            tmem_st32(colS, w);
                        }
                        if (need) m_ref = mx;
                        const float2 mneg = make_float2(-m_ref, -m_ref);
                        uint32_t w[32];
    #pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float2 y = __ffma2_rn(make_float2(__uint_as_float(r[2 * e]),
                                                              __uint_as_float(r[2 * e + 1])), c2, mneg);
                            y.x = fast_exp2(y.x);
                            y.y = fast_exp2(y.y);
                            acc[e & 1] = __fadd2_rn(acc[e & 1], y);
                            w[e] = Elt<__half>::pack2(y.x, y.y);
                        }
                        tmem_st32(colS + hh * 64, w);
                    }
                    if (j > 0 && __any_sync(0xffffffffu, m_ref != m_prev)) {
                        // O holds PV of tiles < j, all complete: S_j's commit (waited
                        // above) covers every MMA issued before it.  Rescale.
                        const float alpha = m_ref != m_prev ? fast_exp2(m_prev - m_ref) : 1.f;
    #pragma unroll
                        for (int cc = 0; cc < D; cc += 32) {
                            uint32_t o[32];
                            tmem_ld32(colO + cc, o);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(colO + cc, o);
                        }
                        l *= alpha;
                    }
                    tmem_wait_st();
                    l += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                } else {
                    // FP8 pools: two passes over the scores (row max, then P).
                    // The one-pass form above measured slower here when scores
                    // spread widely (427 against 378 us on the mixed step's
                    // chunk over unscaled pools).
                    // Pass 1: row max of the raw scores (scale > 0 keeps the
                    // argmax), 64 columns per TMEM round trip, four chains.
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[64];
                        tmem_ld32(colS + hh * 64, *reinterpret_cast<uint32_t (*)[32]>(r));
                        tmem_ld32(colS + hh * 64 + 32, *reinterpret_cast<uint32_t (*)[32]>(r + 32));
                        tmem_wait_ld();
                        if (!full_tile) {
    #pragma unroll
                            for (int k = 0; k < 64; ++k)
                                if (key0 + hh * 64 + k > pos) r[k] = 0xff800000u;
                        }
    #pragma unroll
                        for (int k = 0; k < 64; k += 2)
                            m4[(k >> 1) & 3] = fmaxf(m4[(k >> 1) & 3],
                                                     fmaxf(__uint_as_float(r[k]), __uint_as_float(r[k + 1])));
                    }
                    const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2.x;
                    const bool need = mx > m_ref + kRescaleThreshold;
                    if (j > 0 && __any_sync(0xffffffffu, need)) {
                        // O holds PV of tiles < j, all complete: S_j's commit (waited
                        // above) covers every MMA issued before it.  Rescale.
                        const float alpha = need ? fast_exp2(m_ref - mx) : 1.f;
    #pragma unroll
                        for (int cc = 0; cc < D; cc += 32) {
                            uint32_t o[32];
                            tmem_ld32(colO + cc, o);
                            tmem_wait_ld();
    #pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(colO + cc, o);
                        }
                        tmem_wait_st();
                        if (need) l *= alpha;
                    }
                    if (need) m_ref = mx;
                    // Pass 2: P = exp2(s*c - m_ref) in packed f16 pairs, written
                    // over the scores already read (64 keys -> columns 64hh..64hh+31).
                    // A row with no visible key is never written out, so any NaN
                    // stays in its own row.
                    const float2 mneg = make_float2(-m_ref, -m_ref);
                    float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    #pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t r[64];
                        tmem_ld32(colS + hh * 64, *reinterpret_cast<uint32_t (*)[32]>(r));
                        tmem_ld32(colS + hh * 64 + 32, *reinterpret_cast<uint32_t (*)[32]>(r + 32));
                        tmem_wait_ld();
                        if (!full_tile) {
    #pragma unroll
                            for (int k = 0; k < 64; ++k)
                                if (key0 + hh * 64 + k > pos) r[k] = 0xff800000u;
                        }
                        uint32_t w[32];
    #pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float2 y = __ffma2_rn(make_float2(__uint_as_float(r[2 * e]),
                                                              __uint_as_float(r[2 * e + 1])), c2, mneg);
                            y.x = fast_exp2(y.x);
                            y.y = fast_exp2(y.y);
                            acc[e & 1] = __fadd2_rn(acc[e & 1], y);
                            w[e] = Elt<__half>::pack2(y.x, y.y);
                        }
                        tmem_st32(colS + hh * 64, w);
                    }
                    tmem_wait_st();
                    l += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                }
                if (j == ntS - 1 && ntS == nt && it.L < key0 + kBN) {
                    // Keys past the context in the item's last tile: their V
                    // rows hold stale data (or nothing was loaded); make them
                    // zero so 0 * V stays 0 in the tensor core.  The slot's
                    // four warps reach the barrier even if the wait timed out.
                    const long long tv = t0 + j;
                    const bool landed = mbar_wait_warp(&bar[B_VFULL + (int)(tv % kVSt)],
                                                       (uint32_t)((tv / kVSt) & 1));
                    if (landed) {
                        unsigned char *vt = sV + (int)(tv % kVSt) * C::kTileBytes;
                        const int first = it.L - key0;
                        const int rows = kBN - first;
                        for (int xx = row; xx < rows * C::kHalves * 8; xx += kBM) {
                            const int h = xx / (rows * 8), rem = xx % (rows * 8);
                            *reinterpret_cast<uint4 *>(vt + h * C::kHalfBytes +
                                                       (first + rem / 8) * 128 + (rem % 8) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                    named_bar_sync(1 + slot, kBM);
                    if (!landed) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_PFULL + slot]);
            }
            if (!ok) break;
            // ---- epilogue: O / l for this row (O_DONE: once per item and slot)
            if (!wait_serving(&bar[B_ODONE + slot], (uint32_t)(items_done & 1))) {
                ok = false;
                break;
            }
            ++items_done;
            tc_fence_after();
            const float inv = l > 0.f ? vs / l : 0.f;
            T *dst = reinterpret_cast<T *>(p.out) +
                     ((long long)(it.qstart + tl) * p.Hq + it.g * p.G + row % p.G) * D;
#pragma unroll
            for (int cc = 0; cc < D; cc += 32) {
                uint32_t r[32];
                tmem_ld32(colO + cc, r);
                tmem_wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = Elt<T>::pack2(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv);
                        v.y = Elt<T>::pack2(__uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv);
                        v.z = Elt<T>::pack2(__uint_as_float(r[e + 4]) * inv, __uint_as_float(r[e + 5]) * inv);
                        v.w = Elt<T>::pack2(__uint_as_float(r[e + 6]) * inv, __uint_as_float(r[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + cc + e) = v;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OFREE + slot]);
            t0 += nt;
            if (*abort_flag) ok = false;
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// 3-D TMA map, 128-byte swizzle, 128-byte inner box: q as [T][Hq][D] with a
// {64, G, floor(128/G)} box, or a pool as [NB*bs][Hkv][D] with a {64, 1, 16}
// box (16-bit) or {128, 1, 16} (FP8, head_dim 128).  plain_rows: an FP8 pool
// at head_dim 64, whole 64-byte rows in a {64, 1, 16} box, no swizzle.
bool encode_sw128(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                  uint32_t b1, uint32_t b2, int elt = 2, bool plain_rows = false) {
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    if (!enc) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return false;
        enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * elt, d0 * d1 * elt};
    const cuuint32_t box[3] = {plain_rows ? (cuuint32_t)d0 : 128u / (cuuint32_t)elt, b1, b2};
    const cuuint32_t es[3] = {1u, 1u, 1u};
    return enc(map, elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 3,
               const_cast<void *>(ptr), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               plain_rows ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D, bool F8>
pa_status launch_typed(const Params &prm, long long items, long long max_ctas, bool pdl,
                       cudaStream_t stream) {
    using C = Cfg<D>;
    constexpr int kSmem = (F8 && D == 64) ? C::kSmemF8Land : C::smem(Conv<T, F8>::kV ? 3 : 2);
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static bool configured[64] = {};
    int dev = 0;
    PA_TRY_CUDA(cudaGetDevice(&dev));
    if (dev >= 64 || !configured[dev]) {
        PA_TRY_CUDA(cudaFuncSetAttribute(paged_prefill_kernel<T, D, F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
        if (dev < 64) configured[dev] = true;
    }
    long long grid = max_ctas;
    if (items < grid) grid = items;
    if (grid < 1) return PA_OK;
    if (pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(threads_for(Conv<T, F8>::kAny));
        cfg.dynamicSmemBytes = kSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        PA_TRY_CUDA(cudaLaunchKernelEx(&cfg, paged_prefill_kernel<T, D, F8>, prm));
    } else {
        paged_prefill_kernel<T, D, F8><<<(int)grid, threads_for(Conv<T, F8>::kAny), kSmem, stream>>>(prm);
        PA_TRY_CUDA(cudaGetLastError());
    }
    note_launch();
    return PA_OK;
}

// One launch of the instantiation for these pools and head size.
pa_status launch_kind(const AttnArgs &a, const Params &prm, long long items, long long max_ctas,
                      bool pdl, cudaStream_t stream) {
    const bool f8 = a.cache_dtype == PA_FP8_E4M3;
    const bool bf16 = a.dtype == PA_BF16;
    if (f8 && a.D == 128)
        return bf16 ? launch_typed<__nv_bfloat16, 128, true>(prm, items, max_ctas, pdl, stream)
                    : launch_typed<__half, 128, true>(prm, items, max_ctas, pdl, stream);
    if (f8)
        return bf16 ? launch_typed<__nv_bfloat16, 64, true>(prm, items, max_ctas, pdl, stream)
                    : launch_typed<__half, 64, true>(prm, items, max_ctas, pdl, stream);
    if (a.D == 128)
        return bf16 ? launch_typed<__nv_bfloat16, 128, false>(prm, items, max_ctas, pdl, stream)
                    : launch_typed<__half, 128, false>(prm, items, max_ctas, pdl, stream);
    return bf16 ? launch_typed<__nv_bfloat16, 64, false>(prm, items, max_ctas, pdl, stream)
                : launch_typed<__half, 64, false>(prm, items, max_ctas, pdl, stream);
}

// ---------------------------------------------------------------------------
// bf16 pools: V of the prefill requests widened to f16 once per call
// ---------------------------------------------------------------------------
// PV runs in f16 (P as f16 keeps 11 significant bits), so a bf16 V tile must
// be converted before the tensor core reads it.  Converted inside the kernel,
// every item of a (request, kv head) -- one per pair of 128-row tiles --
// converts the same tiles again; here each page is converted once into a
// token-major copy in the workspace, [token][kv head][dim] like a pool, for
// the requests the prefill kernel takes (more than tau query tokens), in
// request order while the copy has room.  A page holding a value f16 cannot
// represent (|v| > 65280, or not finite) is flagged and its tiles take the
// in-kernel route, which keeps such halves bf16.  Only at head_dim 128: at
// 64 the softmax, not the conversion, bounds the kernel, and the extra pass
// measured slower (bf16 chunk, 32/8 heads: 284 -> 290 us; 16/16: 174 -> 186).
struct WidenParams {
    const __nv_bfloat16 *vc;   // V pool [NB*bs][Hkv][D]
    const int32_t *bt, *qsl, *seq_lens;
    int32_t *w_off;            // [R] out: first token of request r in the copy, or -1
    uint8_t *w_flag;           // [pages_cap][Hkv] out
    __half *w_data;            // [pages_cap*16][Hkv][D]
    int R, MB, NB, Hkv, D, tau, pages_cap;
};
constexpr int kWidenThreads = 256;
constexpr int kWidenMaxReqs = 8192;   // the prefix over requests is kept in shared memory
constexpr size_t kWidenCapBytes = (size_t)64 << 20;   // widened copy: at most 64 MiB

template <int D>
__global__ void __launch_bounds__(kWidenThreads, 4) widen_v_kernel(const WidenParams w) {
    extern __shared__ int32_t s_first[];   // [R + 1]: first page of each request in the copy
    __shared__ int s_scan[33];
    const int tid = threadIdx.x, lane = tid & 31, nthreads = blockDim.x;
    auto pages_of = [&](int r) -> int {
        const int n = w.qsl[r + 1] - w.qsl[r];
        const int L = w.seq_lens[r];
        return (n > w.tau && L > 0) ? (L + kPage - 1) / kPage : 0;
    };
    const int per = (w.R + nthreads - 1) / nthreads;
    const int r0 = min(w.R, tid * per), r1 = min(w.R, r0 + per);
    int local = 0;
    for (int r = r0; r < r1; ++r) local += pages_of(r);
    int total = 0;
    int run = block_exclusive_scan(local, s_scan, total);
    for (int r = r0; r < r1; ++r) {
        s_first[r] = run;
        run += pages_of(r);
    }
    if (tid == 0) s_first[w.R] = total;
    __syncthreads();
    // A request is widened when all its pages fit (the prefix is monotone,
    // so the widened requests are a leading run of the prefill requests).
    if (blockIdx.x == 0)
        for (int r = tid; r < w.R; r += nthreads) {
            const bool has = s_first[r + 1] > s_first[r];
            w.w_off[r] = (has && s_first[r + 1] <= w.pages_cap) ? s_first[r] * kPage : -1;
        }
    // One warp per (page of the copy, kv head): 16 rows of D values, every
    // 16-byte unit of them loaded before any is converted (one memory round
    // trip per page, not one per unit).
    constexpr int upr = D / 8;                   // 16-byte units per row
    constexpr int kPer = kPage * upr / 32;       // units per lane
    const long long units = (long long)min(total, w.pages_cap) * w.Hkv;
    const long long nw = (long long)gridDim.x * (nthreads / 32);
    for (long long u = (long long)blockIdx.x * (nthreads / 32) + (tid >> 5); u < units; u += nw) {
        const int pgc = (int)(u / w.Hkv), h = (int)(u % w.Hkv);
        // the request holding copy page pgc: the last r with s_first[r] <= pgc
        int lo = 0, hi = w.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_first[mid] <= pgc) lo = mid;
            else hi = mid - 1;
        }
        const int r = lo;
        if (s_first[r + 1] > w.pages_cap) continue;   // the request does not fit
        const int pg = pgc - s_first[r];
        const int L = w.seq_lens[r];
        const int blk = w.bt[(long long)r * w.MB + pg];
        // a bad block id: flagged, so the kernel reads (and checks) the pool
        uint32_t fl = (blk < 0 || blk >= w.NB) ? 0x8000u : 0u;
        if (!fl) {
            uint4 vin[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int x = lane + 32 * k, i = x / upr, c = x % upr;
                vin[k] = __ldg(reinterpret_cast<const uint4 *>(
                    w.vc + ((long long)(blk * kPage + i) * w.Hkv + h) * D + c * 8));
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int x = lane + 32 * k, i = x / upr, c = x % upr;
                const uint4 v = vin[k];
                if (pg * kPage + i < L) {
                    // magnitude above 0x477F (65280) sets bit 15 of (m + 0x3880)
                    fl |= (v.x & 0x7fff7fffu) + 0x38803880u;
                    fl |= (v.y & 0x7fff7fffu) + 0x38803880u;
                    fl |= (v.z & 0x7fff7fffu) + 0x38803880u;
                    fl |= (v.w & 0x7fff7fffu) + 0x38803880u;
                }
                uint4 o;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(&v);
                uint32_t *dst = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __half2 hv = __floats2half2_rn(__uint_as_float(src[e] << 16),
                                                   __uint_as_float(src[e] & 0xffff0000u));
                    dst[e] = *reinterpret_cast<uint32_t *>(&hv);
                }
                *reinterpret_cast<uint4 *>(w.w_data + ((long long)(pgc * kPage + i) * w.Hkv + h) * D +
                                           c * 8) = o;
            }
        }
        fl = __reduce_or_sync(0xffffffffu, fl & 0x80008000u);
        if (lane == 0) w.w_flag[(long long)pgc * w.Hkv + h] = fl ? 1 : 0;
    }
}

}  // namespace prefill

size_t prefill_widen_size(int32_t R, int32_t T, int32_t max_q, int32_t max_seq, int32_t Hkv,
                          int32_t D) {
    using namespace prefill;
    if (max_q <= kTauDefault || R <= 0 || R > kWidenMaxReqs || Hkv <= 0 || D != 128) return 0;
    const long long reqs = min((long long)R, (long long)T / (kTauDefault + 1));
    if (reqs <= 0) return 0;
    const long long per_page = (long long)Hkv * (kPage * D * 2 + 1);
    long long pages = reqs * (((long long)max_seq + kPage - 1) / kPage);
    const long long cap = (long long)(kWidenCapBytes / (size_t)per_page);
    if (pages > cap) pages = cap;
    auto up = [](long long x) { return (x + 255) / 256 * 256; };
    return (size_t)(up((long long)R * 4) + up(pages * Hkv) + pages * kPage * Hkv * D * 2);
}

int prefill_tau(const AttnArgs &a) {
    const int G = a.Hq / a.Hkv;
    // The tensor-core kernel takes the row max of unscaled scores: scale > 0.
    if ((a.D != 64 && a.D != 128) || G < 1 || G > prefill::kBM || !(a.scale > 0.f)) return INT_MAX;
    return prefill::kTauDefault;
}

namespace prefill {

// The kernel's parameters for this call (tensor maps, the widened V when
// bf16 pools at head_dim 128 leave room for it in the workspace: its pass is
// launched here) and an upper bound on the work items.
static pa_status build(const AttnArgs &a, int tau, cudaStream_t stream, Params &prm,
                       long long &items) {
    memset(&prm, 0, sizeof prm);
    const int G = a.Hq / a.Hkv;
    const uint64_t slots = (uint64_t)a.NB * a.bs;
    const bool f8 = a.cache_dtype == PA_FP8_E4M3;
    const int elt = f8 ? 1 : 2;
    const int TT = kBM / G;
    if (!encode_sw128(&prm.tmQ, a.q, a.D, a.Hq, a.T, G, TT) ||
        !encode_sw128(&prm.tmK, a.kc, a.D, a.Hkv, slots, 1, kPage, elt, f8 && a.D == 64) ||
        !encode_sw128(&prm.tmV, a.vc, a.D, a.Hkv, slots, 1, kPage, elt, f8 && a.D == 64))
        return PA_ERR_CUDA;
    prm.k_scale = a.k_scale;
    prm.v_scale = a.v_scale;
    // items in order as CTAs free up (the caller zeroed the counter)
    prm.item_counter = a.ctrl ? a.ctrl + kCtrlPrefillCounter : nullptr;
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
    prm.G = G;
    prm.TT = TT;
    prm.tau = tau;
    prm.qscale = a.scale * 1.4426950408889634f;
    prm.status = status_word();
    if (!prm.status) return PA_ERR_CUDA;
    // upper bound on the row tiles
    items = (long long)a.Hkv * ((long long)a.R + ((long long)a.T + 2 * TT - 1) / (2 * TT));
    const bool bf16 = a.dtype == PA_BF16;
    // bf16 pools: the prefill requests' V widened once, into the workspace's
    // tail: [R] first tokens, then [pages][Hkv] flags, then the f16 rows.
    if (bf16 && !f8 && a.D == 128 && a.pf_ws && a.R <= kWidenMaxReqs) {
        auto up = [](size_t x) { return (x + 255) / 256 * 256; };
        const size_t off_bytes = up((size_t)a.R * 4);
        const size_t row_bytes = (size_t)a.Hkv * a.D * 2;   // one token, every kv head
        long long pages = a.pf_bytes > off_bytes
                              ? (long long)((a.pf_bytes - off_bytes) / (kPage * row_bytes + a.Hkv))
                              : 0;
        if (pages > INT32_MAX / (4 * kPage)) pages = INT32_MAX / (4 * kPage);
        while (pages > 0 && off_bytes + up((size_t)pages * a.Hkv) + (size_t)pages * kPage * row_bytes >
                                a.pf_bytes)
            --pages;
        if (pages > 0) {
            unsigned char *base = static_cast<unsigned char *>(a.pf_ws);
            WidenParams w;
            w.vc = static_cast<const __nv_bfloat16 *>(a.vc);
            w.bt = a.bt;
            w.qsl = a.qsl;
            w.seq_lens = a.seq_lens;
            w.w_off = reinterpret_cast<int32_t *>(base);
            w.w_flag = base + off_bytes;
            w.w_data = reinterpret_cast<__half *>(base + off_bytes + up((size_t)pages * a.Hkv));
            w.R = a.R;
            w.MB = a.MB;
            w.NB = a.NB;
            w.Hkv = a.Hkv;
            w.D = a.D;
            w.tau = tau;
            w.pages_cap = (int)pages;
            if (!encode_sw128(&prm.tmVw, w.w_data, a.D, a.Hkv, (uint64_t)pages * kPage, 1, kBN))
                return PA_ERR_CUDA;
            widen_v_kernel<128><<<4 * num_sms(), kWidenThreads, (size_t)(a.R + 1) * sizeof(int32_t),
                                  stream>>>(w);
            PA_TRY_CUDA(cudaGetLastError());
            note_launch();
            prm.w_off = w.w_off;
            prm.w_flag = w.w_flag;
        }
    }
    return PA_OK;
}

}  // namespace prefill

pa_status launch_prefill(const AttnArgs &a, int tau, cudaStream_t stream) {
    using namespace prefill;
    if (tau == INT_MAX || a.max_q <= tau) return PA_OK;
    Params prm;
    long long items = 0;
    const pa_status st = build(a, tau, stream, prm, items);
    if (st != PA_OK) return st;
    return launch_kind(a, prm, items, num_sms(), false, stream);
}

// HBM-bound split-K work and tensor-bound prefill work side by side.  The
// split-K kernel keeps ~96% of its bandwidth on 120 of the 152 SMs and ~80%
// on 100, so the tensor-core kernel's first grid takes two fifths of the
// SMs from the start; the split-K grid (a programmatic dependent: it may start
// at once) fills the rest, and its CTAs that do not fit wait for SMs to free
// up.  A second tensor-core grid, a programmatic dependent of the split-K
// grid, takes the remaining prefill items from the same counter as SMs free
// up.  Items go to CTAs as they free up in both grids, so every item is
// computed once, by one CTA, with the same result as in a single grid.  The
// merge pass comes last as an ordinary launch: it starts once every grid
// before it has finished, so no CTA of it sits on an SM waiting.
pa_status launch_attention_overlapped(const AttnArgs &a, int tau, cudaStream_t stream) {
    using namespace prefill;
    Params prm;
    long long items = 0;
    pa_status st = build(a, tau, stream, prm, items);
    if (st != PA_OK) return st;
    // 60 of 152 SMs: measured against 30-76 on the mixed steps (5000-token
    // chunk + 200 decodes at 32/8 and 28/4 heads, and over FP8 pools)
    const long long first = num_sms() * 2 / 5 > 0 ? num_sms() * 2 / 5 : 1;
    st = launch_kind(a, prm, items, first, false, stream);
    if (st != PA_OK) return st;
    AttnArgs b = a;
    b.pdl = true;
    b.decode_part = 1;
    st = launch_decode(b, tau, stream);
    if (st != PA_OK) return st;
    if (items > first) {
        st = launch_kind(a, prm, items - first, num_sms(), true, stream);
        if (st != PA_OK) return st;
    }
    b.pdl = false;
    b.decode_part = 2;
    return launch_decode(b, tau, stream);
}

}  // namespace pa
