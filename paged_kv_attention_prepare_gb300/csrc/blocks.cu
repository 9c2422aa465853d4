// Whole-block operations on the two cache pools:
//   copy  -- copy-on-write ("How vLLM Works Internally", section
//            "Copy-on-Write for Beam Search", step 3): block dst[i] of each
//            pool becomes a copy of block src[i];
//   zero  -- new-block zeroing ("Inside vLLM: Following One Request", the
//            scheduler output's new_block_ids_to_zero): every byte of the
//            listed blocks, in both pools, becomes 0 before the forward pass.
//
// Both are HBM streams.  A block of one pool is block_bytes contiguous bytes
// (block_size * num_kv_heads * head_dim * element size, a multiple of 16), so
// the work is cut into jobs of (pair, pool, 16 KiB chunk); a CTA of 256
// threads moves one chunk with four independent 16-byte loads in flight per
// thread, then four 16-byte stores.  The grid strides over the jobs and is
// capped at a multiple of the SM count.  Block ids outside the pool are
// flagged (PA_CHECK_BLOCK_ID) and their pair skipped.
#include "pa_internal.cuh"

namespace pa {

constexpr int kBlkThreads = 256;
constexpr int kBlkVecs = 4;                                    // 16-byte vectors per thread
constexpr int64_t kChunkBytes = (int64_t)kBlkThreads * kBlkVecs * 16;  // 16 KiB

__global__ void __launch_bounds__(kBlkThreads)
copy_blocks_kernel(uint8_t *__restrict__ kc, uint8_t *__restrict__ vc, int64_t block_bytes,
                   int32_t num_blocks, const int32_t *__restrict__ src,
                   const int32_t *__restrict__ dst, int32_t n, int64_t chunks,
                   unsigned int *status) {
    const int64_t jobs = (int64_t)n * 2 * chunks;
    for (int64_t job = blockIdx.x; job < jobs; job += gridDim.x) {
        const int64_t pair = job / (2 * chunks);
        const int pool = (int)((job / chunks) & 1);
        const int64_t chunk = job % chunks;
        const int32_t s = src[pair], d = dst[pair];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
            if (threadIdx.x == 0 && pool == 0 && chunk == 0) flag(status, PA_CHECK_BLOCK_ID);
            continue;
        }
        uint8_t *base = pool ? vc : kc;
        const uint4 *from = reinterpret_cast<const uint4 *>(base + (int64_t)s * block_bytes);
        uint4 *to = reinterpret_cast<uint4 *>(base + (int64_t)d * block_bytes);
        const int64_t v0 = chunk * (kChunkBytes / 16) + threadIdx.x;
        const int64_t nv = block_bytes / 16;
        uint4 r[kBlkVecs];
#pragma unroll
        for (int k = 0; k < kBlkVecs; ++k) {
            const int64_t v = v0 + (int64_t)k * kBlkThreads;
            if (v < nv) r[k] = from[v];
        }
#pragma unroll
        for (int k = 0; k < kBlkVecs; ++k) {
            const int64_t v = v0 + (int64_t)k * kBlkThreads;
            if (v < nv) to[v] = r[k];
        }
    }
}

__global__ void __launch_bounds__(kBlkThreads)
zero_blocks_kernel(uint8_t *__restrict__ kc, uint8_t *__restrict__ vc, int64_t block_bytes,
                   int32_t num_blocks, const int32_t *__restrict__ ids, int32_t n, int64_t chunks,
                   unsigned int *status) {
    const int64_t jobs = (int64_t)n * 2 * chunks;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t job = blockIdx.x; job < jobs; job += gridDim.x) {
        const int64_t i = job / (2 * chunks);
        const int pool = (int)((job / chunks) & 1);
        const int64_t chunk = job % chunks;
        const int32_t b = ids[i];
        if (b < 0 || b >= num_blocks) {
            if (threadIdx.x == 0 && pool == 0 && chunk == 0) flag(status, PA_CHECK_BLOCK_ID);
            continue;
        }
        uint4 *to = reinterpret_cast<uint4 *>((pool ? vc : kc) + (int64_t)b * block_bytes);
        const int64_t v0 = chunk * (kChunkBytes / 16) + threadIdx.x;
        const int64_t nv = block_bytes / 16;
#pragma unroll
        for (int k = 0; k < kBlkVecs; ++k) {
            const int64_t v = v0 + (int64_t)k * kBlkThreads;
            if (v < nv) to[v] = zero;
        }
    }
}

static int blocks_grid(int64_t jobs) {
    const int64_t cap = 8LL * num_sms();
    return (int)(jobs < cap ? (jobs > 0 ? jobs : 1) : cap);
}

pa_status launch_copy_blocks(void *kc, void *vc, int64_t block_bytes, int32_t num_blocks,
                             const int32_t *src, const int32_t *dst, int32_t n,
                             cudaStream_t stream) {
    if (n == 0) return PA_OK;
    const int64_t chunks = (block_bytes + kChunkBytes - 1) / kChunkBytes;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    copy_blocks_kernel<<<blocks_grid((int64_t)n * 2 * chunks), kBlkThreads, 0, stream>>>(
        static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), block_bytes, num_blocks, src, dst,
        n, chunks, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

pa_status launch_zero_blocks(void *kc, void *vc, int64_t block_bytes, int32_t num_blocks,
                             const int32_t *ids, int32_t n, cudaStream_t stream) {
    if (n == 0) return PA_OK;
    const int64_t chunks = (block_bytes + kChunkBytes - 1) / kChunkBytes;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    zero_blocks_kernel<<<blocks_grid((int64_t)n * 2 * chunks), kBlkThreads, 0, stream>>>(
        static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), block_bytes, num_blocks, ids, n,
        chunks, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
