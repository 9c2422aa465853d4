// KV cache write ("Inside vLLM: Following One Request", the section on the
// write op): token i's K and V rows are copied to slot slot_mapping[i].
//
// The cache layout [block][slot-in-block][kv head][dim] makes one token's K
// for all kv heads one contiguous row of Hkv*D elements, so the write is a
// row copy.  One CTA handles one token at a time (grid-stride over tokens);
// its threads copy the K row and the V row in the widest unit the addresses
// allow (16 bytes for the usual aligned rows).  Sources are read through the
// read-only path; a negative slot skips the token; a slot past the pool is
// flagged and skipped.
#include "pa_internal.cuh"

namespace pa {

template <typename V>
__global__ void __launch_bounds__(256)
cache_write_kernel(const V *__restrict__ key, const V *__restrict__ value, int64_t stride_v,
                   V *__restrict__ kc, V *__restrict__ vc, const int32_t *__restrict__ slots,
                   int32_t T, int32_t row_v, int64_t num_slots, unsigned int *status) {
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= num_slots) {
            if (threadIdx.x == 0) flag(status, PA_CHECK_SLOT);
            continue;
        }
        const V *ks = key + (int64_t)t * stride_v;
        const V *vs = value + (int64_t)t * stride_v;
        V *kd = kc + s * row_v;
        V *vd = vc + s * row_v;
        for (int i = threadIdx.x; i < row_v; i += blockDim.x) {
            const V a = __ldg(ks + i);
            const V b = __ldg(vs + i);
            kd[i] = a;
            vd[i] = b;
        }
    }
}

template <typename V>
static pa_status launch_as(const void *key, const void *value, int64_t stride_bytes, void *kc,
                           void *vc, const int32_t *slots, int32_t T, int64_t row_bytes,
                           int64_t num_slots, cudaStream_t stream) {
    const int32_t row_v = (int32_t)(row_bytes / sizeof(V));
    int threads = row_v < 256 ? ((row_v + 31) / 32) * 32 : 256;
    long long blocks = T;
    const long long cap = 16LL * num_sms();
    if (blocks > cap) blocks = cap;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    cache_write_kernel<V><<<(int)blocks, threads, 0, stream>>>(
        static_cast<const V *>(key), static_cast<const V *>(value),
        stride_bytes / (int64_t)sizeof(V), static_cast<V *>(kc), static_cast<V *>(vc), slots, T,
        row_v, num_slots, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

pa_status launch_cache_write(const void *key, const void *value, int64_t stride_elems, void *kc,
                             void *vc, const int32_t *slots, int32_t T, int32_t row_elems,
                             int64_t num_slots, cudaStream_t stream) {
    if (T == 0) return PA_OK;
    const int64_t stride_bytes = stride_elems * 2, row_bytes = (int64_t)row_elems * 2;
    const uintptr_t all = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                          reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc) |
                          (uintptr_t)stride_bytes | (uintptr_t)row_bytes;
    if ((all & 15) == 0)
        return launch_as<uint4>(key, value, stride_bytes, kc, vc, slots, T, row_bytes, num_slots,
                                stream);
    if ((all & 7) == 0)
        return launch_as<uint2>(key, value, stride_bytes, kc, vc, slots, T, row_bytes, num_slots,
                                stream);
    if ((all & 3) == 0)
        return launch_as<uint32_t>(key, value, stride_bytes, kc, vc, slots, T, row_bytes,
                                   num_slots, stream);
    return launch_as<uint16_t>(key, value, stride_bytes, kc, vc, slots, T, row_bytes, num_slots,
                               stream);
}

}  // namespace pa
