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
#include <cuda_fp8.h>

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

// The write into FP8 pools ("Inside vLLM: Following One Request", the write
// op's kv_cache_dtype, k_scale and v_scale): each element of the new key is
// divided by *k_scale (IEEE single-precision division) and rounded to the
// nearest E4M3 value, ties to even, saturating at +-448; V likewise with
// *v_scale.  One CTA per token at a time; a thread converts 8 elements (16
// bytes of bf16/fp16 in, 8 bytes out) per step.
template <typename T>
__global__ void __launch_bounds__(256)
cache_write_fp8_kernel(const T *__restrict__ key, const T *__restrict__ value, int64_t stride,
                       uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                       const int32_t *__restrict__ slots, int32_t T_, int32_t row,
                       int64_t num_slots, const float *k_scale, const float *v_scale,
                       unsigned int *status) {
    const float ks = k_scale ? *k_scale : 1.f, vs = v_scale ? *v_scale : 1.f;
    for (int t = blockIdx.x; t < T_; t += gridDim.x) {
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= num_slots) {
            if (threadIdx.x == 0) flag(status, PA_CHECK_SLOT);
            continue;
        }
        const T *ksrc = key + (int64_t)t * stride;
        const T *vsrc = value + (int64_t)t * stride;
        uint8_t *kd = kc + s * row;
        uint8_t *vd = vc + s * row;
        for (int i = threadIdx.x * 8; i < row; i += blockDim.x * 8) {
            const uint4 a = __ldg(reinterpret_cast<const uint4 *>(ksrc + i));
            const uint4 b = __ldg(reinterpret_cast<const uint4 *>(vsrc + i));
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
            uint32_t ka[2] = {0u, 0u}, vb[2] = {0u, 0u};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x0, x1, y0, y1;
                Elt<T>::unpack2(wa[e], x0, x1);
                Elt<T>::unpack2(wb[e], y0, y1);
                const uint32_t kq = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(x0, ks), __fdiv_rn(x1, ks)), __NV_SATFINITE, __NV_E4M3);
                const uint32_t vq = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(y0, vs), __fdiv_rn(y1, vs)), __NV_SATFINITE, __NV_E4M3);
                ka[e >> 1] |= (kq & 0xffffu) << (16 * (e & 1));
                vb[e >> 1] |= (vq & 0xffffu) << (16 * (e & 1));
            }
            *reinterpret_cast<uint2 *>(kd + i) = make_uint2(ka[0], ka[1]);
            *reinterpret_cast<uint2 *>(vd + i) = make_uint2(vb[0], vb[1]);
        }
    }
}

pa_status launch_cache_write_fp8(const void *key, const void *value, int64_t stride_elems,
                                 void *kc, void *vc, const int32_t *slots, int32_t T,
                                 int32_t row_elems, int64_t num_slots, pa_dtype src,
                                 const float *k_scale, const float *v_scale, cudaStream_t stream) {
    if (T == 0) return PA_OK;
    // 16-byte source rows and 8-byte destination rows
    const uintptr_t all = reinterpret_cast<uintptr_t>(key) | reinterpret_cast<uintptr_t>(value) |
                          (uintptr_t)(stride_elems * 2) | (uintptr_t)(row_elems * 2);
    if ((all & 15) != 0 || ((reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc) |
                             (uintptr_t)row_elems) & 7) != 0)
        return PA_ERR_UNSUPPORTED;
    const int threads = row_elems / 8 < 256 ? ((row_elems / 8 + 31) / 32) * 32 : 256;
    long long blocks = T;
    const long long cap = 16LL * num_sms();
    if (blocks > cap) blocks = cap;
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    if (src == PA_BF16)
        cache_write_fp8_kernel<__nv_bfloat16><<<(int)blocks, threads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(value),
            stride_elems, static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), slots, T,
            row_elems, num_slots, k_scale, v_scale, st);
    else
        cache_write_fp8_kernel<__half><<<(int)blocks, threads, 0, stream>>>(
            static_cast<const __half *>(key), static_cast<const __half *>(value), stride_elems,
            static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), slots, T, row_elems,
            num_slots, k_scale, v_scale, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
