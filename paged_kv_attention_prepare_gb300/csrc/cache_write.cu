// KV cache write ("Inside vLLM: Following One Request", the section on the
// write op): token i's K and V rows are copied to slot slot_mapping[i].
//
// The cache layout [block][slot-in-block][kv head][dim] makes one token's K
// for all kv heads one contiguous row of Hkv*D elements, so the write is a
// row copy.  One warp per token: the slot and the token's K and V rows are
// loaded together (the rows' addresses do not depend on the slot), up to four
// K and four V units per lane in flight, in the widest unit the addresses
// allow (16 bytes for the usual aligned rows); then the stores.  The grid
// covers every token in one wave up to five 256-thread CTAs per SM (the
// registers' limit at 48 a thread), more tokens per warp beyond that.
// Sources are read through the read-only path; a negative slot skips the
// token; a slot past the pool is flagged and skipped.
#include <cuda_fp8.h>

#include "pa_internal.cuh"

namespace pa {

constexpr int kWriteThreads = 256;
constexpr int kWriteCtasPerSm = 5;    // 40 warps an SM: registers capped at 48 a thread
constexpr int kWriteF8CtasPerSm = 4;  // FP8: 32 warps an SM, 64 registers (48 spill)
constexpr int kWriteWarps = kWriteThreads / 32;
constexpr int kWriteUnroll = 4;   // units of each row in flight per lane

template <typename V>
__global__ void __launch_bounds__(kWriteThreads, kWriteCtasPerSm)
cache_write_kernel(const V *__restrict__ key, const V *__restrict__ value, int64_t stride_v,
                   V *__restrict__ kc, V *__restrict__ vc, const int32_t *__restrict__ slots,
                   int32_t T, int32_t row_v, int64_t num_slots, unsigned int *status) {
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * kWriteWarps;
    for (long long t = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5); t < T; t += nw) {
        const int64_t s = slots[t];
        const V *ks = key + t * stride_v;
        const V *vs = value + t * stride_v;
        for (int i = lane; i < row_v; i += 32 * kWriteUnroll) {
            V kx[kWriteUnroll], vx[kWriteUnroll];
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u)
                if (i + 32 * u < row_v) {
                    kx[u] = __ldg(ks + i + 32 * u);
                    vx[u] = __ldg(vs + i + 32 * u);
                }
            if (s < 0) break;
            if (s >= num_slots) {
                if (lane == 0) flag(status, PA_CHECK_SLOT);
                break;
            }
            V *kd = kc + s * row_v;
            V *vd = vc + s * row_v;
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u)
                if (i + 32 * u < row_v) {
                    kd[i + 32 * u] = kx[u];
                    vd[i + 32 * u] = vx[u];
                }
        }
    }
}

// CTAs for T tokens, one warp each, up to one wave of them (ctas_per_sm
// resident on each SM).
static int write_blocks(int32_t T, int ctas_per_sm = kWriteCtasPerSm) {
    long long blocks = ((long long)T + kWriteWarps - 1) / kWriteWarps;
    const long long cap = (long long)ctas_per_sm * num_sms();
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : (int)blocks;
}

template <typename V>
static pa_status launch_as(const void *key, const void *value, int64_t stride_bytes, void *kc,
                           void *vc, const int32_t *slots, int32_t T, int64_t row_bytes,
                           int64_t num_slots, cudaStream_t stream) {
    const int32_t row_v = (int32_t)(row_bytes / sizeof(V));
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    cache_write_kernel<V><<<write_blocks(T), kWriteThreads, 0, stream>>>(
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
// *v_scale.  One warp per token as above; a lane converts 8 elements (16
// bytes of bf16/fp16 in, 8 bytes out) per unit, up to four units of K and
// four of V in flight.
template <typename T>
__global__ void __launch_bounds__(kWriteThreads, kWriteF8CtasPerSm)
cache_write_fp8_kernel(const T *__restrict__ key, const T *__restrict__ value, int64_t stride,
                       uint8_t *__restrict__ kc, uint8_t *__restrict__ vc,
                       const int32_t *__restrict__ slots, int32_t T_, int32_t row,
                       int64_t num_slots, const float *k_scale, const float *v_scale,
                       unsigned int *status) {
    const float ks = k_scale ? *k_scale : 1.f, vs = v_scale ? *v_scale : 1.f;
    const int lane = threadIdx.x & 31;
    const int nc = row / 8;   // 8-element units per row
    const long long nw = (long long)gridDim.x * kWriteWarps;
    for (long long t = (long long)blockIdx.x * kWriteWarps + (threadIdx.x >> 5); t < T_; t += nw) {
        const int64_t s = slots[t];
        const uint4 *ksrc = reinterpret_cast<const uint4 *>(key + t * stride);
        const uint4 *vsrc = reinterpret_cast<const uint4 *>(value + t * stride);
        for (int i = lane; i < nc; i += 32 * kWriteUnroll) {
            uint4 kx[kWriteUnroll], vx[kWriteUnroll];
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u)
                if (i + 32 * u < nc) {
                    kx[u] = __ldg(ksrc + i + 32 * u);
                    vx[u] = __ldg(vsrc + i + 32 * u);
                }
            if (s < 0) break;
            if (s >= num_slots) {
                if (lane == 0) flag(status, PA_CHECK_SLOT);
                break;
            }
            uint2 *kd = reinterpret_cast<uint2 *>(kc + s * row);
            uint2 *vd = reinterpret_cast<uint2 *>(vc + s * row);
#pragma unroll
            for (int u = 0; u < kWriteUnroll; ++u)
                if (i + 32 * u < nc) {
                    kd[i + 32 * u] = quantize8_e4m3<T>(kx[u], ks);
                    vd[i + 32 * u] = quantize8_e4m3<T>(vx[u], vs);
                }
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
    unsigned int *st = status_word();
    if (!st) return PA_ERR_CUDA;
    const int blocks = write_blocks(T, kWriteF8CtasPerSm);
    if (src == PA_BF16)
        cache_write_fp8_kernel<__nv_bfloat16><<<blocks, kWriteThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(value),
            stride_elems, static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), slots, T,
            row_elems, num_slots, k_scale, v_scale, st);
    else
        cache_write_fp8_kernel<__half><<<blocks, kWriteThreads, 0, stream>>>(
            static_cast<const __half *>(key), static_cast<const __half *>(value), stride_elems,
            static_cast<uint8_t *>(kc), static_cast<uint8_t *>(vc), slots, T, row_elems,
            num_slots, k_scale, v_scale, st);
    PA_TRY_CUDA(cudaGetLastError());
    note_launch();
    return PA_OK;
}

}  // namespace pa
