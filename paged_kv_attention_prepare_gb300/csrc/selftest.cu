// Diagnostic: a kernel whose bounded wait can never be satisfied.  It takes
// the same mbarrier wait every pipeline in this library uses, on a barrier
// nothing arrives at, so the wait must give up at its time limit, record
// PA_CHECK_TIMEOUT in the status word and let the kernel return.
#include "pa_internal.cuh"

namespace pa {

__global__ void bounded_wait_probe(unsigned int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!mbar_wait_warp(&bar, 0) && threadIdx.x == 0) flag(status, PA_CHECK_TIMEOUT);
}

}  // namespace pa

extern "C" pa_status pa_selftest_wait_timeout(pa_stream_t stream) {
    unsigned int *st = pa::status_word();
    if (!st) return PA_ERR_CUDA;
    pa::bounded_wait_probe<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st);
    PA_TRY_CUDA(cudaGetLastError());
    pa::note_launch();
    return PA_OK;
}
