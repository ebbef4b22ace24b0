// Diagnostic entry point: makes each kind of bounded on-chip wait of the
// library run out on purpose, so that its expiry path (status bit, return,
// a usable context afterwards) can be checked on the device.  Nothing is
// faulted and nothing waits longer than the limit the caller passes.
#include "internal.h"
#include "ptx.cuh"

namespace tcl {
namespace {

// kind 0: an mbarrier phase that never completes (no arrival is made);
// kind 1: a counter in global memory that nothing increments.
__global__ void k_wait_expiry(int kind, uint64_t limit_ns, int32_t *words)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0)
        mbar_init(&bar, 1);
    fence_mbar_init();
    __syncthreads();
    if (threadIdx.x != 0)
        return;
    const uint64_t t0 = global_timer_ns();
    bool ok;
    if (kind == 0)
        ok = mbar_wait_bounded(&bar, 0, words, limit_ns);
    else
        ok = wait_count_bounded(words + 1, 1u, words, limit_ns);
    words[2] = ok ? 1 : 0;
    words[3] = (int32_t)((global_timer_ns() - t0) / 1000ull);  // microseconds waited
}

}  // namespace
}  // namespace tcl

extern "C" lora_status lora_diag_wait_expiry(int kind, long long limit_ns, int32_t *words_dev, lora_stream_t stream)
{
    if (!words_dev || (kind != 0 && kind != 1) || limit_ns < 1000 || limit_ns > 100000000LL)
        return LORA_ERR_INVALID_ARG;
    tcl::k_wait_expiry<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(kind, (uint64_t)limit_ns, words_dev);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}
