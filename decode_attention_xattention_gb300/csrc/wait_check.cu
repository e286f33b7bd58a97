// Self-check of the bounded on-chip waits that the pipelined kernels use.
//
// One CTA waits, through the same bounded mbarrier wait as the kernels, on a phase that
// nothing completes. It must give up after about `limit_cycles` SM cycles, record
// XATTN_STATUS_TIMEOUT and exit, leaving the context usable: the timeout path is exercised
// without any fault. The phase is completed afterwards so that no wait is left pending.
#include "xattn_internal.cuh"
#include "sm100_ptx.cuh"

namespace xattn {
namespace {

__global__ void wait_check_kernel(long long limit_cycles, int32_t* status, long long* waited) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_sh;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_sh = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        const bool ok = ptx::mbar_wait(&bar, 0, &abort_sh, limit_cycles);  // nothing arrives
        if (waited) *waited = clock64() - t0;
        if (!ok) set_status(status, XATTN_STATUS_TIMEOUT);
        ptx::mbar_arrive(&bar);  // complete the phase: nothing stays pending
    }
}

}  // namespace
}  // namespace xattn

extern "C" int xattn_check_bounded_wait(int64_t limit_cycles, int32_t* status, int64_t* waited_cycles,
                                        xattn_stream_t stream) {
    if (!status || limit_cycles < 0 || limit_cycles > (1ll << 32)) return XATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(status) & 3u) || (reinterpret_cast<uintptr_t>(waited_cycles) & 7u))
        return XATTN_ERR_MISALIGNED;
    xattn::wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        (long long)limit_cycles, status, reinterpret_cast<long long*>(waited_cycles));
    return cudaGetLastError() == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}
