// xattn_decode_noalloc: xattn_decode for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs while another component
// owns every device allocation (an inference runtime or plugin host with its own memory
// pool), code on a latency-critical thread where cudaMalloc's implicit synchronisation is
// not acceptable, or a runtime with a fixed memory budget decided at start-up. For them
// the workspace lives in this file: a statically sized device array that the CUDA driver
// places on every device that loads the library and keeps there until the process exits.
//
// The array is named in host code only through cudaGetSymbolAddress: in host code the
// symbol is a host-side stand-in, not a device address, so it is never passed to a kernel
// directly. The first call on each device looks the address up (with that device current)
// and caches it; make that first call before capturing a stream into a CUDA graph.
//
// Every call uses the same array, which keeps the previous call's contents. The status
// word at its start is cleared on the stream at the start of each call (the kernels only
// OR bits into it); the partial results are fully rewritten by each call. Calls whose work
// overlaps on the GPU (different streams, or different host threads on one device) race on
// the array: serialise them.
#include <mutex>

#include "xattn_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // XATTN_NOALLOC_SCRATCH_BYTES

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int xattn_decode_noalloc(const xattn_desc* desc, const void* q, const void* shared_k,
                                    const void* shared_v, const int32_t* shared_len, const void* ns_k_pool,
                                    const void* ns_v_pool, const int32_t* beam_tok_idx, int32_t step, void* out,
                                    float* lse, int32_t* status_out, xattn_stream_t stream) {
    const size_t need = xattn_decode_workspace_size(desc);
    if (need == 0) return XATTN_ERR_INVALID_ARG;  // the descriptor itself is invalid
    if (need > kNoallocScratchBytes) return XATTN_ERR_WORKSPACE_TOO_SMALL;
    if (status_out && reinterpret_cast<uintptr_t>(status_out) % 4 != 0) return XATTN_ERR_MISALIGNED;
    void* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return XATTN_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return XATTN_ERR_CUDA;
    const int rc = xattn_decode(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step,
                                out, lse, ws, kNoallocScratchBytes, stream);
    if (rc != XATTN_OK) return rc;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return XATTN_ERR_CUDA;
    return XATTN_OK;
}
