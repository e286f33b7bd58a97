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
// directly. The first call in each CUDA context looks the address up (with that context
// current) and caches it under the context's unique id; a context made again (after
// cudaDeviceReset, or a primary context released and retained again) has a new id, so its
// first call looks the address up afresh. Make that first call before capturing a stream
// into a CUDA graph.
//
// Every call uses the same array, which keeps the previous call's contents. The status
// word at its start is cleared on the stream at the start of each call that passed its
// host-side checks (the kernels only OR bits into it); the partial results are fully
// rewritten by each call. Calls whose work overlaps on the GPU (different streams, or
// different host threads on one device) race on the array: serialise them.
#include <cudaTypedefs.h>

#include <mutex>

#include "xattn_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(32) << 20;  // XATTN_NOALLOC_SCRATCH_BYTES

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Scratch address per CUDA context, keyed by the context's process-unique id.
constexpr int kMaxContexts = 64;
struct Entry {
    unsigned long long ctx_id;
    void* ptr;
};
std::mutex g_mu;
Entry g_cache[kMaxContexts] = {};
int g_next = 0;

using PFN_ctx_current = CUresult (*)(CUcontext*);
using PFN_ctx_id = CUresult (*)(CUcontext, unsigned long long*);

// Driver entry points for the current context and its id (null when unavailable; the
// address is then looked up on every call).
struct CtxFns {
    PFN_ctx_current current = nullptr;
    PFN_ctx_id id = nullptr;
};
const CtxFns& ctx_fns() {
    static CtxFns f;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult qr;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            f.current = reinterpret_cast<PFN_ctx_current>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            f.id = reinterpret_cast<PFN_ctx_id>(p);
    });
    return f;
}

// Unique id of the current context, 0 when there is none or it cannot be read.
unsigned long long current_ctx_id() {
    const CtxFns& f = ctx_fns();
    if (!f.current || !f.id) return 0;
    CUcontext ctx = nullptr;
    if (f.current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return f.id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of the scratch array in the current context.
cudaError_t scratch_address(void** out) {
    unsigned long long id = current_ctx_id();
    if (id != 0) {
        std::lock_guard<std::mutex> lock(g_mu);
        for (int i = 0; i < kMaxContexts; ++i)
            if (g_cache[i].ctx_id == id) {
                *out = g_cache[i].ptr;
                return cudaSuccess;
            }
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes a context current if none was
    if (e != cudaSuccess) return e;
    if (id == 0) id = current_ctx_id();
    if (id != 0) {
        std::lock_guard<std::mutex> lock(g_mu);
        g_cache[g_next] = Entry{id, p};
        g_next = (g_next + 1) % kMaxContexts;
    }
    *out = p;
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
    // Every host-side check of xattn_decode first: a rejected call enqueues nothing, so it
    // cannot clear the status word of a call already queued on the array.
    int rc = xattn::check_decode_args(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx,
                                      step, out, lse, ws, kNoallocScratchBytes);
    if (rc != XATTN_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return XATTN_ERR_CUDA;
    rc = xattn_decode(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step, out, lse,
                      ws, kNoallocScratchBytes, stream);
    if (rc != XATTN_OK) return rc;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return XATTN_ERR_CUDA;
    return XATTN_OK;
}
