// In-place bookkeeping of one beam-search step for the Non-Shared part.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention):
// the Non-Shared cache is managed per token, so forking beams copies no physical block;
// the update is done in place without read-before-write hazards.
//
// Reading used here: the token a beam emits at step s is written once, to the fresh slot
// s*BW + b (for a request the BW new tokens fill one contiguous run of slots, so the K/V
// write is a straight copy). Only the small ancestry table changes otherwise:
// row b becomes its parent's row followed by the new slot. Column i of the new table
// depends only on column i of the old one, so the table is rewritten in place by CTAs that
// each own a range of columns and stage it in shared memory (all reads, barrier, all
// writes): no entry is read after it has been overwritten.
#include "xattn_internal.cuh"

namespace xattn {
namespace {

constexpr int kThreads = 256;
constexpr int kTableInts = 8192;  // largest shared-memory band: 32 KB (BW up to 8192, one column)

// Table columns per table CTA: at most a 32 KB band, and about 2048 entries so that long
// tables are spread over many CTAs.
__host__ __device__ inline int table_cols(int BW, int step) {
    const int c = 2048 / BW;
    return c < 1 ? 1 : (c > step ? step : c);
}

__global__ void __launch_bounds__(kThreads) beam_update_kernel(
    int BW, int row16, int S, int Tmax, int step, int copy_ctas, const int32_t* __restrict__ parent,
    const uint4* __restrict__ new_k, const uint4* __restrict__ new_v, uint4* __restrict__ pool_k,
    uint4* __restrict__ pool_v, int32_t* __restrict__ idx, int32_t* status) {
    // a decode launched after this kernel as its programmatic dependent may start now: it
    // reads the pool and the table only after waiting for this grid to complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = blockIdx.x;
    if ((int)blockIdx.y < copy_ctas) {
        // 1. K/V of the new tokens: [BW, Hkv, d] of request r -> slots step*BW .. step*BW+BW-1
        //    (row16: 16-byte vectors per slot). All loads of a thread are issued before its
        //    stores (independent 16-byte vectors).
        const size_t n16 = (size_t)BW * row16;
        const uint4* sk = new_k + (size_t)r * BW * row16;
        const uint4* sv = new_v + (size_t)r * BW * row16;
        uint4* dk = pool_k + ((size_t)r * S + (size_t)step * BW) * row16;
        uint4* dv = pool_v + ((size_t)r * S + (size_t)step * BW) * row16;
        const size_t stride = (size_t)copy_ctas * kThreads;
        size_t i = (size_t)blockIdx.y * kThreads + threadIdx.x;
        for (; i + 3 * stride < n16; i += 4 * stride) {
            uint4 a[4], c[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) { a[u] = __ldg(sk + i + u * stride); c[u] = __ldg(sv + i + u * stride); }
#pragma unroll
            for (int u = 0; u < 4; ++u) { dk[i + u * stride] = a[u]; dv[i + u * stride] = c[u]; }
        }
        for (; i < n16; i += stride) {
            const uint4 a = __ldg(sk + i), c = __ldg(sv + i);
            dk[i] = a;
            dv[i] = c;
        }
        return;
    }

    // 2. Ancestry table of request r, in place. Column i of the new table depends only on
    //    column i of the old one, so the columns are split into ranges of `cols` columns, one
    //    per table CTA (blockIdx.y - copy_ctas); each stages its range in shared memory (all
    //    reads, barrier, all writes). These CTAs copy nothing, so their dependent loads
    //    overlap the copies of the others.
    extern __shared__ int32_t band[];  // BW x cols entries (dynamic: the copying CTAs hold none of it)
    const int tc = (int)blockIdx.y - copy_ctas;
    int32_t* tab = idx + (size_t)r * BW * Tmax;
    const int32_t* par = parent ? parent + (size_t)r * BW : nullptr;
    if (tc == 0) {
        for (int b = threadIdx.x; b < BW; b += kThreads) {
            tab[(size_t)b * Tmax + step] = step * BW + b;  // column `step` is never read below
            if (step > 0) {
                const int p = par[b];
                if (p < 0 || p >= BW) set_status(status, XATTN_STATUS_BAD_PARENT);
            }
        }
    }
    if (step == 0) return;
    const int cols = table_cols(BW, step);
    const int c0 = tc * cols, cc = min(cols, step - c0);
    if (cc <= 0) return;
#pragma unroll 4
    for (int i = threadIdx.x; i < BW * cc; i += kThreads) {
        const int b = i / cc, c = i - b * cc;
        band[i] = tab[(size_t)b * Tmax + c0 + c];
    }
    __syncthreads();  // every old entry of the range read before any is overwritten
#pragma unroll 4
    for (int i = threadIdx.x; i < BW * cc; i += kThreads) {
        const int b = i / cc, c = i - b * cc;
        const int p = __ldg(par + b);
        tab[(size_t)b * Tmax + c0 + c] = (p >= 0 && p < BW) ? band[p * cc + c] : -1;
    }
}

}  // namespace

cudaError_t launch_beam_update(int R, int BW, int Hkv, int d, int elem_bytes, int S, int Tmax, int step,
                               const int32_t* parent, const void* new_k, const void* new_v, void* pool_k,
                               void* pool_v, int32_t* idx, int32_t* status, cudaStream_t stream,
                               int vectors_per_thread) {
    if (BW > kTableInts) return cudaErrorInvalidValue;
    if (((size_t)Hkv * d * elem_bytes) % 16 != 0) return cudaErrorInvalidValue;
    const int row16 = (int)((size_t)Hkv * d * elem_bytes / 16);  // 16-byte vectors per slot
    const size_t n16 = (size_t)BW * row16;
    // about vectors_per_thread 16-byte vectors of K and V per thread (all loads of a thread in
    // flight at once): 4 keeps the grid near one CTA per SM, so that the update ends sooner; 1
    // spreads it over more, smaller CTAs
    const int vpt = vectors_per_thread > 0 ? vectors_per_thread : 1;
    int ybl = (int)((n16 + (size_t)vpt * kThreads - 1) / ((size_t)vpt * kThreads));
    ybl = max(1, min(ybl, 1024));
    const int tcols = step > 0 ? (step + table_cols(BW, step) - 1) / table_cols(BW, step) : 1;
    dim3 grid(R, ybl + tcols);  // the last tcols CTAs of each request rewrite its ancestry table
    const size_t band_bytes = step > 0 ? (size_t)BW * table_cols(BW, step) * sizeof(int32_t) : 0;
    beam_update_kernel<<<grid, kThreads, band_bytes, stream>>>(
        BW, row16, S, Tmax, step, ybl, parent, static_cast<const uint4*>(new_k), static_cast<const uint4*>(new_v),
        static_cast<uint4*>(pool_k), static_cast<uint4*>(pool_v), idx, status);
    return cudaGetLastError();
}

}  // namespace xattn
