// Shared stage on CUDA cores, for units with few stacked query rows.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention): the
// Shared stage computes local scores and max/sum statistics over the prompt KV, which is
// stored once per request. When a (request, KV head) unit stacks only a handful of query
// rows (beam width x heads per KV head, e.g. 4 for plain per-sequence decode with GQA 4),
// a 128-row tensor-core tile would be almost all padding; this kernel streams the prefix
// once per unit on CUDA cores instead (HBM-bound work).
//
// CTA = (unit, block of 4 stacked rows, prefix piece). The 4 warps walk interleaved groups
// of 4 tokens of the piece with an online softmax; lanes split the head dimension; the
// warps' states are merged in shared memory and the piece's (normalised output, lse) is
// written for the Merge stage.
#include "xattn_internal.cuh"

namespace xattn {
namespace {

constexpr int kRB = 4;  // stacked rows per CTA
constexpr int kWarps = 4;
// Tokens whose K/V rows a warp has in flight at once: the kernel serves few rows per unit, so
// it is a chain of dependent memory round trips; more per trip, fewer trips (16 at d = 64
// took the Tiny configuration's Shared stage from 19.2 to 15.0 us).
template <int D>
constexpr int kUnrollFor = D == 64 ? 16 : 8;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// E consecutive elements (bf16 or fp32 storage) as floats.
template <int E>
__device__ __forceinline__ void load_in(const __nv_bfloat16* p, float (&x)[E]) {
    if constexpr (E == 4) {
        uint2 u = *reinterpret_cast<const uint2*>(p);
        float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
        float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
        float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        x[0] = a.x; x[1] = a.y;
    }
}
template <int E>
__device__ __forceinline__ void load_in(const float* p, float (&x)[E]) {
    if constexpr (E == 4) {
        const float4 u = *reinterpret_cast<const float4*>(p);
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    } else {
        const float2 u = *reinterpret_cast<const float2*>(p);
        x[0] = u.x; x[1] = u.y;
    }
}

// T: storage type of q, shared_k and shared_v (bf16, or fp32 inputs used unrounded).
template <int D, typename T>
__global__ void __launch_bounds__(kWarps * 32) shared_stage_simt_kernel(
    Geometry g, const T* __restrict__ q, const T* __restrict__ sk, const T* __restrict__ sv,
    const int32_t* __restrict__ shared_len, float* __restrict__ part_o, float* __restrict__ part_lse, int pdl) {
    constexpr int E = D / 32;
    constexpr int kUnroll = kUnrollFor<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrb = (g.M + kRB - 1) / kRB;
    long t = blockIdx.x;
    const int c = (int)(t % g.nsplit);
    t /= g.nsplit;
    const int rb = (int)(t % nrb);
    const long unit = t / nrb;
    const int h = (int)(unit % g.Hkv);
    const int r = (int)(unit / g.Hkv);

    int L = shared_len[r];
    if (L < 0 || L > g.Lmax) L = 0;  // reported by the Merge stage
    const int t0 = c * g.split_tokens;
    const int t1 = min(t0 + g.split_tokens, L);

    float qv[kRB][E], acc[kRB][E], m[kRB], l[kRB];
#pragma unroll
    for (int i = 0; i < kRB; ++i) {
        const int row = rb * kRB + i;
        if (row < g.M) {
            const int b = row / g.G, gg = row - b * g.G;
            load_in<E>(q + (((size_t)r * g.BW + b) * g.Hq + (size_t)h * g.G + gg) * D + lane * E, qv[i]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) qv[i][e] = 0.f;
        }
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
    }

    const size_t tok_stride = (size_t)g.Hkv * D;
    const T* kbase = sk + ((size_t)r * g.Lmax * g.Hkv + h) * D + lane * E;
    const T* vbase = sv + ((size_t)r * g.Lmax * g.Hkv + h) * D + lane * E;
    // Warp w takes groups of kUnroll consecutive tokens (w*kUnroll, w*kUnroll + kWarps*kUnroll, ...);
    // the group's K and V rows are loaded before any is used.
    for (int j0 = t0 + warp * kUnroll; j0 < t1; j0 += kWarps * kUnroll) {
        float kv[kUnroll][E], vv[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (j0 + u < t1) {
                load_in<E>(kbase + (size_t)(j0 + u) * tok_stride, kv[u]);
                load_in<E>(vbase + (size_t)(j0 + u) * tok_stride, vv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (j0 + u >= t1) continue;
#pragma unroll
            for (int i = 0; i < kRB; ++i) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) s = fmaf(qv[i][e], kv[u][e], s);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                s *= g.scale_log2;
                const float mn = fmaxf(m[i], s);
                const float alpha = ex2(m[i] - mn);
                const float p = ex2(s - mn);
                l[i] = l[i] * alpha + p;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][e] = fmaf(p, vv[u][e], acc[i][e] * alpha);
                m[i] = mn;
            }
        }
    }

    __shared__ float sm_m[kWarps][kRB], sm_l[kWarps][kRB];
    __shared__ float sm_acc[kWarps][kRB][D];
#pragma unroll
    for (int i = 0; i < kRB; ++i) {
        if (lane == 0) { sm_m[warp][i] = m[i]; sm_l[warp][i] = l[i]; }
#pragma unroll
        for (int e = 0; e < E; ++e) sm_acc[warp][i][lane * E + e] = acc[i][e];
    }
    __syncthreads();
    // warp w finalises row w of the block
    const int i = warp;
    const int row = rb * kRB + i;
    if (i < kRB && row < g.M) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][i]);
        const size_t prow = ((size_t)unit * g.pieces + c) * g.M + row;
        if (M == -INFINITY) {  // empty piece
            for (int e = lane; e < D; e += 32) part_o[prow * D + e] = 0.f;
            if (lane == 0) part_lse[prow] = -INFINITY;
        } else {
            float wsum = 0.f, wt[kWarps];
            for (int w = 0; w < kWarps; ++w) {
                wt[w] = (sm_m[w][i] == -INFINITY) ? 0.f : ex2(sm_m[w][i] - M);
                wsum += sm_l[w][i] * wt[w];
            }
            const float inv = 1.f / wsum;
            for (int e = lane; e < D; e += 32) {
                float o = 0.f;
                for (int w = 0; w < kWarps; ++w) o += sm_acc[w][i][e] * wt[w];
                part_o[prow * D + e] = o * inv;
            }
            if (lane == 0) part_lse[prow] = (M + __log2f(wsum)) * kLn2;
        }
    }
    // launched as the programmatic dependent of the beam update (it reads nothing the update
    // writes): complete only after it, so that the kernels queued next find the update done
    if (pdl && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_shared_stage_simt(const Geometry& g, const void* q, const void* shared_k, const void* shared_v,
                                     const int32_t* shared_len, float* part_o, float* part_lse, int32_t* status,
                                     cudaStream_t stream, bool pdl, cudaEvent_t started) {
    (void)status;
    const long nrb = (g.M + kRB - 1) / kRB;
    const long ctas = (long)g.R * g.Hkv * nrb * g.nsplit;
    if (ctas > 0x7fffffffL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na++].val.programmaticStreamSerializationAllowed = 1;
    }
    if (started) {
        attr[na].id = cudaLaunchAttributeLaunchCompletionEvent;
        attr[na].val.launchCompletionEvent.event = started;
        attr[na++].val.launchCompletionEvent.flags = 0;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaSuccess;
    auto go = [&](auto kernel, auto tag) {
        using T = decltype(tag);
        e = cudaLaunchKernelEx(&cfg, kernel, g, static_cast<const T*>(q), static_cast<const T*>(shared_k),
                               static_cast<const T*>(shared_v), shared_len, part_o, part_lse, pdl ? 1 : 0);
    };
    if (g.d == 128 && g.in_f32) go(shared_stage_simt_kernel<128, float>, float{});
    else if (g.d == 128) go(shared_stage_simt_kernel<128, __nv_bfloat16>, __nv_bfloat16{});
    else if (g.d == 64 && g.in_f32) go(shared_stage_simt_kernel<64, float>, float{});
    else if (g.d == 64) go(shared_stage_simt_kernel<64, __nv_bfloat16>, __nv_bfloat16{});
    else return cudaErrorInvalidValue;
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace xattn
