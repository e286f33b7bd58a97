// Non-Shared stage fused with the Merge stage.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention):
// the Non-Shared stage computes local scores and max/sum statistics over the tokens a beam
// generated, reached through its ancestry index (token-granularity management); the Merge
// stage combines these with the Shared stage's statistics by an online softmax. Here the
// combine is the log-sum-exp rule: lse = log(sum_i exp(lse_i)), out = sum_i exp(lse_i - lse) o_i,
// over the Non-Shared part and every prefix piece the Shared stage produced.
//
// One warp per (request r, beam b, KV head h) serves the G query heads of that KV head, so
// each gathered pool row is read once for all G heads. Lanes split the head dimension.
#include "xattn_internal.cuh"

namespace xattn {
namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct LaneVec;
template <>
struct LaneVec<128> {  // 4 bf16 per lane = 8 bytes
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[4]) {
        uint2 u = *reinterpret_cast<const uint2*>(p);
        __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
        __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
        float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[4]) {
        __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
        __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = u;
    }
};
template <>
struct LaneVec<64> {  // 2 bf16 per lane = 4 bytes
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[2]) {
        float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
        x[0] = f.x; x[1] = f.y;
    }
    static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&x)[2]) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(x[0], x[1]);
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D, int G>
__global__ void __launch_bounds__(256) ns_merge_kernel(
    Geometry g, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ pool_k,
    const __nv_bfloat16* __restrict__ pool_v, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ shared_len, const float* __restrict__ part_o,
    const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
    int32_t* status) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long warp_id = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long nwarps = (long)g.R * g.BW * g.Hkv;
    if (warp_id >= nwarps) return;
    const int h = (int)(warp_id % g.Hkv);
    const int b = (int)((warp_id / g.Hkv) % g.BW);
    const int r = (int)(warp_id / ((long)g.Hkv * g.BW));

    const size_t qrow0 = ((size_t)r * g.BW + b) * g.Hq + (size_t)h * G;  // first of the G rows

    // Validity of the request's prefix length.
    const int L = shared_len ? shared_len[r] : 0;
    bool bad = (g.Lmax > 0) && (L < 0 || L > g.Lmax);
    if (bad && lane == 0 && h == 0 && b == 0) set_status(status, XATTN_STATUS_BAD_SHARED_LEN);
    const bool have_prefix = !bad && g.Lmax > 0 && L > 0;
    if (!bad && !have_prefix && g.step == 0) {
        bad = true;
        if (lane == 0) set_status(status, XATTN_STATUS_EMPTY_ROW);
    }

    // Non-Shared stage: online softmax over the ancestry tokens (base-2 domain).
    float qv[G][E], acc[G][E], m[G], l[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        LaneVec<D>::load(q + (qrow0 + gg) * D + lane * E, qv[gg]);
        m[gg] = -INFINITY;
        l[gg] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[gg][e] = 0.f;
    }
    const int32_t* row_idx = idx ? idx + ((size_t)r * g.BW + b) * g.Tmax : nullptr;
    for (int i = 0; i < g.step && !bad; ++i) {
        const int slot = __ldg(row_idx + i);
        if (slot < 0 || slot >= g.S) {
            bad = true;
            if (lane == 0) set_status(status, XATTN_STATUS_BAD_SLOT);
            break;
        }
        const size_t off = (((size_t)r * g.S + slot) * g.Hkv + h) * D + lane * E;
        float kv[E], vv[E];
        LaneVec<D>::load(pool_k + off, kv);
        LaneVec<D>::load(pool_v + off, vv);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) s = fmaf(qv[gg][e], kv[e], s);
            s = warp_sum(s) * g.scale_log2;
            const float mn = fmaxf(m[gg], s);
            const float alpha = ex2(m[gg] - mn);
            const float p = ex2(s - mn);
            l[gg] = l[gg] * alpha + p;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[gg][e] = fmaf(p, vv[e], acc[gg][e] * alpha);
            m[gg] = mn;
        }
    }

    // Merge: fold every Shared-stage piece into the running (m, l, acc) state. A piece
    // stores its normalised output o_c and natural-log lse_c; in base 2 it contributes
    // weight 2^(lse_c * log2 e) times o_c.
    if (have_prefix && !bad) {
        const size_t unit = (size_t)r * g.Hkv + h;
        for (int c = 0; c < g.nsplit; ++c) {
            const size_t prow = (unit * g.nsplit + c) * g.M + (size_t)b * G;
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                const float lc = __ldg(part_lse + prow + gg);
                if (lc != lc) bad = true;          // a failed Shared-stage piece poisons the row
                if (!(lc > -INFINITY)) continue;  // empty piece (or NaN)
                const float s2 = lc * kLog2e;
                const float mn = fmaxf(m[gg], s2);
                const float alpha = ex2(m[gg] - mn);
                const float w = ex2(s2 - mn);
                l[gg] = l[gg] * alpha + w;
                const float4* po = reinterpret_cast<const float4*>(part_o + (prow + gg) * D + lane * E);
                float ov[E];
                if constexpr (E == 4) {
                    float4 t = __ldg(po);
                    ov[0] = t.x; ov[1] = t.y; ov[2] = t.z; ov[3] = t.w;
                } else {
                    float2 t = __ldg(reinterpret_cast<const float2*>(po));
                    ov[0] = t.x; ov[1] = t.y;
                }
#pragma unroll
                for (int e = 0; e < E; ++e) acc[gg][e] = fmaf(w, ov[e], acc[gg][e] * alpha);
                m[gg] = mn;
            }
        }
    }

#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        float o[E];
        float row_lse;
        if (bad || !(l[gg] > 0.f)) {
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = __int_as_float(0x7fc00000);
            row_lse = __int_as_float(0x7fc00000);
        } else {
            const float inv = 1.f / l[gg];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = acc[gg][e] * inv;
            row_lse = (m[gg] + __log2f(l[gg])) * kLn2;
        }
        if (g.out_f32) {
            float* dst = reinterpret_cast<float*>(out) + (qrow0 + gg) * D + lane * E;
            if constexpr (E == 4) {
                *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
                *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
            }
        } else {
            LaneVec<D>::store(reinterpret_cast<__nv_bfloat16*>(out) + (qrow0 + gg) * D + lane * E, o);
        }
        if (lane == 0) lse[qrow0 + gg] = row_lse;
    }
}

template <int D>
cudaError_t launch_d(const Geometry& g, dim3 grid, dim3 block, cudaStream_t st, const __nv_bfloat16* q,
                     const __nv_bfloat16* pk, const __nv_bfloat16* pv, const int32_t* idx,
                     const int32_t* slen, const float* po, const float* pl, void* out,
                     float* lse, int32_t* status) {
    switch (g.G) {
#define XATTN_G(GV) \
    case GV: ns_merge_kernel<D, GV><<<grid, block, 0, st>>>(g, q, pk, pv, idx, slen, po, pl, out, lse, status); break;
        XATTN_G(1) XATTN_G(2) XATTN_G(4) XATTN_G(8) XATTN_G(16)
#undef XATTN_G
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

int merge_ctas_for(const Geometry& g) {
    const long warps = (long)g.R * g.BW * g.Hkv;
    return (int)((warps + 7) / 8);
}

cudaError_t launch_ns_merge(const Geometry& g, const __nv_bfloat16* q, const __nv_bfloat16* pool_k,
                            const __nv_bfloat16* pool_v, const int32_t* beam_tok_idx,
                            const int32_t* shared_len, const float* part_o, const float* part_lse,
                            void* out, float* lse, int32_t* status, cudaStream_t stream) {
    dim3 grid(merge_ctas_for(g)), block(256);
    if (g.d == 128)
        return launch_d<128>(g, grid, block, stream, q, pool_k, pool_v, beam_tok_idx, shared_len, part_o,
                             part_lse, out, lse, status);
    if (g.d == 64)
        return launch_d<64>(g, grid, block, stream, q, pool_k, pool_v, beam_tok_idx, shared_len, part_o,
                            part_lse, out, lse, status);
    return cudaErrorInvalidValue;
}

}  // namespace xattn
