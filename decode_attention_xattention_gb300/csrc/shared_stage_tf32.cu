// Shared stage on the tensor cores for fp32 storage (tcgen05.mma kind::tf32).
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention): the
// Shared stage attends the stacked query rows of a (request, KV head) unit to the prompt KV,
// stored once per request, and leaves per-row (normalised output, LSE) pieces for the Merge.
// This kernel does that for Q/K/V held in fp32 and read without a bf16 step: the tf32 form
// of the 5th-generation MMA multiplies fp32 shared-memory operands with 10 explicit mantissa
// bits and accumulates in fp32 in TMEM.
//
// The tf32 form takes both operands K-major (the reduction dimension contiguous), so the two
// products are staged as
//   S = Q . K^T : A = Q (rows x d), B = K tile (keys x d)        -- both as stored;
//   O += P . V  : A = P (rows x keys, fp32), B = V^T (d x keys) -- V transposed on staging.
// CTA = (unit, prefix piece, 128-row tile), one warpgroup of 128 threads, thread = row
// (TMEM lane). Per 64-key tile: the warpgroup stages the K tile and V^T in 128-byte swizzled
// K-major layouts (plain loads; the fp32 configurations are small), thread 0 issues
// S = Q.K^T into TMEM, every thread turns its S row into P (fp32) in shared memory with the
// online softmax (and rescales its O row in TMEM when the running max moved), thread 0
// issues O += P.V, and the next tile is staged once that has completed. The epilogue writes
// the piece's normalised O and LSE in the partial layout the other Shared-stage kernels use.
//
// Every wait is bounded: on a timeout the CTA records XATTN_STATUS_TIMEOUT, writes NaN,
// waits (bounded) for its own MMAs and frees TMEM.
#include "sm100_ptx.cuh"
#include "xattn_internal.cuh"

namespace xattn {
namespace {

using namespace ptx;

constexpr int kRows = 128;   // rows per CTA (the MMA's M)
constexpr int kKeys = 64;    // keys per tile (S's N, P.V's reduction)
constexpr uint32_t kTmemCols = 256;  // S (64 columns) | O (d columns)
constexpr uint32_t kTmemO = 64;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kNaN = 0x7fc00000u;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of fp32 element (row, k) in a K-major operand of `rows` rows with 128-byte
// swizzle: 32 elements (128 bytes) of k per row in each block of k, blocks rows*128 bytes
// apart; in a block, 16-byte chunk c of row `row` sits at chunk c ^ (row % 8).
__device__ __forceinline__ uint32_t sw_off(int rows, int row, int k) {
    return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + (k & 3) * 4);
}

// The descriptor offset of K-step kk (8 fp32 = 32 bytes) of a K-major swizzled operand.
__device__ __forceinline__ uint32_t kstep_off(int rows, int kk) { return (uint32_t)((kk >> 2) * rows * 128 + (kk & 3) * 32); }

template <int D>
struct Tf32Cfg {
    static constexpr int kQBytes = D * 4 * kRows;   // Q: 128 rows x d
    static constexpr int kKBytes = D * 4 * kKeys;   // K tile: 64 keys x d
    static constexpr int kVBytes = D * 4 * kKeys;   // V^T: d rows x 64 keys
    static constexpr int kPBytes = kKeys * 4 * kRows;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kKBytes;
    static constexpr int kOffP = kOffV + kVBytes;
    static constexpr int kSmemBytes = kOffP + kPBytes + 1024;
};

template <int D>
__global__ void __launch_bounds__(kRows, 1) shared_stage_tf32_kernel(
    Geometry g, const float* __restrict__ q, const float* __restrict__ sk, const float* __restrict__ sv,
    const int32_t* __restrict__ shared_len, float* __restrict__ part_o, float* __restrict__ part_lse,
    int32_t* status, int pdl) {
    using C = Tf32Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = smem + C::kOffK;
    uint8_t* sV = smem + C::kOffV;
    uint8_t* sP = smem + C::kOffP;
    __shared__ uint64_t bar_mma, bar_fin;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5;
    long t = blockIdx.x;
    const int mt = (int)(t % g.row_tiles);
    t /= g.row_tiles;
    const int c = (int)(t % g.nsplit);
    const long unit = t / g.nsplit;
    const int h = (int)(unit % g.Hkv);
    const int r = (int)(unit / g.Hkv);
    int L = shared_len[r];
    if (L < 0 || L > g.Lmax) L = 0;  // reported by the Merge stage
    const int t0 = c * g.split_tokens;
    const int t1 = min(t0 + g.split_tokens, L);
    const int ntiles = t1 > t0 ? (t1 - t0 + kKeys - 1) / kKeys : 0;
    const int row = mt * kRows + tid;
    const bool row_ok = row < g.M;

    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_fin, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    {  // this thread's Q row (zero past the unit's rows)
        const int b = row / g.G, gg = row - (row / g.G) * g.G;
        const float4* qr = row_ok ? reinterpret_cast<const float4*>(
                                        q + (((size_t)r * g.BW + b) * g.Hq + (size_t)h * g.G + gg) * D)
                                  : nullptr;
#pragma unroll 4
        for (int k4 = 0; k4 < D / 4; ++k4) {
            const float4 v = row_ok ? __ldg(qr + k4) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(sQ + sw_off(kRows, tid, 4 * k4)) = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base, tO = tmem + lane_base + kTmemO;

    constexpr uint32_t idesc_qk = idesc_tf32_f32(kRows, kKeys);
    constexpr uint32_t idesc_pv = idesc_tf32_f32(kRows, D);
    const uint64_t qdesc = smem_desc_sw128(smem_addr(sQ), 16, 1024);
    const uint64_t kdesc = smem_desc_sw128(smem_addr(sK), 16, 1024);
    const uint64_t pdesc = smem_desc_sw128(smem_addr(sP), 16, 1024);
    const uint64_t vdesc = smem_desc_sw128(smem_addr(sV), 16, 1024);

    const size_t tok_stride = (size_t)g.Hkv * D;
    const float* kb = sk + ((size_t)r * g.Lmax * g.Hkv + h) * D;
    const float* vb = sv + ((size_t)r * g.Lmax * g.Hkv + h) * D;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint32_t phase = 0;
    for (int j = 0; j < ntiles; ++j) {
        const int k0 = t0 + j * kKeys, cnt = min(kKeys, t1 - k0);
        // ---- stage the K tile (keys x d) and V^T (d x keys); keys past the piece are zero
        for (int e = tid; e < kKeys * (D / 4); e += kRows) {
            const int key = e / (D / 4), k4 = e - key * (D / 4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (key < cnt) {
                kv = __ldg(reinterpret_cast<const float4*>(kb + (size_t)(k0 + key) * tok_stride) + k4);
                vv = __ldg(reinterpret_cast<const float4*>(vb + (size_t)(k0 + key) * tok_stride) + k4);
            }
            *reinterpret_cast<float4*>(sK + sw_off(kKeys, key, 4 * k4)) = kv;
            *reinterpret_cast<float*>(sV + sw_off(D, 4 * k4 + 0, key)) = vv.x;
            *reinterpret_cast<float*>(sV + sw_off(D, 4 * k4 + 1, key)) = vv.y;
            *reinterpret_cast<float*>(sV + sw_off(D, 4 * k4 + 2, key)) = vv.z;
            *reinterpret_cast<float*>(sV + sw_off(D, 4 * k4 + 3, key)) = vv.w;
        }
        fence_proxy_async_smem();  // this thread's stores, visible to the tensor core
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- S = Q . K^T
        if (tid == 0 && !abort_sh) {
#pragma unroll
            for (int kk = 0; kk < D / 8; ++kk)
                mma_ss_tf32(tmem, desc_at(qdesc, kstep_off(kRows, kk)), desc_at(kdesc, kstep_off(kKeys, kk)), idesc_qk,
                            kk > 0 ? 1u : 0u);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_all(&bar_mma, phase, &abort_sh) && ok;
        phase ^= 1u;
        tc_fence_after();
        // ---- online softmax of this row: P (fp32) to shared memory, O rescaled in TMEM
        uint32_t s[kKeys];
        {
            uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
            uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
            tmem_ld32(tS, lo);
            tmem_ld32(tS + 32, hi);
            tmem_wait_ld();
        }
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kKeys; ++i) {
            if (i >= cnt) s[i] = 0xff800000u;  // -inf: keys past the piece
            mx = fmaxf(mx, __uint_as_float(s[i]));
        }
        const float m_new = fmaxf(m_run, mx * g.scale_log2);
        const float alpha = m_run == -INFINITY ? 0.f : ex2(m_run - m_new);
        float sum = 0.f;
#pragma unroll
        for (int i4 = 0; i4 < kKeys / 4; ++i4) {
            float4 p;
            p.x = ex2(fmaf(__uint_as_float(s[4 * i4 + 0]), g.scale_log2, -m_new));
            p.y = ex2(fmaf(__uint_as_float(s[4 * i4 + 1]), g.scale_log2, -m_new));
            p.z = ex2(fmaf(__uint_as_float(s[4 * i4 + 2]), g.scale_log2, -m_new));
            p.w = ex2(fmaf(__uint_as_float(s[4 * i4 + 3]), g.scale_log2, -m_new));
            sum += (p.x + p.y) + (p.z + p.w);
            *reinterpret_cast<float4*>(sP + sw_off(kRows, tid, 4 * i4)) = p;
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t o[32];
                tmem_ld32(tO + k * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(tO + k * 32, o);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // ---- O += P . V
        if (tid == 0 && !abort_sh) {
#pragma unroll
            for (int kk = 0; kk < kKeys / 8; ++kk)
                mma_ss_tf32(tmem + kTmemO, desc_at(pdesc, kstep_off(kRows, kk)), desc_at(vdesc, kstep_off(D, kk)),
                            idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_all(&bar_mma, phase, &abort_sh) && ok;
        phase ^= 1u;
        tc_fence_after();
        if (!ok) abort_sh = 1;
    }
    if (!ok && tid == 0) set_status(status, XATTN_STATUS_TIMEOUT);

    // ---- the piece's normalised output and LSE (TMEM loads by whole warps)
    const size_t prow = ((size_t)unit * g.pieces + c) * g.M + row;
    const float inv = !ok ? __uint_as_float(kNaN) : (ntiles > 0 ? 1.f / l_run : 0.f);
#pragma unroll 1
    for (int k = 0; k < D / 32; ++k) {
        uint32_t o[32];
        if (ntiles > 0) {
            tmem_ld32(tO + k * 32, o);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(part_o + prow * D + k * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                     __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        }
    }
    if (row_ok)
        part_lse[prow] = !ok ? __uint_as_float(kNaN) : (ntiles > 0 ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY);

    if (tid == 0) {  // every MMA issued above has completed before TMEM is released
        mma_commit(&bar_fin);
        volatile int never = 0;
        mbar_wait(&bar_fin, 0, &never);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    // launched as the programmatic dependent of the beam update (it reads nothing the update
    // writes): complete only after it, so that the kernels queued next find the update done
    if (pdl && tid == 0) grid_dependency_wait();
}

template <int D>
cudaError_t launch_d(const Geometry& g, const float* q, const float* sk, const float* sv, const int32_t* slen,
                     float* po, float* pl, int32_t* status, cudaStream_t stream, bool pdl) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(shared_stage_tf32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Tf32Cfg<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const long ctas = (long)g.R * g.Hkv * g.nsplit * g.row_tiles;
    if (ctas <= 0 || ctas > 0x7fffffffL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kRows);
    cfg.dynamicSmemBytes = Tf32Cfg<D>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, shared_stage_tf32_kernel<D>, g, q, sk, sv, slen, po, pl, status,
                                             pdl ? 1 : 0);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_shared_stage_tf32(const Geometry& g, const void* q, const void* shared_k, const void* shared_v,
                                     const int32_t* shared_len, float* part_o, float* part_lse, int32_t* status,
                                     cudaStream_t stream, bool pdl) {
    auto fq = static_cast<const float*>(q);
    auto fk = static_cast<const float*>(shared_k);
    auto fv = static_cast<const float*>(shared_v);
    if (g.d == 64) return launch_d<64>(g, fq, fk, fv, shared_len, part_o, part_lse, status, stream, pdl);
    if (g.d == 128) return launch_d<128>(g, fq, fk, fv, shared_len, part_o, part_lse, status, stream, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace xattn
