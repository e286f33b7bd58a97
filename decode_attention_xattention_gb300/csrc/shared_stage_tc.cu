// Shared stage on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention): the
// prompt KV is stored once per request, so the Shared stage serves every beam of a
// request from one copy; it produces local scores and max/sum statistics that the Merge
// stage later combines with an online softmax. The same section fuses the batched matmul
// with the softmax and pipelines the stages across hardware units; on GB300 that becomes
// one warp-specialised CTA: a TMA warp streams K/V tiles, an MMA warp drives the tensor
// core, and a softmax warpgroup turns scores into probabilities between the two matmuls.
//
// Work unit: (request r, KV head h). All BW beams x G query heads of that KV head are
// stacked into M = BW*G rows (row m = b*G + g), so one K/V tile read from HBM feeds every
// beam. A CTA owns one 128-row tile of those rows and one piece of the prefix:
//   for each 128-token K/V tile j of the piece:
//     S_j = Q . K_j^T               (tcgen05, bf16 in, fp32 in TMEM; S double-buffered)
//     P_j = exp2(S_j*scale*log2e - m) (softmax warpgroup: one thread per row)
//     O  += P_j . V_j               (tcgen05, P from shared memory, V as MN-major operand)
// The running max is only raised when it grows by more than 2^8, so O is rescaled rarely;
// every P stays below 2^8. The piece's normalised output and natural-log LSE are written
// to the workspace for the Merge stage.
//
// Every on-chip wait is bounded: on a timeout the CTA records XATTN_STATUS_TIMEOUT, writes
// NaN partials, waits (bounded) for its own TMA copies and MMAs, frees TMEM and returns.
#include "sm100_ptx.cuh"
#include "xattn_internal.cuh"

namespace xattn {
namespace {

using namespace ptx;

constexpr int kThreads = 192;  // warps 0-3 softmax / epilogue, warp 4 TMA, warp 5 MMA
constexpr int kMaxStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// K/V pipeline depth: 2 stages at d = 128, 4 at d = 64. Either way the shared memory
// admits one CTA per SM, so a CTA never waits for another's 512 TMEM columns.
template <int D>
struct Cfg {
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr int KB = D / 64;            // 128-byte swizzle blocks along d
    static constexpr int kTileBytes = KB * 16384; // 128 rows (or tokens) x d bf16
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffP = kOffV + kStages * kTileBytes;
    static constexpr int kPBytes = 2 * 16384;     // 128 rows x 128 tokens bf16
    static constexpr int kSmemBytes = kOffP + kPBytes + 1024;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `ch` (along the contraction dim) of row `row` in a tile
// stored as [ch/8 block][128 rows][128 B] with the 128-byte swizzle (chunk ^= row % 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int ch) {
    return (uint32_t)((ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
}

struct Bars {
    uint64_t k_full[kMaxStages], v_full[kMaxStages], kv_empty[kMaxStages];
    uint64_t s_full[2], s_free[2];
    uint64_t p_full, pv_done, q_ready, final_mma;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) shared_stage_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    Geometry g, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ shared_len,
    float* __restrict__ part_o, float* __restrict__ part_lse, int32_t* status) {
    using C = Cfg<D>;
    constexpr int kStages = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sK = smem + C::kOffK;
    uint8_t* sV = smem + C::kOffV;
    uint8_t* sP = smem + C::kOffP;
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Work item: CTAs of one (unit, piece) are adjacent so its K/V tiles are shared in L2.
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
    const int ntiles = t1 > t0 ? (t1 - t0 + kTileKeys - 1) / kTileKeys : 0;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.s_free[s], 128);
        }
        mbar_init(&bars.p_full, 128);
        mbar_init(&bars.pv_done, 1);
        mbar_init(&bars.q_ready, 128);
        mbar_init(&bars.final_mma, 1);
        abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 5 && ntiles > 0) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    const size_t prow0 = ((size_t)unit * g.nsplit + c) * g.M;  // first partial row of this piece

    if (warp < 4) {
        // ------------------------------------------------ softmax warpgroup: thread = row
        const int row = mt * kTileRows + tid;
        const bool row_ok = row < g.M;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        if (ntiles > 0) {
            {  // Q tile -> shared memory, K-major, 128-byte swizzle; rows past M are zero
                const __nv_bfloat16* src = nullptr;
                if (row_ok) {
                    const int b = row / g.G, gg = row - b * g.G;
                    src = q + (((size_t)r * g.BW + b) * g.Hq + (size_t)h * g.G + gg) * D;
                }
#pragma unroll
                for (int ch = 0; ch < D / 8; ++ch) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (row_ok) v = __ldg(reinterpret_cast<const uint4*>(src) + ch);
                    *reinterpret_cast<uint4*>(sQ + sw128_offset(tid, ch)) = v;
                }
                fence_proxy_async_smem();
                mbar_arrive(&bars.q_ready);
            }
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
            for (int j = 0; j < ntiles; ++j) {
                const int sb = j & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&bars.s_full[sb], (j >> 1) & 1, &abort_sh))) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int k = 0; k < 4; ++k) tmem_ld32(tmem + lane_base + (sb ? kTmemS1 : kTmemS0) + k * 32, sr[k]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars.s_free[sb]);  // S buffer may be overwritten now

                const int lim = t1 - (t0 + j * kTileKeys);  // valid columns of this tile (>= 1)
                float mx = -INFINITY;
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x = __uint_as_float(sr[k][i]) * g.scale_log2;
                        x = (k * 32 + i < lim) ? x : -INFINITY;
                        sr[k][i] = __float_as_uint(x);
                        mx = fmaxf(mx, x);
                    }
                const float m_new = fmaxf(m_run, mx);
                const bool resc = m_new > m_run + kRescaleThreshold;
                const float alpha = resc ? ex2(m_run - m_new) : 1.f;
                const float m_use = resc ? m_new : m_run;
                float sum = 0.f;
                uint32_t pk[4][16];
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float p0 = ex2(__uint_as_float(sr[k][2 * i]) - m_use);
                        const float p1 = ex2(__uint_as_float(sr[k][2 * i + 1]) - m_use);
                        sum += p0 + p1;
                        pk[k][i] = pack_bf16(p0, p1);
                    }
                l_run = l_run * alpha + sum;
                m_run = m_use;

                // O and the P buffer are free once the previous P.V has completed.
                if (j > 0) {
                    if (!__all_sync(0xffffffffu, mbar_wait(&bars.pv_done, (j - 1) & 1, &abort_sh))) { ok = false; break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {  // 16-byte chunk = 8 tokens
                        const int ch = k * 4 + cc;
                        *reinterpret_cast<uint4*>(sP + sw128_offset(tid, ch)) =
                            make_uint4(pk[k][cc * 4 + 0], pk[k][cc * 4 + 1], pk[k][cc * 4 + 2], pk[k][cc * 4 + 3]);
                    }
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + kTmemO + k * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tmem + lane_base + kTmemO + k * 32, o);
                    }
                    tmem_wait_st();
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars.p_full);
            }
            if (ok && !__all_sync(0xffffffffu, mbar_wait(&bars.pv_done, (ntiles - 1) & 1, &abort_sh))) ok = false;
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (!ok) {
                abort_sh = 1;
                if (lane == 0) set_status(status, XATTN_STATUS_TIMEOUT);
            }
            // Epilogue: normalised O row and its LSE.
            const float inv = ok ? 1.f / l_run : __int_as_float(0x7fc00000);
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + kTmemO + k * 32, o);
                tmem_wait_ld();
                if (row_ok) {
                    float4* dst = reinterpret_cast<float4*>(part_o + (prow0 + row) * D + k * 32);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                             __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
                }
            }
            if (row_ok) part_lse[prow0 + row] = ok ? (m_run + __log2f(l_run)) * kLn2 : __int_as_float(0x7fc00000);
        } else if (row_ok) {  // empty piece (past this request's prefix)
            float4* dst = reinterpret_cast<float4*>(part_o + (prow0 + row) * D);
#pragma unroll
            for (int i = 0; i < D / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            part_lse[prow0 + row] = -INFINITY;
        }
    } else if (warp == 4) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && ntiles > 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % kStages, u = j / kStages;
                if (u > 0 && !mbar_wait(&bars.kv_empty[st], (u - 1) & 1, &abort_sh)) break;
                const int tok = t0 + j * kTileKeys;
                mbar_arrive_expect_tx(&bars.k_full[st], C::kTileBytes);
#pragma unroll
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_4d(sK + st * C::kTileBytes + kb * 16384, &tmap_k, &bars.k_full[st], kb * 64, h, tok, r);
                mbar_arrive_expect_tx(&bars.v_full[st], C::kTileBytes);
#pragma unroll
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_4d(sV + st * C::kTileBytes + kb * 16384, &tmap_v, &bars.v_full[st], kb * 64, h, tok, r);
                issued = j + 1;
            }
            if (abort_sh) {  // let the copies still in flight land before the CTA exits
                volatile int never = 0;
                for (int j = max(0, issued - kStages); j < issued; ++j) {
                    mbar_wait(&bars.k_full[j % kStages], (j / kStages) & 1, &never);
                    mbar_wait(&bars.v_full[j % kStages], (j / kStages) & 1, &never);
                }
            }
        }
    } else {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && ntiles > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kTileKeys, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
            bool ok = mbar_wait(&bars.q_ready, 0, &abort_sh);
            tc_fence_after();
            auto issue_pv = [&](int i) -> bool {
                if (!mbar_wait(&bars.p_full, i & 1, &abort_sh)) return false;
                const int st = i % kStages;
                if (!mbar_wait(&bars.v_full[st], (i / kStages) & 1, &abort_sh)) return false;
                tc_fence_after();
                const uint32_t pbase = smem_addr(sP), vbase = smem_addr(sV + st * C::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(pbase + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, 16384, 1024);
                    mma_ss(tmem + kTmemO, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(&bars.pv_done);
                mma_commit(&bars.kv_empty[st]);
                return true;
            };
            for (int j = 0; ok && j < ntiles; ++j) {
                const int st = j % kStages, sb = j & 1;
                if (!mbar_wait(&bars.k_full[st], (j / kStages) & 1, &abort_sh)) { ok = false; break; }
                if (j >= 2 && !mbar_wait(&bars.s_free[sb], ((j >> 1) - 1) & 1, &abort_sh)) { ok = false; break; }
                tc_fence_after();
                const uint32_t qbase = smem_addr(sQ), kbase = smem_addr(sK + st * C::kTileBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + (sb ? kTmemS1 : kTmemS0), smem_desc_sw128(qbase + off, 16, 1024),
                           smem_desc_sw128(kbase + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars.s_full[sb]);
                if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok && !issue_pv(ntiles - 1)) ok = false;
            if (!ok) {
                abort_sh = 1;
                set_status(status, XATTN_STATUS_TIMEOUT);
            }
            // Every MMA issued above has completed before TMEM is released.
            mma_commit(&bars.final_mma);
            volatile int never = 0;
            mbar_wait(&bars.final_mma, 0, &never);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5 && ntiles > 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_d(const Geometry& g, const CUtensorMap& tk, const CUtensorMap& tv,
                     const __nv_bfloat16* q, const int32_t* slen, float* po, float* pl,
                     int32_t* status, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(shared_stage_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Cfg<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const long ctas = (long)g.R * g.Hkv * g.nsplit * g.row_tiles;
    shared_stage_tc_kernel<D><<<(unsigned)ctas, kThreads, Cfg<D>::kSmemBytes, stream>>>(tk, tv, g, q, slen, po, pl, status);
    return cudaGetLastError();
}

}  // namespace

int shared_tc_ctas_for(const Geometry& g) { return g.R * g.Hkv * g.nsplit * g.row_tiles; }

cudaError_t launch_shared_stage_tc(const Geometry& g, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                   const __nv_bfloat16* q, const int32_t* shared_len, float* part_o,
                                   float* part_lse, int32_t* status, cudaStream_t stream) {
    if (g.d == 128) return launch_d<128>(g, tmap_k, tmap_v, q, shared_len, part_o, part_lse, status, stream);
    if (g.d == 64) return launch_d<64>(g, tmap_k, tmap_v, q, shared_len, part_o, part_lse, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace xattn
