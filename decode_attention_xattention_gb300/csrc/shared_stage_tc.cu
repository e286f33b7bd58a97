// Shared stage on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a,
// optionally with the Non-Shared stage and the Merge in the same kernel.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention): the
// prompt KV is stored once per request, so the Shared stage serves every beam of a
// request from one copy; it produces local scores and max/sum statistics that the Merge
// stage combines with those of the Non-Shared stage by an online softmax. The section fuses
// the batched matmul with the softmax and pipelines the stages across hardware units; on
// GB300 that becomes one warp-specialised CTA: producer warps stream K/V tiles with TMA, an
// MMA warp drives the tensor core, and two softmax warpgroups turn scores into
// probabilities between the two matmuls, each on its own 128-row tile so the tensor core
// has the other tile's work while one warpgroup computes exponentials.
//
// Work unit: (request r, KV head h). All BW beams x G query heads of that KV head are
// stacked into M = BW*G rows (row m = b*G + g), so one K/V tile read from HBM feeds every
// beam. A CTA owns two 128-row tiles (rows 256p .. 256p+255) and one piece of the prefix.
// Per 128-token K/V tile j and row tile i:
//     S_i = Q_i . K_j^T                 tcgen05 (SS), fp32 in TMEM columns [128 i, 128 i + 128)
//     P_i = exp2(S_i*scale*log2e - m_i) softmax warpgroup i; P written back over S_i as bf16
//     O_i += P_i . V_j                  tcgen05 (TS: P read from TMEM), V as MN-major operand
// The MMA warp issues, per tile j and row tile i: PV_i(j-1) then QK_i(j), then commits
// s_full[i]; the commit therefore also tells softmax i that O_i is up to date. The running
// max is raised only when it grows by more than 2^8, so O is rescaled rarely and every P
// stays below 2^8.
//
// P enters the P.V product rounded to bf16 while the row sum adds the unrounded values. A
// row dominated by one key would then carry that key's rounding error (up to 2^-9
// relative) straight into its output, so each row also tracks its largest score (and the
// reference max its p was computed with), and the output is normalised by the row sum with
// that one term rounded as the tensor core saw it; the LSE keeps the exact row sum.
//
// Non-Shared part, three ways:
//   * in the tile (xattn_decode, one prefix piece, (128/G) x step <= 128): each softmax
//     warpgroup first copies its row tile's Non-Shared K/V rows from the pool (through the
//     ancestry index) into the two unit slots, laid out like a prefix K/V tile (key c of row tile i
//     = token c % step of its beam c / step). Each row tile attends to that tile first, with
//     every key outside its own beam's masked, and then to the prefix tiles: the online
//     softmax merges the two parts, and the epilogue writes out / lse.
//   * staged (one prefix piece, longer Non-Shared parts): the Non-Shared kernel runs first
//     and leaves each row's (normalised output, LSE) as a piece in the workspace; the
//     epilogue merges it with O (log-sum-exp rule) and writes out / lse.
//   * separate: this kernel writes the prefix piece's normalised output and LSE for the
//     Merge kernel.
//
// Every on-chip wait is bounded: on a timeout the CTA records XATTN_STATUS_TIMEOUT, writes
// NaN, waits (bounded) for its own TMA copies and MMAs, frees TMEM and returns.
#include "sm100_ptx.cuh"
#include "xattn_internal.cuh"

namespace xattn {
namespace {

using namespace ptx;

// Warp roles: 0-7 two softmax warpgroups (which first gather their row tile's Non-Shared
// rows, in-tile mode); 8 TMA producer; 9 MMA issuer (and TMEM owner). Every role that spins
// on an mbarrier has a warp of its own: divergent lanes of one warp run one path at a time,
// so a spinning lane would starve its neighbours.
constexpr int kThreads = 320;
constexpr int kWarpLoad = 8, kWarpMma = 9;
constexpr int kMaxStages = 4;
constexpr uint32_t kTmemCols = 512;  // S0 | S1 | O0 | O1, 128 columns each
constexpr uint32_t kTmemO = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kNaN = 0x7fc00000u;

// K/V pipeline. Iteration j of the MMA warp consumes V of tile j-1 (P.V) and K of tile j
// (Q.K^T), so the producer loads them together as load unit j = {K(j), V(j-1)} under one
// mbarrier: one data wait per tile on the MMA warp. Two unit slots at d = 128 (four at
// d = 64), each one K tile and one V tile; the shared memory admits one CTA per SM, so a
// CTA never waits for another's 512 TMEM columns. With the Non-Shared part in the tile,
// units 0 and 1 are the gathered Non-Shared K tiles (both row tiles) and V tiles (their own
// barriers, one per row tile), and the prefix units follow as units 2, 3, ...; the full
// barrier of slot 0 or 1 then sees its first TMA unit as phase 0.
template <int D, int U = (D == 64 ? 4 : 2)>
struct Cfg {
    static constexpr int kUnits = U;
    // query tiles held: two row tiles, or one when a third unit slot takes the second's place
    static constexpr int kQTiles = (D == 128 && U == 3) ? 1 : 2;
    static constexpr int KB = D / 64;              // 128-byte swizzle blocks along d
    static constexpr int kTileBytes = KB * 16384;  // 128 rows (or tokens) x d bf16
    static constexpr int kUnitBytes = 2 * kTileBytes;  // K tile, then V tile
    static constexpr int kOffQ = 0;                // kQTiles row tiles
    static constexpr int kOffU = kOffQ + kQTiles * kTileBytes;
    static constexpr int kSmemBytes = kOffU + kUnits * kUnitBytes + 1024;
    // in-tile mode: one more K tile after the unit slots (prefix tile 0, loaded at the start
    // while the gathered Non-Shared tiles hold the slots)
    static constexpr int kOffX = kOffU + kUnits * kUnitBytes;
    static constexpr int kSmemBytesNst = kSmemBytes + kTileBytes;
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

// Two fp32 lanes in one 64-bit register for the packed (f32x2) FMA-pipe instructions.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

struct Bars {
    uint64_t u_full[kMaxStages], u_empty[kMaxStages];
    uint64_t s_full[2], p_full[2], q_ready[2];
    uint64_t o_full[2], final_mma;
    uint64_t q_free, ns_full[2];  // last Q.K^T done; staged Non-Shared piece of row tile i in place
    uint64_t ns_kfull[2], ns_vfull[2];  // in-tile mode: row tile i's gathered K / V rows (and flags) in place
    uint64_t x_full;  // in-tile mode: prefix tile 0's K tile in its own region
};

// Epilogue mode and the Non-Shared inputs of the fused decode.
struct FusedArgs {
    void* out;
    float* lse;
    int enabled;  // write out / lse (else the prefix piece's partial result)
    int ns_tile;  // with enabled and step > 0: the Non-Shared part is gathered into tile 0
    const __nv_bfloat16* pool_k;
    const __nv_bfloat16* pool_v;
    const int32_t* idx;
    // launched as the programmatic dependent of the beam update that writes the pool and table:
    // in-tile mode the gather waits for it; otherwise nothing here reads what it writes, and
    // thread 0 of every CTA waits for it at the end, so that the kernels queued after this one
    // (the Non-Shared part) find the update complete
    int pdl;
};

// NST: the in-tile Non-Shared mode, compiled as its own instantiation so that the other
// modes' loops carry none of its branches (the MMA-issuing thread shares its issue slots
// with two softmax warps, and every instruction in its loop shows in the tile period).
// U: unit slots (default 2 at d = 128; 3 with a single row tile per CTA, whose query tile
// leaves room for a third).
template <int D, bool NST, int U = (D == 64 ? 4 : 2)>
__global__ void __launch_bounds__(kThreads, 1) shared_stage_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_ns, Geometry g,
    const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ shared_len, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* status, FusedArgs fa) {
    using C = Cfg<D, U>;
    constexpr int kU = C::kUnits;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::kOffQ;
    uint8_t* sU = smem + C::kOffU;  // unit slot u: K tile at sU + u * kUnitBytes, V tile after it
    __shared__ Bars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ uint32_t bad_beam[2][4];  // in-tile Non-Shared part: local beams with a bad ancestry slot

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Work item: CTAs of one (unit, piece) are adjacent so its K/V tiles are shared in L2.
    const int row_pairs = (g.row_tiles + 1) >> 1;
    long t = blockIdx.x;
    const int mp = (int)(t % row_pairs);
    t /= row_pairs;
    const int c = (int)(t % g.nsplit);
    const long unit = t / g.nsplit;
    const int h = (int)(unit % g.Hkv);
    const int r = (int)(unit / g.Hkv);
    const int L_raw = shared_len[r];
    const bool bad_len = L_raw < 0 || L_raw > g.Lmax;
    const int L = bad_len ? 0 : L_raw;
    const int t0 = c * g.split_tokens;
    const int t1 = min(t0 + g.split_tokens, L);
    const int ntiles = t1 > t0 ? (t1 - t0 + kTcTileKeys - 1) / kTcTileKeys : 0;  // prefix tiles
    const int ntile_m = (2 * mp + 1 < g.row_tiles) ? 2 : 1;  // row tiles this CTA owns
    // In-tile Non-Shared part (uniform over the grid): (128 / G) beams per row tile, `step`
    // keys each, at most 128 keys (checked by the host).
    constexpr bool ns = NST;  // the host launches this instantiation only for fused decodes with step > 0
    const int nb = kTileRows / g.G;
    const int nk = ns ? nb * g.step : 0;
    const int nt = ntiles + (ns ? 1 : 0);  // tiles every row tile attends to (tile 0: Non-Shared)
    // unit index of prefix unit p = u0 + p. In-tile mode: units 0 and 1 are the gathered
    // Non-Shared K and V tiles, prefix unit 0 (K(0) alone) sits in region X, and prefix units
    // p >= 1 follow as units 2, 3, ...
    const int u0 = ns ? 1 : 0;

    if (tid == 0) {
        for (int s = 0; s < kU; ++s) {
            mbar_init(&bars.u_full[s], 1);
            mbar_init(&bars.u_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.s_full[i], 1);
            mbar_init(&bars.p_full[i], 4);
            mbar_init(&bars.q_ready[i], 1);
        }
        mbar_init(&bars.o_full[0], 1);
        mbar_init(&bars.o_full[1], 1);
        mbar_init(&bars.final_mma, 1);
        mbar_init(&bars.x_full, 1);
        mbar_init(&bars.q_free, 1);
        mbar_init(&bars.ns_full[0], 1);
        mbar_init(&bars.ns_full[1], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.ns_kfull[i], 4);  // one arrival per warp of the gathering warpgroup
            mbar_init(&bars.ns_vfull[i], 4);
        }
        abort_sh = 0;
        fence_barrier_init();
    }
    if (tid < 8) bad_beam[tid >> 2][tid & 3] = 0u;
    if (warp == kWarpMma && nt > 0) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp < 8) {
        // ============================================ softmax warpgroups: thread = row
        const int wg = warp >> 2;
        const int rloc = tid & 127;
        const int mt = 2 * mp + wg;
        const bool tile_ok = wg < ntile_m;
        const int row = mt * kTileRows + rloc;
        const bool row_ok = tile_ok && row < g.M;
        const int b = row / g.G, gg = row - (row / g.G) * g.G;
        float m_run = -INFINITY, l_run = 0.f;
        // the row's largest raw score so far and the reference max its p was computed with
        float s_top = -INFINITY, m_top = 0.f;
        bool ok = true;
        if (ns && tile_ok) {
            // ---- Non-Shared gather of this warpgroup's row tile (in-tile mode). Key c < nk is
            // token c % step of the tile's local beam c / step; its K row goes to row c of the
            // K tile in slot 0 (row tile i at i * kTileBytes), its V row to the same row of the
            // V tile in slot 1, in the 128-byte-swizzled layout TMA gives a prefix tile (16-byte
            // chunk x of row c at chunk x ^ (c % 8)). Thread rloc copies chunk rloc % CH of
            // keys rloc / CH + KPS * j. A slot outside the pool is not read: the row is zeroed,
            // the beam marked bad (NaN output) and XATTN_STATUS_BAD_SLOT set.
            constexpr int CH = D / 8;       // 16-byte chunks per row
            constexpr int KPS = 128 / CH;   // keys per sweep of the warpgroup
            constexpr int NSW = kTcTileKeys / KPS;
            const int ch = rloc % CH, kb0 = rloc / CH;
            const int b0 = mt * nb;
            // (after a beam update launched just before this kernel, which wrote the pool and the
            // table: wait for it; nothing read above is written by it)
            if (fa.pdl) grid_dependency_wait();
            int sl[NSW];  // the slots first, every load in flight at once
#pragma unroll
            for (int j = 0; j < NSW; ++j) {
                const int cc = kb0 + KPS * j, bl = cc / g.step, bg = b0 + bl;
                const int v = (cc < nk && bg < g.BW)
                                  ? __ldg(fa.idx + ((size_t)r * g.BW + bg) * g.Tmax + (cc - bl * g.step))
                                  : -1;
                sl[j] = v;
                if (ch == 0 && cc < nk && bg < g.BW && (v < 0 || v >= g.S)) {
                    atomicOr(&bad_beam[wg][bl >> 5], 1u << (bl & 31));
                    set_status(status, XATTN_STATUS_BAD_SLOT);
                }
            }
            const uint32_t toff = (uint32_t)wg * C::kTileBytes + (ch >> 3) * 16384;
#pragma unroll
            for (int pass = 0; pass < 2; ++pass) {  // K rows, then V rows (two commit groups)
                const __nv_bfloat16* pool = pass == 0 ? fa.pool_k : fa.pool_v;
                const uint32_t dt = smem_addr(sU) + pass * C::kUnitBytes + toff;
#pragma unroll
                for (int j = 0; j < NSW; ++j) {
                    const int cc = kb0 + KPS * j;
                    if (cc < nk) {
                        const uint32_t dst = dt + cc * 128 + (((ch & 7) ^ (cc & 7)) << 4);
                        if (sl[j] >= 0 && sl[j] < g.S) {
                            cp_async_16(dst, pool + (((size_t)r * g.S + sl[j]) * g.Hkv + h) * D + ch * 8);
                        } else {
                            st_shared_zero16(dst);
                        }
                    } else if (pass == 1 && cc < ((nk + 15) & ~15)) {
                        // V rows past the last key, up to the end of its 16-key step: zero
                        st_shared_zero16(dt + cc * 128 + (((ch & 7) ^ (cc & 7)) << 4));
                    }
                }
                cp_async_commit_group();
            }
            cp_async_wait_group<1>();  // this thread's K rows have landed
            fence_proxy_async_smem();  // ... and are visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ns_kfull[wg]);
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.ns_vfull[wg]);
        }
        if (tile_ok && nt > 0) {
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + lane_base + wg * 128;
            const uint32_t tO = tmem + lane_base + kTmemO + wg * 128;
            // One tile: its S row in, P (bf16) back over it, running max and sum, O rescaled when
            // the max moved; valid columns [lo, lo + cnt), the rest get -inf.
            auto tile = [&](uint32_t parity, unsigned lo, unsigned cnt, bool first) -> bool {
                if (!mbar_wait_all(&bars.s_full[wg], parity, &abort_sh)) return false;
                tc_fence_after();
                // the whole 128-column row of S in registers with one wide load
                uint32_t s[kTcTileKeys];
                tmem_ld128(tS, s);
                tmem_wait_ld();
                if (lo != 0u || cnt < (unsigned)kTcTileKeys) {
#pragma unroll
                    for (int i = 0; i < kTcTileKeys; ++i)
                        if ((unsigned)i - lo >= cnt) s[i] = 0xff800000u;
                }
                float mx;
                {  // row max: eight independent chains of three-input max
                    float m8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) m8[u] = fmaxf(__uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1]));
#pragma unroll
                    for (int i = 8; i < kTcTileKeys / 2; ++i)
                        m8[i & 7] = max3(m8[i & 7], __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
                    mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                }
                const float m_new = fmaxf(m_run, mx * g.scale_log2);
                const bool resc = m_new > m_run + kRescaleThreshold;
                const float alpha = resc ? ex2(m_run - m_new) : 1.f;
                const float m_use = resc ? m_new : m_run;
                if (mx > s_top) {  // the row's largest p so far is this tile's
                    s_top = mx;
                    m_top = m_use;
                }
                // P = exp2(S*scale*log2e - m) as bf16, written over the consumed S columns
                // (masked columns hold -inf, so their P is exactly 0).
                // (column pairs through the packed fp32x2 FMA and add: fewer issue slots, which
                // the MMA warp on the same sub-partition needs)
                const uint64_t scale2 = f2_pack(g.scale_log2, g.scale_log2);
                const uint64_t negm2 = f2_pack(-m_use, -m_use);
                uint64_t sum2[2] = {0ull, 0ull};  // (0.f, 0.f)
                uint32_t p[kTcTileKeys / 2];
#pragma unroll
                for (int i = 0; i < kTcTileKeys / 2; ++i) {
                    const float2 x = f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                                                      scale2, negm2));
                    const float p0 = ex2(x.x), p1 = ex2(x.y);
                    sum2[i & 1] = f2_add(sum2[i & 1], f2_pack(p0, p1));
                    p[i] = pack_bf16(p0, p1);
                }
                tmem_st64(tS, p);
                const float2 sa = f2_unpack(sum2[0]), sb = f2_unpack(sum2[1]);
                const float tile_sum = (sa.x + sb.x) + (sa.y + sb.y);
                l_run = l_run * alpha + tile_sum;
                m_run = m_use;
                if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int k = 0; k < D / 32; ++k) {
                        uint32_t o[32];
                        tmem_ld32(tO + k * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + k * 32, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[wg]);  // one arrival per warp
                return true;
            };
            // In-tile mode: the Non-Shared tile first (only this row's beam's `step` keys count),
            // then the prefix tiles; a ragged last prefix tile ends at the prefix.
            if (ns) ok = tile(0u, (unsigned)((rloc / g.G) * g.step), (unsigned)g.step, true);
            for (int j = 0; ok && j < ntiles; ++j)
                ok = tile((uint32_t)(j + (ns ? 1 : 0)) & 1u, 0u,
                          (unsigned)min(kTcTileKeys, t1 - (t0 + j * kTcTileKeys)), !ns && j == 0);
        }
        const uint32_t tO = tmem + ((uint32_t)((warp & 3) * 32) << 16) + kTmemO + wg * 128;
        const bool have_o = tile_ok && nt > 0;  // O_i holds accumulated P.V (TMEM allocated)
        // O is normalised by the row sum with its largest term as the tensor core saw it: that
        // p recomputed with the element's own arithmetic, its bf16 rounding error carried to the
        // final reference max.
        float l_nrm = l_run;
        if (s_top > -INFINITY) {
            const float pt = ex2(fmaf(s_top, g.scale_log2, -m_top));
            l_nrm += (__bfloat162float(__float2bfloat16_rn(pt)) - pt) * ex2(m_top - m_run);
        }

        // Staged Non-Shared piece of this row (Non-Shared kernel ran first). With prefix tiles it
        // is staged in shared memory by the producer (tile 0 over the Q tiles, tile 1 over the
        // last unit's slot); its LSE is loaded before the wait for the last P.V.
        const bool staged = fa.enabled && g.step > 0 && !ns && C::kQTiles == 2;
        const bool fused_ns = staged && row_ok;
        const bool ns_staged = staged && have_o;  // warp-uniform
        const size_t nsrow = ((size_t)unit * g.pieces + g.nsplit) * g.M + row;
        const uint8_t* ns_sm = (wg == 0 ? sQ : sU + ((ntiles - 1) % kU) * C::kUnitBytes) + rloc * 128;
        float lns = -INFINITY;
        if (fused_ns) {
            grid_dependency_wait();  // the Non-Shared kernel launched before this one has finished
            lns = __ldg(part_lse + nsrow);
        }
        bool beam_bad = false;
        if (have_o) {
            if (ok && !mbar_wait_all(&bars.o_full[wg], 0, &abort_sh)) ok = false;
            if (ok && ns_staged && !mbar_wait_all(&bars.ns_full[wg], 0, &abort_sh)) ok = false;
            if (ok && ns && !mbar_wait_all(&bars.ns_vfull[wg], 0, &abort_sh)) ok = false;  // bad_beam written
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (!ok) {
                abort_sh = 1;
                if (lane == 0) set_status(status, XATTN_STATUS_TIMEOUT);
            } else if (ns) {
                const int bl = rloc / g.G;
                beam_bad = ((bad_beam[wg][bl >> 5] >> (bl & 31)) & 1u) != 0;
            }
        }

        if (fa.enabled) {
            // ---------------------------------------- final output (merged with a staged piece)
            bool bad = !ok || bad_len || beam_bad;
            if (tile_ok && rloc == 0 && mt == 0 && h == 0 && bad_len) set_status(status, XATTN_STATUS_BAD_SHARED_LEN);
            const size_t qrow = ((size_t)r * g.BW + b) * g.Hq + (size_t)h * g.G + gg;
            float m_tot = m_run, w_ns = 0.f, alpha = 1.f;
            if (fused_ns) {
                if (lns != lns) bad = true;  // a bad ancestry slot was reported by the Non-Shared kernel
                const float s_ns = lns * 1.4426950408889634f;
                m_tot = fmaxf(m_run, s_ns);
                alpha = (m_run == -INFINITY) ? 0.f : ex2(m_run - m_tot);
                w_ns = (s_ns > -INFINITY) ? ex2(s_ns - m_tot) : 0.f;
            }
            if (row_ok && !bad_len && L == 0 && g.step == 0) {
                bad = true;
                set_status(status, XATTN_STATUS_EMPTY_ROW);
            }
            const float l_tot = l_run * alpha + w_ns;  // exact: the LSE
            bad = bad || !(l_tot > 0.f);
            const float inv = bad ? __uint_as_float(kNaN) : 1.f / (l_nrm * alpha + w_ns);
            const size_t obase = qrow * D;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
                uint32_t o[32];
                if (have_o) {
                    tmem_ld32(tO + k * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0u;
                }
                float of[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) of[i] = __uint_as_float(o[i]) * alpha;
                if (w_ns != 0.f) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        // staged: 16-byte chunk i of this row's quarter k sits at chunk i ^ (row % 8)
                        const float4 v = ns_staged
                                             ? *reinterpret_cast<const float4*>(ns_sm + k * 16384 + ((i ^ (rloc & 7)) << 4))
                                             : __ldg(reinterpret_cast<const float4*>(part_o + nsrow * D) + k * 8 + i);
                        of[4 * i] = fmaf(w_ns, v.x, of[4 * i]);
                        of[4 * i + 1] = fmaf(w_ns, v.y, of[4 * i + 1]);
                        of[4 * i + 2] = fmaf(w_ns, v.z, of[4 * i + 2]);
                        of[4 * i + 3] = fmaf(w_ns, v.w, of[4 * i + 3]);
                    }
                }
                if (row_ok) {
                    if (g.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(fa.out) + obase + k * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(of[4 * i] * inv, of[4 * i + 1] * inv, of[4 * i + 2] * inv,
                                                 of[4 * i + 3] * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(fa.out) + obase + k * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pack_bf16(of[8 * i] * inv, of[8 * i + 1] * inv),
                                                pack_bf16(of[8 * i + 2] * inv, of[8 * i + 3] * inv),
                                                pack_bf16(of[8 * i + 4] * inv, of[8 * i + 5] * inv),
                                                pack_bf16(of[8 * i + 6] * inv, of[8 * i + 7] * inv));
                    }
                }
            }
            if (row_ok) fa.lse[qrow] = bad ? __uint_as_float(kNaN) : (m_tot + __log2f(l_tot)) * kLn2;
        } else if (tile_ok) {
            // ---------------------------------------- this piece's partial result
            const size_t prow = ((size_t)unit * g.pieces + c) * g.M + row;
            const float inv = !ok ? __uint_as_float(kNaN) : (ntiles > 0 ? 1.f / l_nrm : 0.f);
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                uint32_t o[32];
                if (have_o) {
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
                part_lse[prow] = !ok ? __uint_as_float(kNaN)
                                     : (ntiles > 0 ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY);
        }
    } else if (warp == kWarpLoad) {
        // ============================================ TMA producer
        // Prefix unit p = {K(p) if p < ntiles, V(p-1) if p >= 1} (unit index u0 + p) goes into
        // slot (u0 + p) % kU as soon as the unit kU before it has been consumed. (L2 prefetches
        // of later units, tried here, made the kernel 1-1.5 % slower and were taken out.)
        if (lane == 0 && nt > 0) {
            // the Q tiles first: per row tile one 64 d x G heads x 128/G beams box per 64 d
            // (128-byte swizzle, the K-major layout the MMA reads); beams past BW are zero-filled
            prefetch_tmap(&tmap_q);
            for (int i = 0; i < ntile_m; ++i) {
                mbar_arrive_expect_tx(&bars.q_ready[i], C::kTileBytes);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_4d(sQ + i * C::kTileBytes + kb * 16384, &tmap_q, &bars.q_ready[i], kb * 64, h * g.G,
                                ((2 * mp + i) * kTileRows) / g.G, r);
            }
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
            const int npu = ntiles > 0 ? ntiles + 1 : 0;  // prefix units
            int issued = 0;
            // the prefix tiles first out of L2 (each is read by the CTAs of its unit about at once,
            // then never again): the partials, the Non-Shared rows and the queries stay there
            uint64_t l2_first;
            asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(l2_first));
            if (ns && ntiles > 0) {  // prefix tile 0's K tile into region X at once
                mbar_arrive_expect_tx(&bars.x_full, C::kTileBytes);
                for (int kb = 0; kb < C::KB; ++kb)
                    tma_load_4d(smem + C::kOffX + kb * 16384, &tmap_k, &bars.x_full, kb * 64, h, t0, r);
                issued = 1;
            }
            for (int p = ns ? 1 : 0; p < npu; ++p) {
                const int u = u0 + p, st = u % kU, use = u / kU;
                if (use > 0 && !mbar_wait(&bars.u_empty[st], (use - 1) & 1, &abort_sh)) break;
                uint8_t* slot = sU + st * C::kUnitBytes;
                mbar_arrive_expect_tx(&bars.u_full[st], (p < ntiles ? C::kTileBytes : 0) + (p >= 1 ? C::kTileBytes : 0));
                for (int kb = 0; kb < C::KB; ++kb) {
                    if (p < ntiles)
                        tma_load_4d_hint(slot + kb * 16384, &tmap_k, &bars.u_full[st], kb * 64, h,
                                         t0 + p * kTcTileKeys, r, l2_first);
                    if (p >= 1)
                        tma_load_4d_hint(slot + C::kTileBytes + kb * 16384, &tmap_v, &bars.u_full[st], kb * 64, h,
                                         t0 + (p - 1) * kTcTileKeys, r, l2_first);
                }
                issued = p + 1;

            }
            // Staged Non-Shared piece: each row tile's piece (128 rows x d fp32, as 128-byte
            // swizzled boxes of 32 columns) for the epilogue: row tile 0 into the Q tiles once the
            // last Q.K^T is done, row tile 1 into the slot of unit ntiles - 1 once it is consumed.
            bool ns_issued[2] = {false, false};
            if (fa.enabled && g.step > 0 && !ns && C::kQTiles == 2 && issued == npu) {
                grid_dependency_wait();  // the Non-Shared kernel launched before this one has finished
                for (int i = 0; i < ntile_m; ++i) {
                    const int jl = ntiles - 1, st = jl % kU;
                    if (i == 0 ? !mbar_wait(&bars.q_free, 0, &abort_sh)
                               : !mbar_wait(&bars.u_empty[st], (jl / kU) & 1, &abort_sh))
                        break;
                    uint8_t* dst = i == 0 ? sQ : sU + st * C::kUnitBytes;
                    const int row0 = (int)(((size_t)unit * g.pieces + g.nsplit) * g.M) + (2 * mp + i) * kTileRows;
                    mbar_arrive_expect_tx(&bars.ns_full[i], (D / 32) * 16384);
                    for (int k = 0; k < D / 32; ++k) tma_load_2d(dst + k * 16384, &tmap_ns, &bars.ns_full[i], k * 32, row0);
                    ns_issued[i] = true;
                }
            }
            if (abort_sh) {  // let the copies still in flight land before the CTA exits
                volatile int never = 0;
                for (int p = max(ns ? 1 : 0, issued - kU); p < issued; ++p) {
                    const int u = u0 + p;
                    mbar_wait(&bars.u_full[u % kU], (u / kU - ((ns && u % kU < 2) ? 1 : 0)) & 1, &never);
                }
                if (ns && issued > 0) mbar_wait(&bars.x_full, 0, &never);
                for (int i = 0; i < ntile_m; ++i) mbar_wait(&bars.q_ready[i], 0, &never);
                for (int i = 0; i < 2; ++i)
                    if (ns_issued[i]) mbar_wait(&bars.ns_full[i], 0, &never);
            }
        }
    } else if (warp == kWarpMma) {
        // ============================================ MMA issuer (lane 0: every MMA and commit)
        if (lane == 0 && nt > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kTcTileKeys, 0, 0);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
            bool ok = mbar_wait(&bars.q_ready[0], 0, &abort_sh);
            if (ok && ntile_m > 1) ok = mbar_wait(&bars.q_ready[1], 0, &abort_sh);
            tc_fence_after();
            // The last prefix tile may be ragged: its P columns past the prefix are exact zeros,
            // the P.V product stops at the 16-token step holding the last valid token, and the
            // V rows of that step past the prefix are zeroed, so whatever the cache holds there
            // (even NaN) never reaches O. The gathered Non-Shared V tile has its rows past the
            // last key of the last 16-key step zeroed by the gather warp.
            const int lim_last = ntiles > 0 ? t1 - (t0 + (ntiles - 1) * kTcTileKeys) : 0;
            const int pv_steps_last = (lim_last + 15) / 16;
            const int ns_steps = (nk + 15) / 16;
            // Descriptors: an operand's descriptor for a byte offset only adds offset / 16 to the
            // start-address field (addresses stay below 256 KB, so no carry leaves the field).
            // Each tile's operand bases are formed once; every MMA then adds a constant.
            const uint64_t qdesc = smem_desc_sw128(smem_addr(sQ), 16, 1024);
            const uint64_t kdesc = smem_desc_sw128(smem_addr(sU), 16, 1024);
            const uint64_t vdesc = smem_desc_sw128(smem_addr(sU + C::kTileBytes), 16384, 1024);
            // S_i = Q_i . K^T, the K tile at byte offset ko from the first slot's K tile.
            auto issue_qk = [&](int i, uint32_t ko) {
                const uint64_t qb = desc_at(qdesc, (uint32_t)i * C::kTileBytes), kb = desc_at(kdesc, ko);
                const uint32_t d = tmem + i * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(d, desc_at(qb, off), desc_at(kb, off), idesc_qk, kk > 0 ? 1u : 0u);
                }
            };
            // O_i (+)= P_i . V for `steps` 16-key steps, the V tile at byte offset vo from the
            // first slot's V tile (a full tile's eight steps as one straight run of MMAs).
            auto issue_pv = [&](int i, uint32_t vo, int steps, uint32_t acc0) {
                const uint64_t vb = desc_at(vdesc, vo);
                const uint32_t d = tmem + kTmemO + i * 128, a = tmem + i * 128;
                if (steps == kTcTileKeys / 16) {
#pragma unroll
                    for (int kk = 0; kk < kTcTileKeys / 16; ++kk)
                        mma_ts(d, a + kk * 8, desc_at(vb, kk * 2048), idesc_pv, kk > 0 ? 1u : acc0);
                } else {
                    for (int kk = 0; kk < steps; ++kk)
                        mma_ts(d, a + kk * 8, desc_at(vb, kk * 2048), idesc_pv, kk > 0 ? 1u : acc0);
                }
            };
            auto pv_tile = [&](int i, int jt, int st) {
                issue_pv(i, (uint32_t)st * C::kUnitBytes, jt == ntiles - 1 ? pv_steps_last : kTcTileKeys / 16,
                         (jt > 0 || ns) ? 1u : 0u);
            };
            // Zeroes the V rows lim_last .. end of their 16-token step in slot st (whole 128-byte
            // rows, so the swizzle does not matter) and makes them visible to the tensor core
            // before the last P.V.
            auto zero_v_tail = [&](int st) {
                uint8_t* vt = sU + st * C::kUnitBytes + C::kTileBytes;
                for (int row = lim_last; row < pv_steps_last * 16; ++row)
#pragma unroll
                    for (int kb = 0; kb < C::KB; ++kb)
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            *reinterpret_cast<uint4*>(vt + kb * 16384 + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
            };
            if constexpr (NST) {
                // ---- in-tile mode. The Non-Shared tile: per row tile, Q.K^T against the gathered
                // K tile (slot 0), whose slot is then released.
                for (int i = 0; i < ntile_m; ++i) {
                    if (!mbar_wait(&bars.ns_kfull[i], 0, &abort_sh)) { ok = false; break; }
                    tc_fence_after();
                    issue_qk(i, (uint32_t)i * C::kTileBytes);
                    mma_commit(&bars.s_full[i]);
                }
                if (ok) mma_commit(&bars.u_empty[0]);
                // Iteration 0: per row tile, P.V of the Non-Shared tile (gathered V tile, slot 1),
                // then Q.K^T of prefix tile 0 (its K tile in region X, loaded at the start).
                if (ok && ntiles > 0 && !mbar_wait(&bars.x_full, 0, &abort_sh)) ok = false;
                for (int i = 0; ok && i < ntile_m; ++i) {
                    if (!mbar_wait(&bars.p_full[i], 0, &abort_sh) ||
                        !mbar_wait(&bars.ns_vfull[i], 0, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the gathered V tile of row tile i sits at slot 1's K position + i tiles
                    issue_pv(i, (uint32_t)(C::kUnitBytes + (i - 1) * C::kTileBytes), ns_steps, 0u);
                    if (ntiles == 0) {
                        mma_commit(&bars.o_full[i]);  // O_i complete
                    } else {
                        tc_fence_after();
                        issue_qk(i, (uint32_t)(C::kOffX - C::kOffU));
                        mma_commit(&bars.s_full[i]);
                    }
                }
                if (ok) {
                    if (ntiles == 1) mma_commit(&bars.q_free);
                    mma_commit(&bars.u_empty[1]);
                }
                // Prefix iterations j >= 1 read unit j + 1 = {K(j), V(j-1)}; its full barrier phase
                // is one less in slots 0 and 1 (the gathered tiles held them first), and the P
                // phases are one on (the Non-Shared tile took the first).
                for (int j = 1; ok && j <= ntiles; ++j) {
                    const int u = j + 1, st = u % kU;
                    if (!mbar_wait(&bars.u_full[st], (u / kU - (st < 2 ? 1 : 0)) & 1, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    if (j == ntiles && (lim_last & 15) != 0) zero_v_tail(st);
                    for (int i = 0; i < ntile_m; ++i) {
                        if (!mbar_wait(&bars.p_full[i], j & 1, &abort_sh)) { ok = false; break; }
                        tc_fence_after();
                        pv_tile(i, j - 1, st);
                        if (j == ntiles) mma_commit(&bars.o_full[i]);  // O_i complete
                        if (j < ntiles) {
                            issue_qk(i, (uint32_t)st * C::kUnitBytes);  // after the P wait's fence
                            mma_commit(&bars.s_full[i]);
                        }
                    }
                    if (!ok) break;
                    if (j == ntiles - 1) mma_commit(&bars.q_free);  // the Q tiles are no longer read
                    mma_commit(&bars.u_empty[st]);
                }
            } else {
                // Iteration j reads unit j = {K(j), V(j-1)}: per row tile, P.V of tile j-1 first (it
                // needs only V(j-1) and P_i), then Q.K^T of tile j into the same TMEM columns, then one
                // commit.
                for (int j = 0; ok && j <= ntiles; ++j) {
                    const int st = j % kU;
                    if (!mbar_wait(&bars.u_full[st], (j / kU) & 1, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    if (j == ntiles && (lim_last & 15) != 0) zero_v_tail(st);
                    for (int i = 0; i < ntile_m; ++i) {
                        if (j > 0) {
                            if (!mbar_wait(&bars.p_full[i], (j - 1) & 1, &abort_sh)) { ok = false; break; }
                            tc_fence_after();
                            pv_tile(i, j - 1, st);
                            if (j == ntiles) mma_commit(&bars.o_full[i]);  // O_i complete
                        }
                        if (j < ntiles) {
                            if (j == 0) tc_fence_after();  // later tiles: after the P wait's fence
                            issue_qk(i, (uint32_t)st * C::kUnitBytes);
                            mma_commit(&bars.s_full[i]);
                        }
                    }
                    if (!ok) break;
                    if (j == ntiles - 1) mma_commit(&bars.q_free);  // the Q tiles are no longer read
                    mma_commit(&bars.u_empty[st]);
                }
            }
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
    if (warp == kWarpMma && nt > 0) tmem_dealloc(tmem, kTmemCols);
    if (!ns && fa.pdl && tid == 0) grid_dependency_wait();
}

template <int D, bool NST, int U = (D == 64 ? 4 : 2)>
cudaError_t launch_d(const Geometry& g, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                     const CUtensorMap& tn, const __nv_bfloat16* q, const int32_t* slen, float* po, float* pl, int32_t* status,
                     const FusedArgs& fa, cudaStream_t stream, cudaEvent_t started) {
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(shared_stage_tc_kernel<D, NST, U>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             NST ? Cfg<D, U>::kSmemBytesNst : Cfg<D, U>::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    const long ctas = shared_tc_ctas_for(g);
    // In the staged fused decode the Non-Shared kernel runs just before this one and signals
    // early launch: CTAs of this kernel may start while its last wave drains (only the
    // epilogue reads its result, after griddepcontrol.wait).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = NST ? Cfg<D, U>::kSmemBytesNst : Cfg<D, U>::kSmemBytes;
    cfg.stream = stream;
    // `started` (optional) is recorded once every CTA has begun: a launch on another stream
    // that waits for it finds this kernel's CTAs already placed.
    cudaLaunchAttribute attr[2];
    int na = 0;
    if ((fa.enabled && g.step > 0 && !fa.ns_tile) || fa.pdl) {
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
    return cudaLaunchKernelEx(&cfg, shared_stage_tc_kernel<D, NST, U>, tk, tv, tq, tn, g, q, slen, po, pl, status, fa);
}

}  // namespace

int shared_tc_ctas_for(const Geometry& g) { return g.R * g.Hkv * g.nsplit * ((g.row_tiles + 1) / 2); }

cudaError_t launch_shared_stage_tc(const Geometry& g, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                   const CUtensorMap& tq, const CUtensorMap& tn, const __nv_bfloat16* q,
                                   const int32_t* shared_len, float* part_o, float* part_lse, int32_t* status, void* out,
                                   float* lse, bool fused, const NsTileArgs& nst_args, cudaStream_t stream) {
    FusedArgs fa{out,
                 lse,
                 fused ? 1 : 0,
                 nst_args.enabled ? 1 : 0,
                 reinterpret_cast<const __nv_bfloat16*>(nst_args.pool_k),
                 reinterpret_cast<const __nv_bfloat16*>(nst_args.pool_v),
                 nst_args.idx,
                 nst_args.pdl ? 1 : 0};
    const bool nst = fused && nst_args.enabled && g.step > 0;
    const cudaEvent_t ev = nst_args.started;
    // one row tile per CTA and partials only: a third K/V unit slot in place of the second
    // query tile (more loads in flight for the prefix stream)
    if (g.d == 128 && !fused && !nst && g.row_tiles == 1)
        return launch_d<128, false, 3>(g, tmap_k, tmap_v, tq, tn, q, shared_len, part_o, part_lse, status, fa, stream, ev);
    if (g.d == 128)
        return nst ? launch_d<128, true>(g, tmap_k, tmap_v, tq, tn, q, shared_len, part_o, part_lse, status, fa, stream, ev)
                   : launch_d<128, false>(g, tmap_k, tmap_v, tq, tn, q, shared_len, part_o, part_lse, status, fa, stream,
                                          ev);
    if (g.d == 64)
        return nst ? launch_d<64, true>(g, tmap_k, tmap_v, tq, tn, q, shared_len, part_o, part_lse, status, fa, stream, ev)
                   : launch_d<64, false>(g, tmap_k, tmap_v, tq, tn, q, shared_len, part_o, part_lse, status, fa, stream, ev);
    return cudaErrorInvalidValue;
}

}  // namespace xattn
