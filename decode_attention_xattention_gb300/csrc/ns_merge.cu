// Non-Shared stage and Merge stage.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.1 (xAttention):
// the Non-Shared stage computes local scores and max/sum statistics over the tokens a beam
// generated, reached through its ancestry index (token-granularity management); the Merge
// stage combines these with the Shared stage's statistics by an online softmax. Here the
// combine is the log-sum-exp rule: lse = log(sum_i exp(lse_i)), out = sum_i exp(lse_i - lse) o_i,
// over every piece of the prefix the Shared stage produced and the Non-Shared part.
//
// Kernels:
//   ns_piece_kernel    one warp per (request r, beam b, KV head h, piece of at most kNsChunk
//                      ancestry positions): the Non-Shared stage of that piece, written into
//                      the workspace after the prefix pieces. With one piece (step <= 32) it
//                      runs ahead of the Shared-stage kernel, whose epilogue merges; for long
//                      Non-Shared parts (e.g. a 512-token unshared suffix per sequence) the
//                      pieces are merged by merge_rows_kernel.
//   ns_merge_kernel    one warp per (r, b, h): the G query heads of that KV head (each
//                      gathered pool row is read once for all G); lanes split the head
//                      dimension. It walks the beam's ancestry tokens itself (<= 32 of
//                      them), then folds in every prefix piece stored in the workspace and
//                      writes out / lse (split prefixes).
//   merge_rows_kernel  one warp per query row: folds every stored piece (prefix and
//                      Non-Shared) and writes out / lse; merge_rows_few_kernel does the
//                      same for rows of at most 8 pieces in one round trip.
#include "xattn_internal.cuh"
#include "sm100_ptx.cuh"

namespace xattn {
namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kNsTok = 2;  // Non-Shared tokens per round of the direct walk
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kNaN = 0x7fc00000u;

template <int D>
struct LaneVec;
template <>
struct LaneVec<128> {  // 4 bf16 per lane = 8 bytes
    static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&x)[4]) {
        uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        float2 fa = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
        float2 fb = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
        x[0] = fa.x; x[1] = fa.y; x[2] = fb.x; x[3] = fb.y;
    }
    static __device__ __forceinline__ void load(const float* p, float (&x)[4]) {  // fp32 storage
        const float4 u = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
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
        float2 f = __bfloat1622float2(__ldg(reinterpret_cast<const __nv_bfloat162*>(p)));
        x[0] = f.x; x[1] = f.y;
    }
    static __device__ __forceinline__ void load(const float* p, float (&x)[2]) {  // fp32 storage
        const float2 u = __ldg(reinterpret_cast<const float2*>(p));
        x[0] = u.x; x[1] = u.y;
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

// Online-softmax state of G rows, lanes splitting the head dimension (base-2 domain).
template <int E, int G>
struct RowState {
    float acc[G][E], m[G], l[G];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            m[gg] = -INFINITY;
            l[gg] = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[gg][e] = 0.f;
        }
    }
    // fold in one value vector v with log2-weight s2 for row gg
    __device__ __forceinline__ void add(int gg, float s2, const float (&v)[E]) {
        const float mn = fmaxf(m[gg], s2);
        const float alpha = ex2(m[gg] - mn);
        const float p = ex2(s2 - mn);
        l[gg] = l[gg] * alpha + p;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[gg][e] = fmaf(p, v[e], acc[gg][e] * alpha);
        m[gg] = mn;
    }
};

// Non-Shared stage of one (request r, beam b, KV head h) warp: online softmax over the
// beam's ancestry tokens (step <= 32 of them), kNsTok tokens per round: their K/V rows are
// loaded together, the kNsTok x G partial dot products are reduced across the warp in one
// interleaved butterfly, and the running state takes one rescale per round. Lanes split the
// head dimension. Returns false (status BAD_SLOT) when an ancestry slot is out of range.
template <int D, int G, typename T>
__device__ __forceinline__ bool ns_walk(const Geometry& g, int r, int b, int h, int lane,
                                        const T* __restrict__ q, const T* __restrict__ pool_k,
                                        const T* __restrict__ pool_v, const int32_t* __restrict__ idx,
                                        RowState<D / 32, G>& st, int32_t* status) {
    constexpr int E = D / 32;
    const size_t qrow0 = ((size_t)r * g.BW + b) * g.Hq + (size_t)h * G;
    const int32_t* row_idx = idx + ((size_t)r * g.BW + b) * g.Tmax;
    const int my_slot = lane < g.step ? __ldg(row_idx + lane) : 0;
    float qv[G][E];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) LaneVec<D>::load(q + (qrow0 + gg) * D + lane * E, qv[gg]);
    if (__any_sync(0xffffffffu, lane < g.step && (my_slot < 0 || my_slot >= g.S))) {
        if (lane == 0) set_status(status, XATTN_STATUS_BAD_SLOT);
        return false;
    }
    for (int i0 = 0; i0 < g.step; i0 += kNsTok) {
        float kv[kNsTok][E], vv[kNsTok][E];
#pragma unroll
        for (int u = 0; u < kNsTok; ++u) {
            const int slot = __shfl_sync(0xffffffffu, my_slot, (i0 + u) & 31);
            if (i0 + u < g.step) {
                const size_t off = (((size_t)r * g.S + slot) * g.Hkv + h) * D + lane * E;
                LaneVec<D>::load(pool_k + off, kv[u]);
                LaneVec<D>::load(pool_v + off, vv[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) kv[u][e] = vv[u][e] = 0.f;
            }
        }
        float sc[kNsTok][G];
#pragma unroll
        for (int u = 0; u < kNsTok; ++u)
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float t = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) t = fmaf(qv[gg][e], kv[u][e], t);
                sc[u][gg] = t;
            }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < kNsTok; ++u)
#pragma unroll
                for (int gg = 0; gg < G; ++gg) sc[u][gg] += __shfl_xor_sync(0xffffffffu, sc[u][gg], o);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            float s2[kNsTok];
            float mx = st.m[gg];
#pragma unroll
            for (int u = 0; u < kNsTok; ++u) {
                s2[u] = (i0 + u < g.step) ? sc[u][gg] * g.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s2[u]);
            }
            const float alpha = ex2(st.m[gg] - mx);
            float psum = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) st.acc[gg][e] *= alpha;
#pragma unroll
            for (int u = 0; u < kNsTok; ++u) {
                const float p = ex2(s2[u] - mx);
                psum += p;
#pragma unroll
                for (int e = 0; e < E; ++e) st.acc[gg][e] = fmaf(p, vv[u][e], st.acc[gg][e]);
            }
            st.l[gg] = st.l[gg] * alpha + psum;
            st.m[gg] = mx;
        }
    }
    return true;
}

// 16-byte asynchronous global -> shared copy (L2 only) and its group bookkeeping.
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Warp-level tensor-core MMA, m16n8k16, bf16 inputs, fp32 accumulators (d += a * b).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 bf16 matrices from shared memory (lane i gives row i % 8 of matrix i / 8), plain
// or transposed.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// Transpose of an 8x8 bf16 matrix held in the MMA fragment layout (lane l: row l/4,
// columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&t);
}

constexpr int kPieceBlk = 16;    // positions per block (the k of one P.V MMA)
constexpr int kRingBlocks = 2;   // blocks staged per warp: one being computed, one in flight
constexpr int kPieceHead = 128;  // bytes before the staged rows: mbarriers and flags
// Shared-memory row stride of a staged pool row: the row plus 16 bytes, so that the eight
// rows one ldmatrix reads start in eight different groups of four banks.
__host__ __device__ constexpr int piece_row_stride(int D) { return D * 2 + 16; }
// Dynamic shared memory of one ns_piece_kernel warp (CTA): the K and V rows of the ring.
__host__ __device__ constexpr int piece_smem_bytes(int D) {
    return kPieceHead + 2 * kRingBlocks * kPieceBlk * piece_row_stride(D);
}
// CTAs per SM the shared memory admits (228 KB per SM, 1 KB of it reserved per CTA); the
// kernel's register budget is sized for that many.
__host__ __device__ constexpr int piece_ctas_per_sm(int D) {
    return (228 * 1024) / (piece_smem_bytes(D) + 1024) > 16 ? 16 : (228 * 1024) / (piece_smem_bytes(D) + 1024);
}

// Coordinates of a Non-Shared piece: request r, beam b, KV head h, piece c of the beam's
// ancestry positions, n of them (>= 1).
struct NsPiece {
    int r, b, h, c, n;
};
__device__ __forceinline__ NsPiece ns_piece_of(const Geometry& g, unsigned npc, unsigned t) {
    NsPiece k;
    const unsigned rbh = t / npc;
    k.c = (int)(t - rbh * npc);
    const unsigned rb = rbh / (unsigned)g.Hkv;
    k.h = (int)(rbh - rb * (unsigned)g.Hkv);
    k.r = (int)(rb / (unsigned)g.BW);
    k.b = (int)(rb - (unsigned)k.r * (unsigned)g.BW);
    k.n = min(kNsChunk, g.step - k.c * kNsChunk);
    return k;
}

// Non-Shared stage of (request, beam, KV head) pieces of at most kNsChunk ancestry positions,
// each stored as workspace piece `nsplit + piece` for the Shared-stage epilogue (one piece:
// step <= 32) or the row-merge kernel to merge; prefix-length problems and empty rows are
// reported by those.
//
// One warp per CTA, persistent: the grid is one wave of resident CTAs and CTA w takes the
// pieces w, w + gridDim.x, ... in turn. A piece is cut into blocks of 16 positions; the
// warp's blocks, across piece boundaries, stream through a ring of kRingBlocks buffers:
// the pool rows of a block (2d contiguous bytes of one head each) are copied 16 bytes per
// lane with cp.async (half the warp K rows, half V rows), every lane's copies completing on
// the buffer's mbarrier (one cp.async arrival per lane), and a buffer is refilled with the
// block kRingBlocks ahead as soon as its block is computed. The ring is kept short so that many warps fit on
// an SM: the warps' arithmetic is a chain of dependent steps, and it is the number of
// warps, not the depth of one warp's ring, that keeps both the SM and HBM busy. The
// ancestry slots of the next piece are loaded a piece ahead, its Q rows as soon as the
// current piece's last Q K^T has been issued.
// Arithmetic, transposed so that the 16 positions of a block are the M dimension of the MMA
// (m16n8k16, bf16 inputs, fp32 accumulators) and the G query heads of the KV head its N
// dimension, 8 heads per tile: S^T = K Q^T costs D/16 MMAs per head tile and O^T = V^T P^T
// D/16 more, with K and V read by ldmatrix straight from the staged rows (V transposed).
// The online softmax runs down the columns of S^T (one column per query head), P^T is
// rounded to bf16 (as the Shared-stage kernel rounds P) and moved from the accumulator
// layout to the B operand layout by movmatrix, and O^T is rescaled once per block. The
// running sums take the fp32 weights.
template <int D, int G>
__global__ void __launch_bounds__(32, piece_ctas_per_sm(D)) ns_piece_kernel(
    Geometry g, int npc, int ntasks, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ pool_k,
    const __nv_bfloat16* __restrict__ pool_v, const int32_t* __restrict__ idx, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* status) {
    static_assert(G <= 16, "at most two tiles of 8 query heads");
    static_assert(kNsChunk <= 64 && kNsChunk % kPieceBlk == 0, "a lane holds the slots of positions lane, lane + 32");
    static_assert(kPieceBlk == 16 && 32 % kPieceBlk == 0, "a block's positions lie on one side of position 32");
    static_assert(kRingBlocks >= 2 && kRingBlocks <= 8, "ring of 2..8 buffers (mbarriers at offset 0, flags at 64)");
    constexpr int RB = D * 2;                   // bytes of one pool row (one head)
    constexpr int RS = piece_row_stride(D);     // its stride in shared memory
    constexpr int KS = D / 16;                  // k-steps of K Q^T, and 16-row tiles of O^T
    constexpr int NH = (G + 7) / 8;             // tiles of 8 query heads
    // the Shared-stage kernel that follows in the fused decode may start its CTAs now; it
    // reads this kernel's output only after waiting for its completion
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(128) uint8_t psm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(psm);              // one per ring buffer
    int* buf_bad = reinterpret_cast<int*>(psm + 64);                // the buffer's piece has a bad slot
    volatile int* abort_sh = reinterpret_cast<volatile int*>(psm + 96);
    uint8_t* k_sm = psm + kPieceHead;
    uint8_t* v_sm = k_sm + kRingBlocks * kPieceBlk * RS;
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const int stride = (int)gridDim.x;
    // The pool rows are read once: marked first out of L2, so that they do not push out what
    // is read again soon (the pieces' partial results, which the row merge reads next, and the
    // Shared stage's partials and K/V tiles beside it).
    uint64_t l2_first;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(l2_first));
    if (lane == 0) {
        for (int j = 0; j < kRingBlocks; ++j) ptx::mbar_init(&full[j], 32);  // one cp.async arrival per lane
        *abort_sh = 0;
        ptx::fence_barrier_init();
    }
    __syncwarp();

    // ancestry slots of a piece's positions lane and lane + 32
    auto load_slots = [&](const NsPiece& k, int& sa, int& sb) {
        const int32_t* ri = idx + ((size_t)k.r * g.BW + k.b) * g.Tmax + k.c * kNsChunk;
        sa = lane < k.n ? __ldg(ri + lane) : 0;
        sb = lane + 32 < k.n ? __ldg(ri + lane + 32) : 0;
    };
    // Q^T of a piece as the B operand: head nh*8 + gid, elements 2 tig, 2 tig + 1 (b0) and
    // 8 more (b1) of each 16-element k-step; zero for heads past G
    auto load_q = [&](const NsPiece& k, uint32_t (&f)[KS][NH][2]) {
        const __nv_bfloat16* qb = q + (((size_t)k.r * g.BW + k.b) * g.Hq + (size_t)k.h * G) * D + tig * 2;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
            const int hh = nh * 8 + gid;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                f[kk][nh][0] = hh < G ? __ldg(reinterpret_cast<const uint32_t*>(qb + hh * D + kk * 16)) : 0u;
                f[kk][nh][1] = hh < G ? __ldg(reinterpret_cast<const uint32_t*>(qb + hh * D + kk * 16 + 8)) : 0u;
            }
        }
    };

    // ---- request side: the next block to stage is block ib of piece it (coordinates ip) -
    int it = (int)blockIdx.x, ib = 0;
    uint32_t iseq = 0;  // blocks requested so far
    NsPiece ip = ns_piece_of(g, npc, it), inx = ip;
    int is_a, is_b, nx_a = 0, nx_b = 0;
    load_slots(ip, is_a, is_b);
    if (it + stride < ntasks) {
        inx = ns_piece_of(g, npc, it + stride);
        load_slots(inx, nx_a, nx_b);
    }
    bool ibad = false;
    auto check_slots = [&]() {  // piece ip, its slots in is_a / is_b
        ibad = __any_sync(0xffffffffu, (lane < ip.n && (is_a < 0 || is_a >= g.S)) ||
                                           (lane + 32 < ip.n && (is_b < 0 || is_b >= g.S)));
        if (ibad && lane == 0) set_status(status, XATTN_STATUS_BAD_SLOT);
    };
    auto request_block = [&]() {  // it < ntasks
        const int buf = (int)(iseq % kRingBlocks);
        const int t0 = ib * kPieceBlk;
        const int cnt = min(kPieceBlk, ip.n - t0);
        // this lane's earlier shared-memory accesses to the buffer (MMA operand reads, the
        // zeroing below) are ordered before the copies that overwrite it
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) buf_bad[buf] = ibad ? 1 : 0;
        // position k of the block: lanes 0..15 copy its K row, 16..31 its V row, 16 bytes each
        if (!ibad) {
            const int ch = lane & 15;
            for (int k = 0; k < cnt; ++k) {
                const int tk = t0 + k;
                const int sv = __shfl_sync(0xffffffffu, tk < 32 ? is_a : is_b, tk & 31);
                const size_t off = (((size_t)ip.r * g.S + sv) * g.Hkv + ip.h) * D;
                const __nv_bfloat16* src = (lane < 16 ? pool_k : pool_v) + off;
                uint8_t* dst = (lane < 16 ? k_sm : v_sm) + (buf * kPieceBlk + k) * RS;
                if (ch < RB / 16)
                    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(ptx::smem_addr(dst + ch * 16)),
                                 "l"(reinterpret_cast<const uint8_t*>(src) + ch * 16), "l"(l2_first) : "memory");
                if (RB / 16 > 16)
                    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(ptx::smem_addr(dst + (ch + 16) * 16)),
                                 "l"(reinterpret_cast<const uint8_t*>(src) + (ch + 16) * 16), "l"(l2_first) : "memory");
            }
        }
        // each lane's arrival completes once its copies have landed
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(&full[buf])) : "memory");
        if (cnt < kPieceBlk) {
            // V rows past the piece are read by the MMA with weight 0: make them 0
            for (int e = lane; e < (kPieceBlk - cnt) * (RB / 16); e += 32)
                *reinterpret_cast<uint4*>(v_sm + (buf * kPieceBlk + cnt + e / (RB / 16)) * RS + (e % (RB / 16)) * 16) =
                    make_uint4(0, 0, 0, 0);
        }
        ++iseq;
        if (++ib * kPieceBlk >= ip.n) {  // on to this warp's next piece
            ib = 0;
            it += stride;
            if (it < ntasks) {
                ip = inx;
                is_a = nx_a;
                is_b = nx_b;
                if (it + stride < ntasks) {
                    inx = ns_piece_of(g, npc, it + stride);
                    load_slots(inx, nx_a, nx_b);
                }
                check_slots();
            }
        }
    };

    // ---- compute side ---------------------------------------------------------------------
    uint32_t qf[KS][NH][2];
    NsPiece cp = ip;  // the piece being computed
    load_q(cp, qf);
    check_slots();
    for (int j = 0; j < kRingBlocks && it < ntasks; ++j) request_block();

    // per-lane ldmatrix row offsets. K as the A operand (positions x d): matrix i/8 of the
    // x4 load covers positions ((i/8)%2)*8.., d half (i/16). V^T as the A operand (d x
    // positions, read transposed): positions (i/16)*8.., d half (i/8)%2.
    const uint32_t k_addr = ptx::smem_addr(k_sm) + (((lane >> 3) & 1) * 8 + (lane & 7)) * RS + (lane >> 4) * 16;
    const uint32_t v_addr = ptx::smem_addr(v_sm) + ((lane >> 4) * 8 + (lane & 7)) * RS + ((lane >> 3) & 1) * 16;
    uint32_t cseq = 0;  // blocks computed so far
    bool ok = true;
#pragma unroll 1
    for (int ct = (int)blockIdx.x; ct < ntasks; ct += stride) {
        const bool has_next = ct + stride < ntasks;
        const NsPiece cn = has_next ? ns_piece_of(g, npc, ct + stride) : cp;
        // O^T: d rows mt*16 + gid (c0, c1) and + 8 (c2, c3), heads nh*8 + 2 tig + {0, 1}
        float o[KS][NH][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) o[mt][nh][0] = o[mt][nh][1] = o[mt][nh][2] = o[mt][nh][3] = 0.f;
        // running maximum and lane-partial sum of heads nh*8 + 2 tig + j
        float m[NH][2], l[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) m[nh][0] = m[nh][1] = -INFINITY, l[nh][0] = l[nh][1] = 0.f;
        bool bad = false;
        const int nbk = (cp.n + kPieceBlk - 1) / kPieceBlk;
#pragma unroll 1
        for (int cb = 0; cb < nbk; ++cb) {
            const int buf = (int)(cseq % kRingBlocks);
            if (!ptx::mbar_wait_all(&full[buf], (cseq / kRingBlocks) & 1, abort_sh)) { ok = false; break; }
            __syncwarp();  // the zero rows other lanes stored are visible to this lane's ldmatrix
            bad = bad || buf_bad[buf] != 0;
            const bool last = cb == nbk - 1;
            if (!bad) {
                const uint32_t kb_addr = k_addr + buf * kPieceBlk * RS, vb_addr = v_addr + buf * kPieceBlk * RS;
                // S^T = K Q^T: positions gid (c0, c1) and gid + 8 (c2, c3) of the block
                float s[NH][4];
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) s[nh][0] = s[nh][1] = s[nh][2] = s[nh][3] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    uint32_t ka[4];
                    ldsm_x4(kb_addr + kk * 32, ka);
#pragma unroll
                    for (int nh = 0; nh < NH; ++nh) mma16816(s[nh], ka, qf[kk][nh][0], qf[kk][nh][1]);
                }
                if (last && has_next) load_q(cn, qf);  // Q of the piece after this one
                const int lim = cp.n - cb * kPieceBlk;  // positions of the block in the piece
                uint32_t pb[NH][2];
                float al[NH][2];
                bool moved = false;
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nh][e] *= g.scale_log2;
                    if (lim < kPieceBlk) {  // ragged last block: positions past the piece get -inf
                        if (gid >= lim) s[nh][0] = s[nh][1] = -INFINITY;
                        if (gid + 8 >= lim) s[nh][2] = s[nh][3] = -INFINITY;
                    }
                    float p[4];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        // column maximum over the 16 positions (lanes of equal tig hold a column)
                        float bm = fmaxf(s[nh][j], s[nh][2 + j]);
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
                        const float mn = fmaxf(m[nh][j], bm);  // finite: the block's first position is in
                        al[nh][j] = ex2(m[nh][j] - mn);
                        moved = moved || al[nh][j] != 1.f;
                        m[nh][j] = mn;
                        p[j] = ex2(s[nh][j] - mn);
                        p[2 + j] = ex2(s[nh][2 + j] - mn);
                        l[nh][j] = l[nh][j] * al[nh][j] + (p[j] + p[2 + j]);
                    }
                    // P^T as the B operand: positions 2 tig.. (b0: 0..7, b1: 8..15) of head gid
                    pb[nh][0] = movmatrix_trans(pack_bf16(p[0], p[1]));
                    pb[nh][1] = movmatrix_trans(pack_bf16(p[2], p[3]));
                }
                // rescale O^T when a running maximum moved (a warp-uniform test)
                if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                        for (int nh = 0; nh < NH; ++nh) {
                            o[mt][nh][0] *= al[nh][0];
                            o[mt][nh][1] *= al[nh][1];
                            o[mt][nh][2] *= al[nh][0];
                            o[mt][nh][3] *= al[nh][1];
                        }
                }
                // O^T += V^T P^T
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t va[4];
                    ldsm_x4_trans(vb_addr + mt * 32, va);
#pragma unroll
                    for (int nh = 0; nh < NH; ++nh) mma16816(o[mt][nh], va, pb[nh][0], pb[nh][1]);
                }
            } else if (last && has_next) {
                load_q(cn, qf);
            }
            ++cseq;
            if (it < ntasks) request_block();  // refill the buffer just computed
        }
        if (!ok) break;

        // the piece's partial result: head nh*8 + 2 tig + j, d rows mt*16 + gid (+ 8)
        const size_t prow0 = (((size_t)cp.r * g.Hkv + cp.h) * g.pieces + g.nsplit + cp.c) * g.M + (size_t)cp.b * G;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float lt = l[nh][j];
                lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                const int hh = nh * 8 + tig * 2 + j;
                if (hh >= G) continue;
                const bool empty = !(lt > 0.f);
                const float inv = (empty || bad) ? 0.f : 1.f / lt;
                float* po = part_o + (prow0 + hh) * D + gid;
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    po[mt * 16] = o[mt][nh][j] * inv;
                    po[mt * 16 + 8] = o[mt][nh][2 + j] * inv;
                }
                if (gid == 0)
                    part_lse[prow0 + hh] =
                        bad ? __uint_as_float(kNaN) : (empty ? -INFINITY : (m[nh][j] + __log2f(lt)) * kLn2);
            }
        cp = cn;
    }
    if (!ok) {
        // a wait gave up: record it, then let the copies still in flight land (bounded)
        if (lane == 0) {
            set_status(status, XATTN_STATUS_TIMEOUT);
            for (uint32_t sq = cseq; sq < iseq; ++sq) ptx::mbar_wait(&full[sq % kRingBlocks], (sq / kRingBlocks) & 1, abort_sh);
        }
        __syncwarp();
    }
}

// Short Non-Shared part (the fused decode's common case: a few tokens per beam): one warp
// per (request, beam) for every KV head. The ancestry slots are the same for all heads, and
// a pool slot keeps its heads' rows contiguous, so after the one index load the warp copies
// the beam's whole Non-Shared K/V (step x Hkv rows each) and its Hq query rows into its own
// shared memory with cp.async in one round trip, then computes every head from there. Few,
// fat warps (under one wave) instead of one thin warp per head with its own dependent loads.
constexpr int kBeamWarps = 4;  // warps per CTA of ns_beam_kernel

// Shared memory of one warp of ns_beam_kernel: step x Hkv x {K, V} rows, then Hq rows of q.
inline size_t ns_beam_warp_bytes(const Geometry& g) {
    return ((size_t)g.step * g.Hkv * 2 + g.Hq) * g.d * 2;
}

template <int D, int G>
__global__ void __launch_bounds__(kBeamWarps * 32) ns_beam_kernel(
    Geometry g, int warp_bytes, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ pool_k,
    const __nv_bfloat16* __restrict__ pool_v, const int32_t* __restrict__ idx, float* __restrict__ part_o,
    float* __restrict__ part_lse, int32_t* status) {
    constexpr int HG = G < 4 ? G : 4;  // query heads per pass
    constexpr int LP = 32 / HG;        // lanes per query head
    constexpr int EL = D / LP;         // elements of d per lane (2 .. 16)
    constexpr int NV = EL / 2;         // bf16 pairs per lane
    constexpr int RB = D * 2;          // bytes of one row (one head)
    constexpr int CH = RB / 16;        // 16-byte chunks per row
    extern __shared__ __align__(16) uint8_t dsm[];
    // the Shared-stage kernel that follows may start its CTAs now (it waits for this one's
    // completion before reading its output)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const long w = (long)blockIdx.x * kBeamWarps + wib;
    if (w >= (long)g.R * g.BW) return;
    const int b = (int)(w % g.BW), r = (int)(w / g.BW);
    const int T = g.step, Hkv = g.Hkv;
    uint8_t* wsm = dsm + (size_t)wib * warp_bytes;
    const uint32_t wsm_s = (uint32_t)__cvta_generic_to_shared(wsm);
    const int kv_bytes = T * Hkv * 2 * RB;  // then the q rows

    const int32_t* row_idx = idx + ((size_t)r * g.BW + b) * g.Tmax;
    const int my_slot = lane < T ? __ldg(row_idx + lane) : 0;
    const bool slot_bad = __any_sync(0xffffffffu, lane < T && (my_slot < 0 || my_slot >= g.S));
    if (slot_bad && lane == 0) set_status(status, XATTN_STATUS_BAD_SLOT);
    {   // the beam's q rows (Hq rows, contiguous) and, per token, the K and V rows of all heads
        const uint8_t* qs = reinterpret_cast<const uint8_t*>(q + ((size_t)r * g.BW + b) * g.Hq * D);
        for (int e = lane; e < g.Hq * CH; e += 32) cp_async16(wsm_s + kv_bytes + e * 16, qs + e * 16);
        if (!slot_bad) {
            for (int t = 0; t < T; ++t) {
                const int slot = __shfl_sync(0xffffffffu, my_slot, t);
                const size_t off = ((size_t)r * g.S + slot) * Hkv * RB;  // bytes
                const uint8_t* ks = reinterpret_cast<const uint8_t*>(pool_k) + off;
                const uint8_t* vs = reinterpret_cast<const uint8_t*>(pool_v) + off;
                const uint32_t kd = wsm_s + (2 * t) * Hkv * RB, vd = wsm_s + (2 * t + 1) * Hkv * RB;
                for (int e = lane; e < Hkv * CH; e += 32) {
                    cp_async16(kd + e * 16, ks + e * 16);
                    cp_async16(vd + e * 16, vs + e * 16);
                }
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncwarp();
    }
    const int hg = lane / LP, sl = lane % LP;
    auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
    auto hi = [](uint32_t x) { return __uint_as_float(x & 0xffff0000u); };
    auto read_pairs = [](const uint8_t* p, uint32_t (&w)[NV]) {
        if constexpr (NV >= 4) {
#pragma unroll
            for (int k = 0; k < NV / 4; ++k) {
                const uint4 u = *reinterpret_cast<const uint4*>(p + k * 16);
                w[4 * k] = u.x; w[4 * k + 1] = u.y; w[4 * k + 2] = u.z; w[4 * k + 3] = u.w;
            }
        } else if constexpr (NV == 2) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            w[0] = u.x; w[1] = u.y;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(p);
        }
    };
#pragma unroll 1
    for (int h = 0; h < Hkv; ++h) {
#pragma unroll 1
        for (int pass = 0; pass < G / HG; ++pass) {
            const int gg = pass * HG + hg;
            uint32_t qw[NV];
            read_pairs(wsm + kv_bytes + (h * G + gg) * RB + sl * EL * 2, qw);
            float m = -INFINITY, l = 0.f, acc[EL];
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[e] = 0.f;
            if (!slot_bad) {
                for (int t = 0; t < T; ++t) {
                    uint32_t kw[NV], vw[NV];
                    read_pairs(wsm + ((2 * t) * Hkv + h) * RB + sl * EL * 2, kw);
                    read_pairs(wsm + ((2 * t + 1) * Hkv + h) * RB + sl * EL * 2, vw);
                    float sc = 0.f;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        sc = fmaf(lo(qw[k]), lo(kw[k]), sc);
                        sc = fmaf(hi(qw[k]), hi(kw[k]), sc);
                    }
#pragma unroll
                    for (int o = LP / 2; o > 0; o >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, o);
                    const float s2 = sc * g.scale_log2;
                    const float mn = fmaxf(m, s2);
                    const float alpha = ex2(m - mn), p = ex2(s2 - mn);
                    l = l * alpha + p;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        acc[2 * k] = fmaf(p, lo(vw[k]), acc[2 * k] * alpha);
                        acc[2 * k + 1] = fmaf(p, hi(vw[k]), acc[2 * k + 1] * alpha);
                    }
                    m = mn;
                }
            }
            const size_t prow = (((size_t)r * Hkv + h) * g.pieces + g.nsplit) * g.M + (size_t)b * G + gg;
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            float* po = part_o + prow * D + sl * EL;
            if constexpr (EL >= 4) {
#pragma unroll
                for (int k = 0; k < EL / 4; ++k)
                    reinterpret_cast<float4*>(po)[k] =
                        make_float4(acc[4 * k] * inv, acc[4 * k + 1] * inv, acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
            } else {
                *reinterpret_cast<float2*>(po) = make_float2(acc[0] * inv, acc[1] * inv);
            }
            if (sl == 0)
                part_lse[prow] = slot_bad ? __uint_as_float(kNaN) : (empty ? -INFINITY : (m + __log2f(l)) * kLn2);
        }
    }
}

// T: storage type of q and the pools (bf16, or fp32 inputs used unrounded).
template <int D, int G, typename T>
__global__ void __launch_bounds__(256) ns_merge_kernel(
    Geometry g, const T* __restrict__ q, const T* __restrict__ pool_k,
    const T* __restrict__ pool_v, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ shared_len, float* __restrict__ part_o,
    float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse,
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

    // The pieces' LSEs of the G rows, lane l holding piece l (of the first 32), loaded before the
    // Non-Shared walk so that their round trip overlaps it.
    const size_t unit = (size_t)r * g.Hkv + h;
    const int np = g.nsplit + g.ns_pieces;
    const size_t prow_b = unit * g.pieces * g.M + (size_t)b * G;  // piece c row gg: + c*M + gg
    float lc0[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
        lc0[gg] = (!bad && lane < np) ? __ldg(part_lse + prow_b + (size_t)lane * g.M + gg) : -INFINITY;

    RowState<E, G> st;
    st.init();
    bool slot_bad = false;
    if (g.ns_pieces == 0 && g.step > 0 && !bad && !ns_walk<D, G, T>(g, r, b, h, lane, q, pool_k, pool_v, idx, st, status)) {
        bad = true;
        slot_bad = true;
    }

    // Merge: fold every stored piece (prefix pieces, then Non-Shared pieces) into the
    // running state. A piece stores its normalised output o_c and natural-log lse_c; in
    // base 2 it contributes weight 2^(lse_c * log2 e) times o_c. First pass, the G rows
    // together: each lane keeps a running maximum and sum of its pieces' weights (pieces
    // c = l, l + 32, ...), then the warp combines them. Second pass, row by row: the weighted
    // outputs, eight pieces' rows in flight.
    if (!bad) {
        float pm[G], ps[G];
        bool nan_seen = false;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
            pm[gg] = -INFINITY;
            ps[gg] = 0.f;
        }
        for (int c = lane; c < np; c += 32) {
            float lc[G];
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
                lc[gg] = c < 32 ? lc0[gg] : __ldg(part_lse + prow_b + (size_t)c * g.M + gg);
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                nan_seen |= (lc[gg] != lc[gg]);
                const float sv = lc[gg] * kLog2e;
                if (sv > pm[gg]) {
                    ps[gg] = ps[gg] * ex2(pm[gg] - sv) + 1.f;
                    pm[gg] = sv;
                } else if (sv > -INFINITY) {
                    ps[gg] += ex2(sv - pm[gg]);
                }
            }
        }
        if (__any_sync(0xffffffffu, nan_seen)) bad = true;  // a failed piece poisons the row
        if (!bad) {
#pragma unroll
            for (int gg = 0; gg < G; ++gg) {
                float mp = pm[gg];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
                const float mx = fmaxf(st.m[gg], mp);
                if (mx == -INFINITY) continue;  // nothing at all for this row
                const float lsum = warp_sum(pm[gg] > -INFINITY ? ps[gg] * ex2(pm[gg] - mx) : 0.f);
                const float alpha = ex2(st.m[gg] - mx);  // rescale the Non-Shared state
                float acc[E];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = st.acc[gg][e] * alpha;
                for (int c0 = 0; c0 < np; c0 += 32) {
                    const int c = c0 + lane;
                    const float lc = c0 == 0 ? lc0[gg]
                                             : (c < np ? __ldg(part_lse + prow_b + (size_t)c * g.M + gg) : -INFINITY);
                    const float wl = lc > -INFINITY ? ex2(lc * kLog2e - mx) : 0.f;
                    const int nc = min(32, np - c0);
                    for (int u0 = 0; u0 < nc; u0 += 8) {
                        float ov[8][E], wv[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int cu = u0 + u;
                            wv[u] = __shfl_sync(0xffffffffu, wl, cu & 31);
                            if (cu < nc) {
                                const float* po = part_o + (prow_b + (size_t)(c0 + cu) * g.M + gg) * D + lane * E;
                                if constexpr (E == 4) {
                                    const float4 t = __ldg(reinterpret_cast<const float4*>(po));
                                    ov[u][0] = t.x; ov[u][1] = t.y; ov[u][2] = t.z; ov[u][3] = t.w;
                                } else {
                                    const float2 t = __ldg(reinterpret_cast<const float2*>(po));
                                    ov[u][0] = t.x; ov[u][1] = t.y;
                                }
                            } else {
                                wv[u] = 0.f;
#pragma unroll
                                for (int e = 0; e < E; ++e) ov[u][e] = 0.f;
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u)
#pragma unroll
                            for (int e = 0; e < E; ++e) acc[e] = fmaf(wv[u], wv[u] != 0.f ? ov[u][e] : 0.f, acc[e]);
                    }
                }
                st.l[gg] = st.l[gg] * alpha + lsum;
#pragma unroll
                for (int e = 0; e < E; ++e) st.acc[gg][e] = acc[e];
                st.m[gg] = mx;
            }
        }
    }

#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        float o[E];
        float row_lse;
        if (bad || !(st.l[gg] > 0.f)) {
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = __uint_as_float(kNaN);
            row_lse = __uint_as_float(kNaN);
        } else {
            const float inv = 1.f / st.l[gg];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = st.acc[gg][e] * inv;
            row_lse = (st.m[gg] + __log2f(st.l[gg])) * kLn2;
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

// Row-parallel merge for calls whose Non-Shared part is already in pieces: one warp per
// query row (r, b, h) folds every piece, lanes splitting the head dimension. The row's loads
// are issued without waiting on one another: the LSEs of up to 64 pieces stay in registers
// (lane l: pieces l and l + 32) and reach the other lanes by shuffles, and the output
// vectors of a batch of pieces are requested while the previous batch is folded, whatever
// the pieces' weights (a piece without keys has weight 0 and its vector is never used).
template <int D>
__global__ void __launch_bounds__(256) merge_rows_kernel(
    Geometry g, const int32_t* __restrict__ shared_len, const float* __restrict__ part_o,
    const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse, int32_t* status) {
    constexpr int E = D / 32;
    constexpr int B = 8;  // output vectors per batch
    const int lane = threadIdx.x & 31;
    const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // (r*BW + b)*Hq + hq
    if (row >= (long)g.R * g.BW * g.Hq) return;
    const int hq = (int)(row % g.Hq);
    const int b = (int)((row / g.Hq) % g.BW);
    const int r = (int)(row / ((long)g.Hq * g.BW));
    const int h = hq / g.G, gg = hq - h * g.G;
    const int L = shared_len ? shared_len[r] : 0;
    bool bad = (g.Lmax > 0) && (L < 0 || L > g.Lmax);
    if (bad && lane == 0 && hq == 0 && b == 0) set_status(status, XATTN_STATUS_BAD_SHARED_LEN);
    const int np = g.nsplit + g.ns_pieces;
    const size_t prow_b = ((size_t)r * g.Hkv + h) * g.pieces * g.M + (size_t)b * g.G + gg;  // + c*M
    auto load_o = [&](int c, float (&v)[E]) {  // this lane's slice of piece c's output (0 past np)
        if (c < np) {
            const float* po = part_o + (prow_b + (size_t)c * g.M) * D + lane * E;
            if constexpr (E == 4) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(po));
                v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
            } else {
                const float2 t = __ldg(reinterpret_cast<const float2*>(po));
                v[0] = t.x; v[1] = t.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = 0.f;
        }
    };
    float ov[2][B][E];
#pragma unroll
    for (int k = 0; k < B; ++k) load_o(k, ov[0][k]);  // the first batch rides with the LSEs
    const float lc0 = lane < np ? __ldg(part_lse + prow_b + (size_t)lane * g.M) : -INFINITY;
    const float lc1 = lane + 32 < np ? __ldg(part_lse + prow_b + (size_t)(lane + 32) * g.M) : -INFINITY;
    bool nan_seen = (lc0 != lc0) || (lc1 != lc1);
    float mx = fmaxf(lc0, lc1) * kLog2e;
    for (int c = lane + 64; c < np; c += 32) {
        const float lc = __ldg(part_lse + prow_b + (size_t)c * g.M);
        nan_seen |= (lc != lc);
        mx = fmaxf(mx, lc * kLog2e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    bad = bad || __any_sync(0xffffffffu, nan_seen);
    // weights (base 2, relative to the row maximum) of pieces lane and lane + 32
    const float w0 = lc0 > -INFINITY ? ex2(lc0 * kLog2e - mx) : 0.f;
    const float w1 = lc1 > -INFINITY ? ex2(lc1 * kLog2e - mx) : 0.f;
    float lsum = w0 + w1;
    for (int c = lane + 64; c < np; c += 32) {
        const float lc = __ldg(part_lse + prow_b + (size_t)c * g.M);
        lsum += lc > -INFINITY ? ex2(lc * kLog2e - mx) : 0.f;
    }
    lsum = warp_sum(lsum);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < np; c0 += 2 * B) {
        // two batches per trip so that the double buffer is indexed statically
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int cb = c0 + half * B;
            if (cb >= np) break;
#pragma unroll
            for (int k = 0; k < B; ++k) load_o(cb + B + k, ov[half ^ 1][k]);  // next batch in flight
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const int c = cb + k;
                float w = __shfl_sync(0xffffffffu, c < 32 ? w0 : w1, c & 31);
                if (c >= 64 && c < np) {
                    const float lc = __ldg(part_lse + prow_b + (size_t)c * g.M);
                    w = lc > -INFINITY ? ex2(lc * kLog2e - mx) : 0.f;
                }
                if (c >= np) w = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = w > 0.f ? fmaf(w, ov[half][k][e], acc[e]) : acc[e];
            }
        }
    }
    bad = bad || !(lsum > 0.f);
    const float inv = bad ? __uint_as_float(kNaN) : 1.f / lsum;
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = acc[e] * inv;
    if (g.out_f32) {
        float* dst = reinterpret_cast<float*>(out) + (size_t)row * D + lane * E;
        if constexpr (E == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
        }
    } else {
        LaneVec<D>::store(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)row * D + lane * E, o);
    }
    if (lane == 0) lse[row] = bad ? __uint_as_float(kNaN) : (mx + __log2f(lsum)) * kLn2;
}

// Row merge for rows of at most kMergeFew pieces (a prefix in a few pieces and a short
// Non-Shared part): every piece's LSE and output vector requested at once, one round trip per
// row, in few enough registers that four CTAs fit on an SM (twice the rows in flight of the
// batched form, whose double buffer the long rows need).
constexpr int kMergeFew = 8;
template <int D>
__global__ void __launch_bounds__(256, 4) merge_rows_few_kernel(
    Geometry g, const int32_t* __restrict__ shared_len, const float* __restrict__ part_o,
    const float* __restrict__ part_lse, void* __restrict__ out, float* __restrict__ lse, int32_t* status) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // (r*BW + b)*Hq + hq
    if (row >= (long)g.R * g.BW * g.Hq) return;
    const int hq = (int)(row % g.Hq);
    const int b = (int)((row / g.Hq) % g.BW);
    const int r = (int)(row / ((long)g.Hq * g.BW));
    const int h = hq / g.G, gg = hq - h * g.G;
    const int L = shared_len ? shared_len[r] : 0;
    bool bad = (g.Lmax > 0) && (L < 0 || L > g.Lmax);
    if (bad && lane == 0 && hq == 0 && b == 0) set_status(status, XATTN_STATUS_BAD_SHARED_LEN);
    const int np = g.nsplit + g.ns_pieces;  // <= kMergeFew (checked on the host)
    const size_t prow_b = ((size_t)r * g.Hkv + h) * g.pieces * g.M + (size_t)b * g.G + gg;  // + c*M
    float ov[kMergeFew][E];
#pragma unroll
    for (int c = 0; c < kMergeFew; ++c) {
        if (c < np) {
            const float* po = part_o + (prow_b + (size_t)c * g.M) * D + lane * E;
            if constexpr (E == 4) {
                const float4 t = __ldg(reinterpret_cast<const float4*>(po));
                ov[c][0] = t.x; ov[c][1] = t.y; ov[c][2] = t.z; ov[c][3] = t.w;
            } else {
                const float2 t = __ldg(reinterpret_cast<const float2*>(po));
                ov[c][0] = t.x; ov[c][1] = t.y;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) ov[c][e] = 0.f;
        }
    }
    const float lc = lane < np ? __ldg(part_lse + prow_b + (size_t)lane * g.M) : -INFINITY;
    bad = bad || __any_sync(0xffffffffu, lc != lc);
    float mx = lc * kLog2e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float w = lc > -INFINITY ? ex2(lc * kLog2e - mx) : 0.f;  // piece `lane`'s weight
    const float lsum = warp_sum(w);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int c = 0; c < kMergeFew; ++c) {
        const float wc = __shfl_sync(0xffffffffu, w, c);  // 0 past np
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = wc > 0.f ? fmaf(wc, ov[c][e], acc[e]) : acc[e];
    }
    bad = bad || !(lsum > 0.f);
    const float inv = bad ? __uint_as_float(kNaN) : 1.f / lsum;
    float o[E];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = acc[e] * inv;
    if (g.out_f32) {
        float* dst = reinterpret_cast<float*>(out) + (size_t)row * D + lane * E;
        if constexpr (E == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
        }
    } else {
        LaneVec<D>::store(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)row * D + lane * E, o);
    }
    if (lane == 0) lse[row] = bad ? __uint_as_float(kNaN) : (mx + __log2f(lsum)) * kLn2;
}

// The row merge over nsplit + ns_pieces pieces per row, in the form that suits their number.
template <int D>
void launch_rows(const Geometry& g, cudaStream_t st, const int32_t* slen, const float* po, const float* pl,
                 void* out, float* lse, int32_t* status) {
    const unsigned rows_ctas = (unsigned)(((long)g.R * g.BW * g.Hq + 7) / 8);
    if (g.nsplit + g.ns_pieces <= kMergeFew)
        merge_rows_few_kernel<D><<<rows_ctas, 256, 0, st>>>(g, slen, po, pl, out, lse, status);
    else
        merge_rows_kernel<D><<<rows_ctas, 256, 0, st>>>(g, slen, po, pl, out, lse, status);
}

constexpr int kNsBeamMaxTok = 8;                 // tokens per beam for ns_beam_kernel
constexpr size_t kNsBeamMaxWarpBytes = 48 * 1024;  // its shared memory per warp

template <int D, int G>
cudaError_t launch_beam(const Geometry& g, cudaStream_t st, const __nv_bfloat16* q, const __nv_bfloat16* pk,
                        const __nv_bfloat16* pv, const int32_t* idx, float* po, float* pl, int32_t* status) {
    const int wb = (int)ns_beam_warp_bytes(g);
    const int smem = kBeamWarps * wb;
    static int attr_set[64] = {};  // dynamic shared-memory limit raised, per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || attr_set[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(ns_beam_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kBeamWarps * (int)kNsBeamMaxWarpBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = kBeamWarps * (int)kNsBeamMaxWarpBytes;
    }
    const unsigned ctas = (unsigned)(((long)g.R * g.BW + kBeamWarps - 1) / kBeamWarps);
    ns_beam_kernel<D, G><<<ctas, kBeamWarps * 32, smem, st>>>(g, wb, q, pk, pv, idx, po, pl, status);
    return cudaSuccess;
}

// One wave of resident one-warp CTAs (fewer when there are fewer pieces).
template <int D, int G>
cudaError_t launch_piece(const Geometry& g, int npc, cudaStream_t st, const __nv_bfloat16* q, const __nv_bfloat16* pk,
                         const __nv_bfloat16* pv, const int32_t* idx, float* po, float* pl, int32_t* status,
                         bool equal_split) {
    const long ntasks = (long)g.R * g.BW * g.Hkv * npc;
    if (ntasks <= 0) return cudaSuccess;
    if (ntasks > 0x7fffffffL) return cudaErrorInvalidValue;
    const int smem = piece_smem_bytes(D);
    static int resident[64] = {};  // CTAs of one wave, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (resident[dev] == 0) {
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ns_piece_kernel<D, G>, 32, smem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        resident[dev] = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
    }
    // One wave of warps; with equal_split only as many as give every warp the same number of
    // pieces (no last round run by a few warps), which is faster when the warps start together;
    // when they start one after another behind a long kernel on another stream, the full wave
    // with the smaller last round is.
    const long per = (ntasks + resident[dev] - 1) / resident[dev];
    const int grid = equal_split ? (int)((ntasks + per - 1) / per)
                                 : (int)(ntasks < resident[dev] ? ntasks : resident[dev]);
    ns_piece_kernel<D, G><<<grid, 32, smem, st>>>(g, npc, (int)ntasks, q, pk, pv, idx, po, pl, status);
    return cudaSuccess;
}

template <int D>
cudaError_t launch_d(const Geometry& g, cudaStream_t st, const void* qv, const void* pkv, const void* pvv,
                     const int32_t* idx, const int32_t* slen, float* po, float* pl, void* out, float* lse,
                     int32_t* status, cudaEvent_t join, bool equal_split) {
    const dim3 grid((unsigned)(((long)g.R * g.BW * g.Hkv + 7) / 8)), block(256);
    if (g.in_f32) {
        // fp32 storage: the direct walk (step <= kNsDirectMax, checked on the host) and the merge
        if (g.ns_to_piece || g.ns_pieces > 0) return cudaErrorInvalidValue;
        const float* q = static_cast<const float*>(qv);
        const float* pk = static_cast<const float*>(pkv);
        const float* pv = static_cast<const float*>(pvv);
        switch (g.G) {
#define XATTN_G32(GV)                                                                                             \
    case GV:                                                                                                     \
        ns_merge_kernel<D, GV, float><<<grid, block, 0, st>>>(g, q, pk, pv, idx, slen, po, pl, out, lse, status); \
        break;
            XATTN_G32(1) XATTN_G32(2) XATTN_G32(4) XATTN_G32(8) XATTN_G32(16)
#undef XATTN_G32
            default: return cudaErrorInvalidValue;
        }
        return cudaGetLastError();
    }
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(qv);
    const __nv_bfloat16* pk = static_cast<const __nv_bfloat16*>(pkv);
    const __nv_bfloat16* pv = static_cast<const __nv_bfloat16*>(pvv);
    const int npc = g.ns_to_piece ? 1 : g.ns_pieces;  // Non-Shared pieces per (r, b, h)
    // short Non-Shared part ahead of the fused Shared stage: one warp per (request, beam)
    const bool beam_path = g.ns_to_piece && g.step <= kNsBeamMaxTok && ns_beam_warp_bytes(g) <= kNsBeamMaxWarpBytes;
    switch (g.G) {
#define XATTN_G(GV)                                                                                              \
    case GV:                                                                                                     \
        if (beam_path) {                                                                                         \
            cudaError_t e = launch_beam<D, GV>(g, st, q, pk, pv, idx, po, pl, status);                          \
            if (e != cudaSuccess) return e;                                                                      \
        } else if (g.ns_to_piece || g.ns_pieces > 0) {                                                           \
            cudaError_t e = launch_piece<D, GV>(g, npc, st, q, pk, pv, idx, po, pl, status, equal_split);      \
            if (e != cudaSuccess) return e;                                                                      \
            if (!g.ns_to_piece && join) {                                                                        \
                e = cudaStreamWaitEvent(st, join, 0);                                                            \
                if (e != cudaSuccess) return e;                                                                  \
            }                                                                                                    \
            if (!g.ns_to_piece) launch_rows<D>(g, st, slen, po, pl, out, lse, status);                        \
        } else {                                                                                                 \
            ns_merge_kernel<D, GV, __nv_bfloat16><<<grid, block, 0, st>>>(g, q, pk, pv, idx, slen, po, pl, out, lse, status); \
        }                                                                                                        \
        break;
        XATTN_G(1) XATTN_G(2) XATTN_G(4) XATTN_G(8) XATTN_G(16)
#undef XATTN_G
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

int merge_ctas_for(const Geometry& g) {
    // warp per (r, b, KV head), or per query row when the Non-Shared part is in pieces
    const long warps = (long)g.R * g.BW * (g.ns_pieces > 0 ? g.Hq : g.Hkv);
    return (int)((warps + 7) / 8);
}

cudaError_t launch_ns_merge(const Geometry& g, const void* q, const void* pool_k,
                            const void* pool_v, const int32_t* beam_tok_idx, const int32_t* shared_len,
                            const float* part_o, const float* part_lse, void* out, float* lse, int32_t* status,
                            cudaStream_t stream, cudaEvent_t join, bool equal_split) {
    float* po = const_cast<float*>(part_o);
    float* pl = const_cast<float*>(part_lse);
    if (g.d == 128)
        return launch_d<128>(g, stream, q, pool_k, pool_v, beam_tok_idx, shared_len, po, pl, out, lse, status, join, equal_split);
    if (g.d == 64)
        return launch_d<64>(g, stream, q, pool_k, pool_v, beam_tok_idx, shared_len, po, pl, out, lse, status, join, equal_split);
    return cudaErrorInvalidValue;
}

// The row merge alone over pieces 0 .. np-1 (the prefix pieces and the Non-Shared piece
// `nsplit` the Non-Shared kernel wrote with ns_to_piece).
cudaError_t launch_merge_rows(const Geometry& g, int np, const int32_t* shared_len, const float* part_o,
                              const float* part_lse, void* out, float* lse, int32_t* status, cudaStream_t stream) {
    Geometry gm = g;
    gm.ns_to_piece = 0;
    gm.ns_pieces = np - g.nsplit;  // the kernel folds nsplit + ns_pieces pieces
    if (gm.ns_pieces < 0 || np > g.pieces) return cudaErrorInvalidValue;
    if (g.d == 128) launch_rows<128>(gm, stream, shared_len, part_o, part_lse, out, lse, status);
    else if (g.d == 64) launch_rows<64>(gm, stream, shared_len, part_o, part_lse, out, lse, status);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace xattn
