// Host entry points of libxattn.so (see include/xattn.h): argument validation, the split
// plan of the Shared stage, TMA descriptors, and the launches. Nothing here allocates
// device memory or synchronises (except xattn_read_status).
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "xattn_internal.cuh"

namespace xattn {
namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int device_sms() {
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;  // no device: plan as for a GB300
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult qr;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Shape checks shared by every entry point. Returns XATTN_OK or an error code.
int check_desc(const xattn_desc* d) {
    if (!d) return XATTN_ERR_INVALID_ARG;
    if (d->num_requests <= 0 || d->beam_width <= 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0)
        return XATTN_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads != 0) return XATTN_ERR_INVALID_ARG;
    if (d->max_shared_len < 0 || d->ns_slots < 0 || d->max_steps < 0) return XATTN_ERR_INVALID_ARG;
    if (!(d->softmax_scale >= 0.f) || !std::isfinite(d->softmax_scale)) return XATTN_ERR_INVALID_ARG;
    if (d->split_tokens < 0 || d->split_tokens % kPieceGrain != 0) return XATTN_ERR_INVALID_ARG;
    if (d->shared_kernel < 0 || d->shared_kernel > 2) return XATTN_ERR_INVALID_ARG;
    if (d->dtype != XATTN_DTYPE_BF16 && d->dtype != XATTN_DTYPE_F32) return XATTN_ERR_UNSUPPORTED;
    // fp32 inputs: the Shared stage on CUDA cores or on the tf32 tensor-core kernel; the
    // Non-Shared part by the direct walk of at most kNsDirectMax tokens
    if (d->dtype == XATTN_DTYPE_F32 && d->max_steps > kNsDirectMax) return XATTN_ERR_UNSUPPORTED;
    if (d->out_dtype != XATTN_DTYPE_BF16 && d->out_dtype != XATTN_DTYPE_F32) return XATTN_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return XATTN_ERR_UNSUPPORTED;
    const int G = d->num_q_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return XATTN_ERR_UNSUPPORTED;
    // Index arithmetic inside the kernels uses 32-bit products of these.
    const int64_t rows = (int64_t)d->num_requests * d->beam_width * d->num_q_heads;
    if (rows > (1ll << 30) || (int64_t)d->beam_width * G > (1ll << 24)) return XATTN_ERR_UNSUPPORTED;
    if ((int64_t)d->beam_width * d->max_steps > (1ll << 30)) return XATTN_ERR_UNSUPPORTED;
    if (d->max_shared_len > (1 << 30) || d->ns_slots > (1 << 30)) return XATTN_ERR_UNSUPPORTED;
    return XATTN_OK;
}

int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Split plan of the Shared stage. A piece is a run of whole 128-token tiles. The automatic
// choice minimises (waves of CTAs) x (tiles per CTA + one tile of fixed cost per CTA), so
// that short units are split until they fill the GPU but not beyond. with_ns: the plan of a
// whole decode (xattn_decode, xattn_decode_step), which also weighs a long Non-Shared part
// run beside the Shared stage; without it (xattn_decode_shared and xattn_decode_merge, whose
// pieces must agree whatever the step) the split does not depend on the step.
void plan(const xattn_desc* d, int step, Geometry* g, int* kernel, bool with_ns = true) {
    g->R = d->num_requests;
    g->BW = d->beam_width;
    g->Hq = d->num_q_heads;
    g->Hkv = d->num_kv_heads;
    g->G = g->Hq / g->Hkv;
    g->d = d->head_dim;
    g->Lmax = d->max_shared_len;
    g->S = d->ns_slots;
    g->Tmax = d->max_steps;
    g->step = step;
    g->M = g->BW * g->G;
    g->row_tiles = cdiv(g->M, kTileRows);
    const float scale = d->softmax_scale > 0.f ? d->softmax_scale : 1.0f / std::sqrt((float)g->d);
    g->scale_log2 = scale * 1.4426950408889634f;
    g->out_f32 = d->out_dtype == XATTN_DTYPE_F32 ? 1 : 0;
    g->in_f32 = d->dtype == XATTN_DTYPE_F32 ? 1 : 0;

    // Tensor cores by default, even for few stacked rows: a 128-row tile that is mostly
    // padding still streams the prefix at HBM speed (the MMA and exp work hide under the
    // loads), which the CUDA-core kernel does not reach. The CUDA-core kernel stays
    // selectable (shared_kernel = 2).
    // fp32 storage: CUDA cores by default (fp32 arithmetic throughout), the tf32 tensor-core
    // kernel (3) when asked for tensor cores.
    int k = 0;
    if (g->Lmax > 0) k = g->in_f32 ? (d->shared_kernel == 1 ? 3 : 2) : (d->shared_kernel ? d->shared_kernel : 1);
    *kernel = k;
    const int tiles = g->Lmax > 0 ? cdiv(g->Lmax, kPieceGrain) : 1;
    if (d->split_tokens > 0) {
        g->split_tokens = d->split_tokens;
    } else if (k == 0) {
        g->split_tokens = kPieceGrain;
    } else {
        // tensor-core CTAs own two 128-row tiles (tf32: one); CUDA-core CTAs own four rows
        const int64_t units =
            (int64_t)g->R * g->Hkv * (k == 1 ? cdiv(g->row_tiles, 2) : (k == 3 ? g->row_tiles : cdiv(g->M, 4)));
        const int64_t slots = (int64_t)device_sms() * (k == 2 ? 8 : 1);
        int best_n = 1;
        double best = 1e30;
        for (int n = 1; n <= tiles; ++n) {
            const int per = cdiv(tiles, n);
            if (n > 1 && cdiv(tiles, per) != n) continue;  // same pieces as a smaller n
            const double waves = (double)cdiv(units * n, slots);
            const double cost = waves * (per + 1.0) + 0.02 * n;  // small charge for merge traffic
            if (cost < best) { best = cost; best_n = n; }
        }
        // A long Non-Shared part (its own piece kernel, bf16) runs beside the tensor-core Shared
        // stage on the SMs that stage leaves free. In units of one 128-key tile of a Shared-stage
        // CTA (about 1.75 us): the Shared stage takes its waves x (tiles per CTA + about 5 for
        // the prologue and epilogue); the piece kernel's work is its pool bytes at about
        // 4.4 TB/s, done at the free SMs' share of that rate while the Shared stage runs and at
        // the full rate after it. The step ends with the later of the two. Never more pieces
        // than without the Non-Shared part (the workspace is sized by the plan of step 0).
        if (with_ns && k == 1 && !g->in_f32 && step > kNsDirectMax) {
            const double ns_units = (double)g->R * g->BW * step * g->Hkv * g->d * 2 * 2 / 4.4e12 / 1.75e-6;
            const int base_n = best_n;
            best = 1e30;
            for (int n = 1; n <= base_n; ++n) {
                const int per = cdiv(tiles, n);
                if (n > 1 && cdiv(tiles, per) != n) continue;
                const double waves = (double)cdiv(units * n, slots);
                const double t_sh = waves * (per + 5.0);
                const double free_frac = waves > 1.0 ? 0.0 : 1.0 - (double)(units * n) / (double)slots;
                const double during = t_sh * free_frac;
                const double t_ns = ns_units <= during ? ns_units / free_frac : t_sh + (ns_units - during);
                const double cost = (t_sh > t_ns ? t_sh : t_ns) + 0.02 * n;
                if (cost < best) { best = cost; best_n = n; }
            }
        }
        g->split_tokens = cdiv(tiles, best_n) * kPieceGrain;
    }
    g->nsplit = g->Lmax > 0 ? cdiv(g->Lmax, g->split_tokens) : 0;
    g->ns_pieces = step > kNsDirectMax ? cdiv(step, kNsChunk) : 0;
    g->pieces = g->nsplit + (g->Tmax > kNsDirectMax ? cdiv(g->Tmax, kNsChunk) : (g->Tmax > 0 ? 1 : 0));
    g->ns_to_piece = 0;
}

size_t workspace_bytes_for(const Geometry& g) {
    const size_t rows = part_rows(g);
    return kStatusBytes + rows * (size_t)g.d * sizeof(float) + ((rows * sizeof(float) + 255) / 256) * 256;
}

CUresult make_kv_map(CUtensorMap* map, const void* base, const Geometry& g) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_FOUND;
    // [R, Lmax, Hkv, d] viewed innermost-first as {d, Hkv, Lmax, R}; box = 64 x 1 x 128 x 1.
    cuuint64_t dims[4] = {(cuuint64_t)g.d, (cuuint64_t)g.Hkv, (cuuint64_t)g.Lmax, (cuuint64_t)g.R};
    cuuint64_t strides[3] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.Hkv * g.d * 2, (cuuint64_t)g.Lmax * g.Hkv * g.d * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)kTcTileKeys, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Q [R, BW, Hq, d] viewed innermost-first as {d, Hq, BW, R}; box = 64 x G x (128 / G) x 1:
// the 128 stacked rows (beam, query head of KV head h) of one row tile, row m = b*G + g
// (G is a power of two up to 16, so it divides 128).

CUresult make_q_map(CUtensorMap* map, const void* base, const Geometry& g) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[4] = {(cuuint64_t)g.d, (cuuint64_t)g.Hq, (cuuint64_t)g.BW, (cuuint64_t)g.R};
    cuuint64_t strides[3] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.Hq * g.d * 2, (cuuint64_t)g.BW * g.Hq * g.d * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)g.G, (cuuint32_t)(kTileRows / g.G), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// part_o [rows, d] fp32 viewed as {d, rows}; box = 32 x 128 (128 bytes x 128 rows, 128-byte
// swizzle): a quarter of the d columns of one 128-row tile of a piece, for the fused
// epilogue's staging of the Non-Shared piece in shared memory.
CUresult make_ns_map(CUtensorMap* map, const void* part_o, const Geometry& g) {
    auto enc = tensor_map_encoder();
    if (!enc) return CUDA_ERROR_NOT_FOUND;
    cuuint64_t dims[2] = {(cuuint64_t)g.d, (cuuint64_t)part_rows(g)};
    cuuint64_t strides[1] = {(cuuint64_t)g.d * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)kTileRows};
    cuuint32_t es[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(part_o), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace
}  // namespace xattn

using namespace xattn;

extern "C" {

size_t xattn_decode_workspace_size(const xattn_desc* desc) {
    if (check_desc(desc) != XATTN_OK) return 0;
    Geometry g;
    int k;
    plan(desc, 0, &g, &k);
    return workspace_bytes_for(g);
}

int xattn_query_plan(const xattn_desc* desc, int32_t step, xattn_plan* out) {
    int rc = check_desc(desc);
    if (rc != XATTN_OK) return rc;
    if (!out || step < 0 || step > desc->max_steps) return XATTN_ERR_INVALID_ARG;
    Geometry g;
    int k;
    plan(desc, step, &g, &k);
    *out = xattn_plan{};
    out->shared_kernel = k;
    out->num_splits = g.nsplit;
    out->split_tokens = g.split_tokens;
    out->rows_per_unit = g.M;
    out->row_tiles = g.row_tiles;
    out->shared_ctas = k == 0   ? 0
                       : k == 1 ? shared_tc_ctas_for(g)
                       : k == 3 ? g.R * g.Hkv * g.row_tiles * g.nsplit
                                : g.R * g.Hkv * ((g.M + 3) / 4) * g.nsplit;
    out->fused = decode_is_fused(g, k, step) ? 1 : 0;
    out->ns_tile = ns_tile_fits(g, k, step) ? 1 : 0;
    out->piece_stride = g.pieces;
    out->merge_ctas = out->fused ? 0 : merge_ctas_for(g);
    return XATTN_OK;
}

}  // extern "C"

namespace {

int check_common(const xattn_desc* desc, const void* q, void* workspace) {
    int rc = check_desc(desc);
    if (rc != XATTN_OK) return rc;
    if (!q || !workspace) return XATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(workspace, 256)) return XATTN_ERR_MISALIGNED;
    return XATTN_OK;
}

int check_shared_args(const xattn_desc* desc, const void* shared_k, const void* shared_v,
                      const int32_t* shared_len) {
    if (desc->max_shared_len == 0) return XATTN_OK;
    if (!shared_k || !shared_v || !shared_len) return XATTN_ERR_INVALID_ARG;
    if (!aligned(shared_k, 16) || !aligned(shared_v, 16) || !aligned(shared_len, 4)) return XATTN_ERR_MISALIGNED;
    return XATTN_OK;
}

int check_merge_args(const xattn_desc* desc, const void* ns_k_pool, const void* ns_v_pool,
                     const int32_t* beam_tok_idx, int32_t step, const void* out, const float* lse) {
    if (step < 0 || step > desc->max_steps) return XATTN_ERR_INVALID_ARG;
    if (step == 0 && desc->max_shared_len == 0) return XATTN_ERR_INVALID_ARG;
    if (step > 0 && (int64_t)step * desc->beam_width > desc->ns_slots) return XATTN_ERR_INVALID_ARG;
    if (!out || !lse) return XATTN_ERR_INVALID_ARG;
    if (step > 0 && (!ns_k_pool || !ns_v_pool || !beam_tok_idx)) return XATTN_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(lse, 4)) return XATTN_ERR_MISALIGNED;
    if (step > 0 && (!aligned(ns_k_pool, 16) || !aligned(ns_v_pool, 16) || !aligned(beam_tok_idx, 4)))
        return XATTN_ERR_MISALIGNED;
    return XATTN_OK;
}

struct WsView {
    int32_t* status;
    float* part_o;
    float* part_lse;
};

WsView ws_view(void* workspace, const Geometry& g) {
    WsView v;
    v.status = reinterpret_cast<int32_t*>(workspace);
    v.part_o = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + kStatusBytes);
    v.part_lse = v.part_o + part_rows(g) * g.d;
    return v;
}

// Shared stage; with `fused` (tensor-core kernel only) it also runs the Non-Shared stage and
// the Merge and writes out / lse.
int run_shared(const Geometry& g, int kernel, const void* q, const void* shared_k, const void* shared_v,
               const int32_t* shared_len, const WsView& ws, cudaStream_t st, bool fused = false,
               const void* ns_k_pool = nullptr, const void* ns_v_pool = nullptr,
               const int32_t* beam_tok_idx = nullptr, void* out = nullptr, float* lse = nullptr,
               bool ns_tile = false, const NsTileArgs* ns_args = nullptr) {
    cudaError_t e = cudaSuccess;
    if (kernel == 1) {
        auto qb = reinterpret_cast<const __nv_bfloat16*>(q);
        CUtensorMap mk, mv, mq, mn;
        if (make_kv_map(&mk, shared_k, g) != CUDA_SUCCESS || make_kv_map(&mv, shared_v, g) != CUDA_SUCCESS)
            return XATTN_ERR_CUDA;
        if (make_q_map(&mq, q, g) != CUDA_SUCCESS || make_ns_map(&mn, ws.part_o, g) != CUDA_SUCCESS)
            return XATTN_ERR_CUDA;
        NsTileArgs nst{ns_tile, ns_k_pool, ns_v_pool, beam_tok_idx, false};
        if (ns_args) nst = *ns_args;
        e = launch_shared_stage_tc(g, mk, mv, mq, mn, qb, shared_len, ws.part_o, ws.part_lse, ws.status, out, lse,
                                   fused, nst, st);
    } else if (kernel == 2) {
        e = launch_shared_stage_simt(g, q, shared_k, shared_v, shared_len, ws.part_o, ws.part_lse, ws.status, st,
                                     ns_args && ns_args->pdl, ns_args ? ns_args->started : nullptr);
    } else if (kernel == 3) {
        e = launch_shared_stage_tf32(g, q, shared_k, shared_v, shared_len, ws.part_o, ws.part_lse, ws.status, st,
                                     ns_args && ns_args->pdl);
    }
    return e == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

int run_merge(const Geometry& g, const xattn_desc* desc, const void* q, const int32_t* shared_len,
              const void* ns_k_pool, const void* ns_v_pool, const int32_t* beam_tok_idx, void* out, float* lse,
              const WsView& ws, cudaStream_t st, cudaEvent_t join = nullptr, bool equal_split = true) {
    cudaError_t e = launch_ns_merge(g, q, ns_k_pool, ns_v_pool, beam_tok_idx,
                                    desc->max_shared_len > 0 ? shared_len : nullptr, ws.part_o, ws.part_lse,
                                    out, lse, ws.status, st, join, equal_split);
    return e == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

// A second stream and three events per host thread and device, created on first use and
// kept for the thread's lifetime: with a long Non-Shared part the Shared stage (prefix
// pieces) and the Non-Shared piece kernel do not depend on each other, so the Shared stage
// runs on this stream, forked from the caller's stream by one event and joined back by
// another before the row merge (graph capture follows the fork and the join). The third is
// recorded once every CTA of the Shared stage has begun. Per thread, so calls from different
// host threads never share one.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, started = nullptr;
    ~SideStream() {
        if (started) cudaEventDestroy(started);
        if (join) cudaEventDestroy(join);
        if (fork) cudaEventDestroy(fork);
        if (s) cudaStreamDestroy(s);
    }
};
SideStream* side_stream() {
    static thread_local SideStream tbl[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    SideStream& x = tbl[dev];
    if (!x.s) {
        if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess) {
            x.s = nullptr;
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&x.started, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
    }
    return (x.fork && x.join && x.started) ? &x : nullptr;
}

// Whether the decode takes the two-stream form: a prefix with storage, no fusion, bf16, and
// either a long Non-Shared part (its own piece kernel) or a short one next to a prefix cut in
// pieces (the Non-Shared part then written as one more piece and folded by the row merge).
bool decode_two_streams(const Geometry& g, int kernel, int step) {
    if (kernel == 0 || decode_is_fused(g, kernel, step) || g.in_f32) return false;
    return g.ns_pieces > 0 || (step > 0 && step <= kNsDirectMax && g.nsplit > 1);
}

// The Non-Shared part and the merge of the two-stream form, on `st`, the row merge after
// `join` (the Shared stage's completion on the side stream).
// started: when not null, the piece kernel waits for it (every CTA of the Shared stage has
// begun), so that its many small CTAs cannot take the SMs first and hold the Shared stage's
// one-per-SM CTAs back until they are done. xattn_decode uses it; in xattn_decode_step the
// beam update ahead of the piece kernel gives the Shared stage that head start, and a second
// dependency there made the wait last until the Shared stage's end.
int run_ns_then_merge(const Geometry& g, int kernel, const xattn_desc* desc, const void* q,
                      const int32_t* shared_len, const void* ns_k_pool, const void* ns_v_pool,
                      const int32_t* beam_tok_idx, void* out, float* lse, const WsView& ws, cudaStream_t st,
                      cudaEvent_t join, cudaEvent_t started) {
    if (g.ns_pieces > 0) {
        if (started && cudaStreamWaitEvent(st, started, 0) != cudaSuccess) {
            cudaStreamWaitEvent(st, join, 0);  // leave nothing of this call unjoined
            return XATTN_ERR_CUDA;
        }
        // the piece kernel, then (after the join) the row merge. The piece kernel's warps take an
        // equal number of pieces when the Shared stage beside it is short (one wave of at most 8
        // tiles per CTA): they then start together; behind a longer one they start one after
        // another as its CTAs end, and the full wave finishes sooner.
        const int sms = device_sms();
        const long ctas = kernel == 1 ? shared_tc_ctas_for(g) : 0;
        const long tiles = (g.split_tokens + kTcTileKeys - 1) / kTcTileKeys;
        const bool short_shared = kernel == 1 && tiles * ((ctas + sms - 1) / sms) <= 8;
        return run_merge(g, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws, st, join,
                         short_shared);
    }
    Geometry gn = g;
    gn.ns_to_piece = 1;  // the Non-Shared part as piece nsplit
    int rc = run_merge(gn, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws, st);
    if (cudaStreamWaitEvent(st, join, 0) != cudaSuccess && rc == XATTN_OK) rc = XATTN_ERR_CUDA;
    if (rc != XATTN_OK) return rc;
    const cudaError_t e = launch_merge_rows(g, g.nsplit + 1, desc->max_shared_len > 0 ? shared_len : nullptr,
                                            ws.part_o, ws.part_lse, out, lse, ws.status, st);
    return e == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

// The Shared stage forked onto the side stream; returns the event the row merge waits for, or
// null when the fork could not be made (then nothing was enqueued). *started: the event
// recorded once every CTA of the Shared stage has begun.
cudaEvent_t fork_shared(const Geometry& g, int kernel, const void* q, const void* shared_k, const void* shared_v,
                        const int32_t* shared_len, const WsView& ws, cudaStream_t st, int* rc,
                        cudaEvent_t* started) {
    *rc = XATTN_OK;
    SideStream* ss = side_stream();
    if (!ss) return nullptr;
    if (cudaEventRecord(ss->fork, st) != cudaSuccess || cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess) {
        *rc = XATTN_ERR_CUDA;
        return nullptr;
    }
    NsTileArgs launch{false, nullptr, nullptr, nullptr, false, ss->started};
    *rc = run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, ss->s, false, nullptr, nullptr, nullptr,
                     nullptr, nullptr, false, &launch);
    *started = ss->started;
    if (*rc == XATTN_OK && cudaEventRecord(ss->join, ss->s) != cudaSuccess) *rc = XATTN_ERR_CUDA;
    if (*rc != XATTN_OK) {
        // join whatever was enqueued before returning the error
        cudaEventRecord(ss->join, ss->s);
        cudaStreamWaitEvent(st, ss->join, 0);
        return nullptr;
    }
    return ss->join;
}

}  // namespace

// Every host-side check xattn_decode makes before it launches anything (descriptor, pointers,
// alignment, step, workspace size); nothing is enqueued.
int xattn::check_decode_args(const xattn_desc* desc, const void* q, const void* shared_k, const void* shared_v,
                             const int32_t* shared_len, const void* ns_k_pool, const void* ns_v_pool,
                             const int32_t* beam_tok_idx, int32_t step, const void* out, const float* lse,
                             const void* workspace, size_t workspace_bytes) {
    int rc = check_common(desc, q, const_cast<void*>(workspace));
    if (rc == XATTN_OK) rc = check_shared_args(desc, shared_k, shared_v, shared_len);
    if (rc == XATTN_OK) rc = check_merge_args(desc, ns_k_pool, ns_v_pool, beam_tok_idx, step, out, lse);
    if (rc != XATTN_OK) return rc;
    Geometry g;
    int kernel;
    plan(desc, step, &g, &kernel);
    return workspace_bytes < workspace_bytes_for(g) ? XATTN_ERR_WORKSPACE_TOO_SMALL : XATTN_OK;
}

extern "C" {

int xattn_decode(const xattn_desc* desc, const void* q, const void* shared_k, const void* shared_v,
                 const int32_t* shared_len, const void* ns_k_pool, const void* ns_v_pool,
                 const int32_t* beam_tok_idx, int32_t step, void* out, float* lse, void* workspace,
                 size_t workspace_bytes, xattn_stream_t stream) {
    int rc = xattn::check_decode_args(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx,
                                      step, out, lse, workspace, workspace_bytes);
    if (rc != XATTN_OK) return rc;
    Geometry g;
    int kernel;
    plan(desc, step, &g, &kernel);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WsView ws = ws_view(workspace, g);
    if (ns_tile_fits(g, kernel, step)) {
        // One launch: the Shared-stage kernel gathers the Non-Shared rows itself and attends to
        // them as the first tile of each row tile; its online softmax merges the two parts.
        return run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, true, ns_k_pool, ns_v_pool,
                          beam_tok_idx, out, lse, true);
    }
    if (decode_is_fused(g, kernel, step)) {
        // Non-Shared part first, as one piece in the workspace; then the Shared stage, whose
        // epilogue merges it and writes out / lse.
        if (step > 0) {
            Geometry gn = g;
            gn.ns_to_piece = 1;
            rc = run_merge(gn, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws, st);
            if (rc != XATTN_OK) return rc;
        }
        return run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, true, nullptr, nullptr, nullptr, out,
                          lse);
    }
    if (decode_two_streams(g, kernel, step)) {
        // the Shared stage beside the Non-Shared piece kernel; the row merge waits for both
        cudaEvent_t started = nullptr;
        cudaEvent_t join = fork_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, &rc, &started);
        if (rc != XATTN_OK) return rc;
        if (join)
            return run_ns_then_merge(g, kernel, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse,
                                     ws, st, join, started);
    }
    rc = run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st);
    if (rc != XATTN_OK) return rc;
    return run_merge(g, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws, st);
}

int xattn_decode_step(const xattn_desc* desc, const int32_t* parent, const void* new_k, const void* new_v,
                      const void* q, const void* shared_k, const void* shared_v, const int32_t* shared_len,
                      void* ns_k_pool, void* ns_v_pool, int32_t* beam_tok_idx, int32_t step, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, xattn_stream_t stream) {
    int rc = xattn::check_decode_args(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx,
                                      step, out, lse, workspace, workspace_bytes);
    if (rc != XATTN_OK) return rc;
    if (step < 1) return XATTN_ERR_INVALID_ARG;
    if (desc->beam_width > 8192) return XATTN_ERR_UNSUPPORTED;
    if (!new_k || !new_v || (step > 1 && !parent)) return XATTN_ERR_INVALID_ARG;
    if (!aligned(new_k, 16) || !aligned(new_v, 16) || (parent && !aligned(parent, 4))) return XATTN_ERR_MISALIGNED;
    Geometry g;
    int kernel;
    plan(desc, step, &g, &kernel);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const WsView ws = ws_view(workspace, g);
    if (decode_two_streams(g, kernel, step)) {
        // the Shared stage (which reads nothing the update writes) forked first, beside the
        // update and the Non-Shared piece kernel; the row merge waits for both
        cudaEvent_t started = nullptr;
        cudaEvent_t join = fork_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, &rc, &started);
        if (rc != XATTN_OK) return rc;
        if (join) {
            rc = xattn_beam_update(desc, parent, new_k, new_v, ns_k_pool, ns_v_pool, beam_tok_idx, step - 1,
                                   ws.status, stream);
            if (rc != XATTN_OK) {
                cudaStreamWaitEvent(st, join, 0);  // leave nothing of this call unjoined
                return rc;
            }
            return run_ns_then_merge(g, kernel, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse,
                                     ws, st, join, nullptr);
        }
    }
    rc = beam_update(desc, parent, new_k, new_v, ns_k_pool, ns_v_pool, beam_tok_idx, step - 1, ws.status, st, 4);
    if (rc != XATTN_OK) return rc;
    if (ns_tile_fits(g, kernel, step)) {
        // The decode as the beam update's programmatic dependent: its set-up, Q loads and first K/V
        // loads overlap the update; its gather waits for the update to complete.
        const NsTileArgs pdl{true, ns_k_pool, ns_v_pool, beam_tok_idx, true};
        return run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, true, ns_k_pool, ns_v_pool,
                          beam_tok_idx, out, lse, true, &pdl);
    }
    if (kernel != 0 && !decode_is_fused(g, kernel, step)) {
        // Shared stage (prefix pieces) as the beam update's programmatic dependent: it reads
        // nothing the update writes and runs beside it, waiting for it only at its end; then
        // the Non-Shared + Merge kernel(s).
        const NsTileArgs pdl{false, nullptr, nullptr, nullptr, true};
        rc = run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws, st, false, nullptr, nullptr, nullptr,
                        nullptr, nullptr, false, &pdl);
        if (rc != XATTN_OK) return rc;
        return run_merge(g, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws, st);
    }
    return xattn_decode(desc, q, shared_k, shared_v, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, step, out, lse,
                        workspace, workspace_bytes, stream);
}

int xattn_decode_shared(const xattn_desc* desc, const void* q, const void* shared_k, const void* shared_v,
                        const int32_t* shared_len, void* workspace, size_t workspace_bytes,
                        xattn_stream_t stream) {
    int rc = check_common(desc, q, workspace);
    if (rc == XATTN_OK && desc->max_shared_len == 0) rc = XATTN_ERR_INVALID_ARG;
    if (rc == XATTN_OK) rc = check_shared_args(desc, shared_k, shared_v, shared_len);
    if (rc != XATTN_OK) return rc;
    Geometry g;
    int kernel;
    plan(desc, 0, &g, &kernel);
    if (workspace_bytes < workspace_bytes_for(g)) return XATTN_ERR_WORKSPACE_TOO_SMALL;
    return run_shared(g, kernel, q, shared_k, shared_v, shared_len, ws_view(workspace, g),
                      reinterpret_cast<cudaStream_t>(stream));
}

int xattn_decode_merge(const xattn_desc* desc, const void* q, const int32_t* shared_len, const void* ns_k_pool,
                       const void* ns_v_pool, const int32_t* beam_tok_idx, int32_t step, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, xattn_stream_t stream) {
    int rc = check_common(desc, q, workspace);
    if (rc == XATTN_OK && desc->max_shared_len > 0 && !shared_len) rc = XATTN_ERR_INVALID_ARG;
    if (rc == XATTN_OK && shared_len && !aligned(shared_len, 4)) rc = XATTN_ERR_MISALIGNED;
    if (rc == XATTN_OK) rc = check_merge_args(desc, ns_k_pool, ns_v_pool, beam_tok_idx, step, out, lse);
    if (rc != XATTN_OK) return rc;
    Geometry g;
    int kernel;
    plan(desc, step, &g, &kernel, false);
    if (workspace_bytes < workspace_bytes_for(g)) return XATTN_ERR_WORKSPACE_TOO_SMALL;
    return run_merge(g, desc, q, shared_len, ns_k_pool, ns_v_pool, beam_tok_idx, out, lse, ws_view(workspace, g),
                     reinterpret_cast<cudaStream_t>(stream));
}

int xattn_beam_update(const xattn_desc* desc, const int32_t* parent, const void* new_k, const void* new_v,
                      void* ns_k_pool, void* ns_v_pool, int32_t* beam_tok_idx, int32_t step, int32_t* status,
                      xattn_stream_t stream) {
    return xattn::beam_update(desc, parent, new_k, new_v, ns_k_pool, ns_v_pool, beam_tok_idx, step, status,
                              reinterpret_cast<cudaStream_t>(stream), 4);
}

}  // extern "C"

int xattn::beam_update(const xattn_desc* desc, const int32_t* parent, const void* new_k, const void* new_v,
                       void* ns_k_pool, void* ns_v_pool, int32_t* beam_tok_idx, int32_t step, int32_t* status,
                       cudaStream_t stream, int vectors_per_thread) {
    int rc = check_desc(desc);
    if (rc != XATTN_OK) return rc;
    if (step < 0 || step >= desc->max_steps) return XATTN_ERR_INVALID_ARG;
    if ((int64_t)(step + 1) * desc->beam_width > desc->ns_slots) return XATTN_ERR_INVALID_ARG;
    if (desc->beam_width > 8192) return XATTN_ERR_UNSUPPORTED;
    if (!new_k || !new_v || !ns_k_pool || !ns_v_pool || !beam_tok_idx || (step > 0 && !parent))
        return XATTN_ERR_INVALID_ARG;
    if (!aligned(new_k, 16) || !aligned(new_v, 16) || !aligned(ns_k_pool, 16) || !aligned(ns_v_pool, 16) ||
        !aligned(beam_tok_idx, 4) || (parent && !aligned(parent, 4)) || (status && !aligned(status, 4)))
        return XATTN_ERR_MISALIGNED;
    cudaError_t e = launch_beam_update(
        desc->num_requests, desc->beam_width, desc->num_kv_heads, desc->head_dim,
        desc->dtype == XATTN_DTYPE_F32 ? 4 : 2, desc->ns_slots, desc->max_steps, step, parent, new_k, new_v,
        ns_k_pool, ns_v_pool, beam_tok_idx, status, stream, vectors_per_thread);
    return e == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

extern "C" {

int xattn_beam_select(int32_t num_requests, int32_t beam_width, int32_t cand_per_beam, int32_t out_width,
                      const float* beam_score, const float* cand_logp, const int32_t* cand_token, int32_t* parent,
                      int32_t* token, float* score, xattn_stream_t stream) {
    if (num_requests < 1 || beam_width < 1 || cand_per_beam < 1 || out_width < 1) return XATTN_ERR_INVALID_ARG;
    if ((int64_t)beam_width * cand_per_beam > (1ll << 30)) return XATTN_ERR_UNSUPPORTED;
    if (out_width > (int64_t)beam_width * cand_per_beam) return XATTN_ERR_INVALID_ARG;
    if (beam_width > 1024 || out_width > 1024) return XATTN_ERR_UNSUPPORTED;
    if (!beam_score || !cand_logp || !cand_token || !parent || !token || !score) return XATTN_ERR_INVALID_ARG;
    if (!aligned(beam_score, 4) || !aligned(cand_logp, 4) || !aligned(cand_token, 4) || !aligned(parent, 4) ||
        !aligned(token, 4) || !aligned(score, 4))
        return XATTN_ERR_MISALIGNED;
    cudaError_t e = launch_beam_select(num_requests, beam_width, cand_per_beam, out_width, beam_score, cand_logp,
                                       cand_token, parent, token, score, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

int xattn_read_status(void* workspace, int32_t* status_out, int32_t clear, xattn_stream_t stream) {
    if (!workspace || !status_out) return XATTN_ERR_INVALID_ARG;
    if (!aligned(workspace, 4)) return XATTN_ERR_MISALIGNED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(status_out, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return XATTN_ERR_CUDA;
    if (clear && cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return XATTN_ERR_CUDA;
    return cudaStreamSynchronize(st) == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

const char* xattn_status_string(int code) {
    switch (code) {
        case XATTN_OK: return "ok";
        case XATTN_ERR_INVALID_ARG: return "invalid argument";
        case XATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case XATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case XATTN_ERR_MISALIGNED: return "tensor not 16-byte aligned";
        case XATTN_ERR_CUDA: return "CUDA error";
        case XATTN_ERR_HOST_MEMORY: return "host allocation failed";
        default: return "unknown status";
    }
}

}  // extern "C"
