// Internal declarations shared by the kernels and the host entry points of libxattn.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/xattn.h"

namespace xattn {

constexpr int kTileRows = 128;   // rows of one tensor-core M tile (stacked beam x head rows)
constexpr int kPieceGrain = 128; // prefix pieces are whole multiples of this many tokens
constexpr int kTcTileKeys = 128; // prefix tokens per K/V tile of the tensor-core kernel (TMA box)
constexpr int kStatusBytes = 256;
constexpr int kNsDirectMax = 32;   // up to this many Non-Shared tokens the merge kernel walks them
constexpr int kNsChunk = 64;       // beyond it, pieces of this many tokens are computed in parallel

// Device status word helpers ----------------------------------------------------------
__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// Geometry of one decode call, precomputed on the host.
struct Geometry {
    int R, BW, Hq, Hkv, G, d;
    int Lmax, S, Tmax, step;
    int M;            // BW * G stacked rows per (request, KV head)
    int row_tiles;    // ceil(M / 128)
    int nsplit;       // prefix pieces
    int split_tokens; // tokens per piece (multiple of 128)
    float scale_log2; // softmax scale * log2(e)
    int out_f32;      // output dtype: 0 bf16, 1 fp32
    int ns_pieces;    // Non-Shared pieces of this call (0: the merge kernel walks the tokens)
    int pieces;       // piece stride of the workspace: nsplit + Non-Shared pieces for max_steps
    int ns_to_piece;  // ns_merge_kernel writes the Non-Shared part as piece `nsplit` (no merge)
    int in_f32;       // q, K and V stored as fp32 (CUDA-core kernels only), else bf16
};

// Workspace layout: [status (256 B)] [part_o: R*Hkv*pieces*M*d fp32] [part_lse: R*Hkv*pieces*M fp32].
// Pieces 0 .. nsplit-1 are the prefix pieces, nsplit .. the Non-Shared ones (one piece when
// the Non-Shared part is short, else one per kNsChunk ancestry positions).
inline size_t part_rows(const Geometry& g) { return (size_t)g.R * g.Hkv * g.pieces * g.M; }

// Launchers (each returns cudaGetLastError()).
// fused = the CTA merges its (whole-prefix) result with the Non-Shared piece already in the
// workspace and writes out / lse (requires a single prefix piece); otherwise it writes the
// piece's partial result into part_o / part_lse.
// tmap_q: the Q tiles by TMA (box 64 x G x 128/G; G divides 128 since it is a power of two
// up to 16); tmap_ns: part_o as {d, rows} fp32, box 32 x 128 (the fused epilogue stages the
// Non-Shared piece through it).
// ns_tile.enabled (with fused and g.step > 0): the kernel gathers the Non-Shared K/V rows
// itself (pool_k / pool_v through the ancestry table idx) and attends to them as one more
// 128-key tile per row tile; requires (128 / G) * step <= 128 (ns_tile_fits). pdl: launched
// as the programmatic dependent of the beam update just before it (its gather waits for it).
struct NsTileArgs {
    bool enabled;
    const void* pool_k;
    const void* pool_v;
    const int32_t* idx;
    bool pdl;
    cudaEvent_t started = nullptr;  // recorded once every CTA of the launch has begun (optional)
};
cudaError_t launch_shared_stage_tc(const Geometry& g, const CUtensorMap& tmap_k,
                                   const CUtensorMap& tmap_v, const CUtensorMap& tmap_q,
                                   const CUtensorMap& tmap_ns, const __nv_bfloat16* q,
                                   const int32_t* shared_len, float* part_o, float* part_lse,
                                   int32_t* status, void* out, float* lse, bool fused,
                                   const NsTileArgs& ns_tile, cudaStream_t stream);
// q, shared_k, shared_v: bf16, or fp32 when g.in_f32.
cudaError_t launch_shared_stage_simt(const Geometry& g, const void* q, const void* shared_k, const void* shared_v,
                                     const int32_t* shared_len, float* part_o, float* part_lse,
                                     int32_t* status, cudaStream_t stream, bool pdl = false,
                                     cudaEvent_t started = nullptr);
// Shared stage for fp32 storage on the tensor cores (tcgen05 kind::tf32), writing the same
// per-piece partials as launch_shared_stage_simt. pdl (both): launched as the programmatic
// dependent of the beam update just queued; the kernel completes only after it.
cudaError_t launch_shared_stage_tf32(const Geometry& g, const void* q, const void* shared_k, const void* shared_v,
                                     const int32_t* shared_len, float* part_o, float* part_lse, int32_t* status,
                                     cudaStream_t stream, bool pdl = false);
// q and the pools: bf16, or fp32 when g.in_f32 (then only the direct walk of at most
// kNsDirectMax Non-Shared tokens, which the host checks). join: with a long Non-Shared part,
// an event the row merge waits for after the piece kernel (the Shared stage's completion when
// that runs on another stream); may be null.
cudaError_t launch_ns_merge(const Geometry& g, const void* q, const void* pool_k, const void* pool_v,
                            const int32_t* beam_tok_idx, const int32_t* shared_len,
                            const float* part_o, const float* part_lse, void* out,
                            float* lse, int32_t* status, cudaStream_t stream, cudaEvent_t join = nullptr,
                            bool equal_split = true);
// The row merge alone over pieces 0 .. np-1 of each row (np <= g.pieces).
cudaError_t launch_merge_rows(const Geometry& g, int np, const int32_t* shared_len, const float* part_o,
                              const float* part_lse, void* out, float* lse, int32_t* status, cudaStream_t stream);
// One CTA per request; 1 <= BW, W <= 1024 (checked by the caller).
cudaError_t launch_beam_select(int R, int BW, int K, int W, const float* beam_score, const float* cand_logp,
                               const int32_t* cand_token, int32_t* parent, int32_t* token, float* score,
                               cudaStream_t stream);
// elem_bytes: bytes per K/V element (2: bf16, 4: fp32).
cudaError_t launch_beam_update(int R, int BW, int Hkv, int d, int elem_bytes, int S, int Tmax, int step,
                               const int32_t* parent, const void* new_k, const void* new_v, void* pool_k,
                               void* pool_v, int32_t* idx, int32_t* status, cudaStream_t stream,
                               int vectors_per_thread = 4);
// xattn_beam_update with the copy's vectors per thread (launch_beam_update).
int beam_update(const xattn_desc* desc, const int32_t* parent, const void* new_k, const void* new_v,
                void* ns_k_pool, void* ns_v_pool, int32_t* beam_tok_idx, int32_t step, int32_t* status,
                cudaStream_t stream, int vectors_per_thread);

int merge_ctas_for(const Geometry& g);
// The host-side argument checks of xattn_decode, without launching anything.
int check_decode_args(const xattn_desc* desc, const void* q, const void* shared_k, const void* shared_v,
                      const int32_t* shared_len, const void* ns_k_pool, const void* ns_v_pool,
                      const int32_t* beam_tok_idx, int32_t step, const void* out, const float* lse,
                      const void* workspace, size_t workspace_bytes);
// Whether xattn_decode runs the Shared stage and the Merge in one tensor-core kernel (after
// a short Non-Shared kernel when step > 0): one prefix piece and a short Non-Shared part.
inline bool decode_is_fused(const Geometry& g, int kernel, int step) {
    return kernel == 1 && g.nsplit == 1 && step <= kNsDirectMax;
}
// Whether the fused decode computes the Non-Shared part inside the Shared-stage kernel (one
// launch): every row tile's beams' Non-Shared keys fit one 128-key tile.
inline bool ns_tile_fits(const Geometry& g, int kernel, int step) {
    return decode_is_fused(g, kernel, step) && step > 0 && (kTileRows / g.G) * step <= kTcTileKeys;
}
int shared_tc_ctas_for(const Geometry& g);

}  // namespace xattn
