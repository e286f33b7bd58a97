/*
 * xattn.h - C ABI of libxattn.so: beam-search decode attention over a KV cache split
 * into a Shared prefix part and a Non-Shared per-token part (GB300, sm_103a).
 *
 * The operation is the staged attention of "xGR: Efficient Generative Recommendation
 * Serving at Scale", section 2.1 (xAttention):
 *   - Separated KV cache: the Shared part holds the prompt (user history), computed once
 *     at prefill and stored once per request; the Non-Shared part holds only the tokens
 *     generated at each decode step.
 *   - Token-granularity management: each generated token is stored once, in its own pool
 *     slot; a beam reaches its tokens through an ancestry index, so forking copies nothing.
 *   - Staged computation: a Shared stage and a Non-Shared stage each produce local scores
 *     plus max/sum statistics; a Merge stage combines them with an online softmax.
 *   - In-place update: the Non-Shared structures are updated in place after each beam
 *     step without read-before-write hazards.
 * The same call serves prefix-homogeneous batches ("Requests of a Feather Must Flock
 * Together", method): a prefix group is a request and each sequence is a beam whose
 * unshared suffix is its Non-Shared part.
 *
 * Result. For request r, beam b, query head h (KV head h / G, G = Hq / Hkv), the keys are
 * the prefix tokens shared_k[r, 0 .. shared_len[r]-1, h/G] followed by the pool tokens
 * ns_k_pool[r, beam_tok_idx[r, b, i], h/G] for i < step (values alike), and
 *     out[r, b, h] = softmax(scale * q[r, b, h] . K^T) . V,
 *     lse[r, b, h] = natural-log log-sum-exp of the scaled scores.
 *
 * Conventions.
 *   - Every pointer except `desc`, `status_out` (xattn_read_status) is a DEVICE pointer
 *     on the current device. The caller owns every buffer; the library allocates no device
 *     buffers and keeps no data between calls. Its only CUDA objects of its own: per host
 *     thread and device, one stream and three events, created at the first bf16 decode that
 *     does not fuse its Non-Shared part into the Shared stage and has either a Non-Shared
 *     part long enough for its own piece kernel (more than 32 tokens) or a short one next
 *     to a prefix cut in several pieces: the Shared stage of such a decode runs on that
 *     stream, forked from `stream` by one event at the start of the call and joined back by
 *     another before the row merge, so it overlaps the Non-Shared kernel (and, in
 *     xattn_decode_step, the beam update). In xattn_decode the piece kernel of a long
 *     Non-Shared part also waits for the third, recorded once every CTA of the Shared stage
 *     has begun. The fork and the joins follow graph capture of `stream`.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream) and never
 *     synchronise, except xattn_read_status.
 *   - Tensors are dense, row-major (innermost dimension last), 16-byte aligned.
 *   - A call returns XATTN_OK or a negative code. Argument errors are detected on the host
 *     before anything is launched; nothing is written then.
 *   - Data errors that only the device can see (a shared_len outside [0, max_shared_len],
 *     an ancestry slot outside [0, ns_slots), a parent outside [0, beam_width)) OR a bit
 *     into the status word held in the workspace and make the affected rows NaN; kernels
 *     never trap. Read (and clear) the word with xattn_read_status.
 */
#ifndef XATTN_H_
#define XATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define XATTN_API __attribute__((visibility("default")))
#else
#define XATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t). */
typedef struct CUstream_st* xattn_stream_t;

/* Return codes. */
enum {
    XATTN_OK = 0,
    XATTN_ERR_INVALID_ARG = -1,          /* a size, pointer or step is out of range         */
    XATTN_ERR_UNSUPPORTED = -2,          /* valid but not implemented (e.g. head_dim 96)    */
    XATTN_ERR_WORKSPACE_TOO_SMALL = -3,  /* workspace_bytes < xattn_decode_workspace_size   */
    XATTN_ERR_MISALIGNED = -4,           /* a tensor is not 16-byte aligned                 */
    XATTN_ERR_CUDA = -5,                 /* a CUDA call or launch failed                    */
    XATTN_ERR_HOST_MEMORY = -6           /* a host allocation failed (host-side structures) */
};

/* Bits of the device status word (sticky until read with clear = 1). */
enum {
    XATTN_STATUS_BAD_SHARED_LEN = 1, /* shared_len[r] outside [0, max_shared_len]      */
    XATTN_STATUS_BAD_SLOT = 2,       /* beam_tok_idx entry outside [0, ns_slots)        */
    XATTN_STATUS_BAD_PARENT = 4,     /* parent[r, b] outside [0, beam_width)            */
    XATTN_STATUS_EMPTY_ROW = 8,      /* shared_len[r] == 0 and step == 0: no keys       */
    XATTN_STATUS_TIMEOUT = 16,       /* an on-chip wait gave up (internal error)        */
    XATTN_STATUS_BAD_TRIE = 32,      /* valid-path trie index out of range              */
    XATTN_STATUS_TOO_MANY_VALID = 64 /* sparse valid-path list: > 4096 valid tokens      */
};

enum { XATTN_DTYPE_BF16 = 0, XATTN_DTYPE_F32 = 1 };

/* Shapes of one decode batch. */
typedef struct xattn_desc {
    int32_t num_requests;   /* R: requests (or Feather prefix groups)                      */
    int32_t beam_width;     /* BW: beams (or sequences) per request                        */
    int32_t num_q_heads;    /* Hq                                                          */
    int32_t num_kv_heads;   /* Hkv; Hq % Hkv == 0, G = Hq / Hkv                            */
    int32_t head_dim;       /* d: 64 or 128                                                */
    int32_t max_shared_len; /* Lmax: token stride of shared_k / shared_v per request       */
    int32_t ns_slots;       /* S: pool slots per request (>= BW * max_steps)               */
    int32_t max_steps;      /* Tmax: row length of beam_tok_idx                            */
    float softmax_scale;    /* 0 selects 1/sqrt(d)                                         */
    int32_t dtype;          /* storage of q, K, V, the pools and new tokens: XATTN_DTYPE_BF16,
                               or XATTN_DTYPE_F32 (read without a bf16 step; max_steps <= 32,
                               else XATTN_ERR_UNSUPPORTED). fp32 Shared stage: shared_kernel
                               0 or 2 runs it on CUDA cores in fp32, 1 on the tensor cores
                               with tcgen05 kind::tf32 (operands multiplied with 10 mantissa
                               bits, fp32 accumulation); the Non-Shared part stays fp32.   */
    int32_t shared_kernel;  /* Shared-stage kernel: 0 automatic (tensor cores for bf16, CUDA
                               cores for fp32), 1 tensor cores, 2 CUDA cores               */
    int32_t split_tokens;   /* prefix tokens per Shared-stage piece: 0 automatic, else a
                               multiple of 128                                             */
    int32_t out_dtype;      /* dtype of `out`: XATTN_DTYPE_BF16 (0) or XATTN_DTYPE_F32      */
} xattn_desc;

/* Bytes of workspace xattn_decode needs for these shapes (at least 256). The workspace
 * holds the device status word (first 4 bytes; zero it once before first use, or call
 * xattn_read_status with clear = 1) and the per-split partial results of the Shared stage.
 * Returns 0 if the descriptor is invalid. */
XATTN_API size_t xattn_decode_workspace_size(const xattn_desc* desc);

/* One decode step of attention: Shared stage (prefix, tensor cores, split along the
 * prefix), Non-Shared stage (ancestry-indexed gathers) and the log-sum-exp Merge.
 *   q             [R, BW, Hq, d]        bf16 (fp32 when desc->dtype is XATTN_DTYPE_F32)
 *   shared_k/v    [R, Lmax, Hkv, d]     bf16 (or fp32)  prefix KV, stored once per request
 *   shared_len    [R]                   int32  valid prefix tokens per request (<= Lmax)
 *   ns_k/v_pool   [R, S, Hkv, d]        bf16 (or fp32)  Non-Shared tokens, one slot per token
 *   beam_tok_idx  [R, BW, Tmax]         int32  ancestry: slots of the beam's tokens
 *   step          0 <= step <= Tmax: positions 0 .. step-1 of each ancestry row are used
 *   out           [R, BW, Hq, d]        bf16 (or fp32, desc->out_dtype)  normalised output
 *   lse           [R, BW, Hq]           fp32   natural-log LSE of the scaled scores
 *   workspace     >= xattn_decode_workspace_size(desc) bytes, 256-byte aligned
 * Pointers that a zero-sized part does not touch may be NULL (shared_* when Lmax == 0;
 * pools and beam_tok_idx when step == 0). step == 0 with Lmax == 0 is INVALID_ARG. */
XATTN_API int xattn_decode(const xattn_desc* desc, const void* q, const void* shared_k,
                 const void* shared_v, const int32_t* shared_len, const void* ns_k_pool,
                 const void* ns_v_pool, const int32_t* beam_tok_idx, int32_t step, void* out,
                 float* lse, void* workspace, size_t workspace_bytes, xattn_stream_t stream);

/* The two halves of xattn_decode, for callers that schedule the stages themselves (and
 * for measuring them apart). xattn_decode_shared(...) followed by xattn_decode_merge(...) on
 * the same stream and workspace computes what xattn_decode(...) computes. The two halves cut
 * the prefix as xattn_query_plan(desc, 0, ...) reports, whatever the step; xattn_decode with a
 * long Non-Shared part (step > 32, bf16 storage, tensor-core Shared stage) may cut it into
 * fewer pieces (xattn_query_plan(desc, step, ...)), leaving SMs to the Non-Shared kernel that
 * runs beside the Shared stage, and then agrees with the halves to rounding.
 *
 * xattn_decode_shared: the Shared stage alone. For every (request r, KV head h) it stacks
 * the BW*G query rows of that KV head (row m = b*G + g) against the prefix, cut into
 * pieces of plan.split_tokens tokens, and writes each piece's normalised output and
 * natural-log LSE into the workspace:
 *   part_o   fp32 [R, Hkv, piece_stride, M, d]  at byte offset 256 (pieces 0 .. num_splits-1)
 *   part_lse fp32 [R, Hkv, piece_stride, M]     right after part_o
 * (a piece past shared_len[r] has lse = -inf and output 0). Requires max_shared_len > 0.
 *
 * xattn_decode_merge: the Non-Shared stage (ancestry-indexed gathers of the first `step`
 * pool tokens of every beam) and the Merge (log-sum-exp combine with the pieces in the
 * workspace), writing out and lse. When max_shared_len == 0 the workspace holds no pieces
 * and only the Non-Shared part is used. */
XATTN_API int xattn_decode_shared(const xattn_desc* desc, const void* q, const void* shared_k,
                                  const void* shared_v, const int32_t* shared_len,
                                  void* workspace, size_t workspace_bytes, xattn_stream_t stream);
XATTN_API int xattn_decode_merge(const xattn_desc* desc, const void* q, const int32_t* shared_len,
                                 const void* ns_k_pool, const void* ns_v_pool,
                                 const int32_t* beam_tok_idx, int32_t step, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, xattn_stream_t stream);

/* Bookkeeping of one beam-search step, in place (section 2.1, token-granularity
 * management and in-place updates). For every request r and beam b:
 *   the new token's K/V, new_k/new_v[r, b] ([R, BW, Hkv, d], desc->dtype), is written to pool
 *   slot step*BW + b (no other slot changes: nothing is copied when beams fork);
 *   beam_tok_idx[r, b, 0:step] becomes the old beam_tok_idx[r, parent[r, b], 0:step]
 *   and beam_tok_idx[r, b, step] becomes step*BW + b.
 * parent [R, BW] int32 is ignored at step 0. Requires step < Tmax and (step+1)*BW <= S.
 * A parent outside [0, BW) sets XATTN_STATUS_BAD_PARENT in *status (a device int32, may
 * be NULL) and writes -1 into that beam's ancestry positions 0 .. step-1. */
XATTN_API int xattn_beam_update(const xattn_desc* desc, const int32_t* parent, const void* new_k,
                      const void* new_v, void* ns_k_pool, void* ns_v_pool,
                      int32_t* beam_tok_idx, int32_t step, int32_t* status,
                      xattn_stream_t stream);

/* One decode step with its bookkeeping: exactly xattn_beam_update(desc, parent, new_k, new_v,
 * ns_k_pool, ns_v_pool, beam_tok_idx, step - 1, <workspace status word>) followed by
 * xattn_decode(desc, q, ..., beam_tok_idx, step, out, lse, workspace, ...) on `stream`: the
 * same output, LSE, pool contents, ancestry table and status bits, bit for bit (section 2.1:
 * the Non-Shared cache is updated in place after each beam step). Requires
 * 1 <= step <= Tmax and step*BW <= S; parent may be NULL when step == 1. The Shared-stage
 * kernel is launched as the beam update's programmatic dependent: when it takes the Non-Shared
 * part in its own tile (xattn_plan.ns_tile), its set-up, query loads and first prefix loads
 * overlap the update and it reads the pool and the table only after the update has completed;
 * when the decode is unfused (xattn_plan.fused == 0; every Shared-stage kernel, fp32 storage
 * included), it reads nothing the update writes, runs beside it, and completes only after it,
 * so that the Non-Shared + Merge kernel(s) queued next find the update complete. */
XATTN_API int xattn_decode_step(const xattn_desc* desc, const int32_t* parent, const void* new_k,
                                const void* new_v, const void* q, const void* shared_k, const void* shared_v,
                                const int32_t* shared_len, void* ns_k_pool, void* ns_v_pool,
                                int32_t* beam_tok_idx, int32_t step, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, xattn_stream_t stream);

/* Beam selection of one beam-search step (section 2.2, xBeam: early sort termination). For
 * each request r, candidate (b, k) with b < BW = beam_width and k < K = cand_per_beam scores
 *   beam_score[r, b] + cand_logp[r, b, k]          (one fp32 addition)
 * and the W = out_width candidates with the largest scores are selected, equal scores
 * ordered by the smaller flat index b*K + k, and written best first:
 *   parent[r, j] = b,   token[r, j] = cand_token[r, b, k],   score[r, j] = its score.
 * Each list cand_logp[r, b, 0:K] must be in non-increasing order (as a per-beam top-K
 * returns it); -inf is allowed (masked candidates), NaN is not. The walk down a beam's list
 * stops at the first candidate that cannot enter the best W found so far, so the work
 * follows the lists' order, not BW*K. One CTA per request.
 *   beam_score [R, BW] fp32, cand_logp [R, BW, K] fp32, cand_token [R, BW, K] int32: device
 *   parent, token [R, W] int32, score [R, W] fp32: device, written
 * Returns INVALID_ARG for a size < 1, W > BW*K or a NULL pointer; UNSUPPORTED for
 * BW > 1024, W > 1024 or BW*K > 2^30; MISALIGNED for a pointer not 4-byte aligned. Lists
 * out of order give an unspecified selection (not detected). */
/* Self-check of the bounded on-chip waits: one CTA waits, through the same bounded mbarrier
 * wait as the kernels, on a phase that nothing completes; after about limit_cycles SM cycles
 * (0 .. 2^32) it gives up, sets XATTN_STATUS_TIMEOUT in *status (device int32) and returns;
 * *waited_cycles (device int64, may be NULL) gets the cycles it waited. This exercises the
 * kernels' timeout path without a fault; the context stays usable. INVALID_ARG for a NULL
 * status or a limit out of range, MISALIGNED for a misaligned pointer. */
XATTN_API int xattn_check_bounded_wait(int64_t limit_cycles, int32_t* status, int64_t* waited_cycles,
                                       xattn_stream_t stream);

XATTN_API int xattn_beam_select(int32_t num_requests, int32_t beam_width, int32_t cand_per_beam,
                                int32_t out_width, const float* beam_score, const float* cand_logp,
                                const int32_t* cand_token, int32_t* parent, int32_t* token, float* score,
                                xattn_stream_t stream);

/* Allocation-free decode. xAttention as published has no counterpart to this call; it
 * exists for callers that cannot allocate device memory or hand the library a workspace (a
 * runtime that owns every allocation, a latency-critical thread that must not trigger
 * cudaMalloc, a fixed memory budget). It does exactly what xattn_decode does, with its
 * workspace taken from a static device array of XATTN_NOALLOC_SCRATCH_BYTES (32 MiB) inside
 * the library; every device that loads the library holds that array until the process
 * exits.
 *   - Shapes whose xattn_decode_workspace_size exceeds that limit return
 *     XATTN_ERR_WORKSPACE_TOO_SMALL before anything is launched; an invalid descriptor
 *     returns XATTN_ERR_INVALID_ARG.
 *   - The first call in each CUDA context looks up the array's device address (with that
 *     context current) and caches it under the context's unique id; make that first call
 *     before any stream capture.
 *   - Every host-side check of xattn_decode runs before anything is enqueued: a rejected
 *     call leaves the array untouched.
 *   - All calls share the array: calls whose GPU work overlaps (other streams or threads on
 *     the same device) race and must be serialised by the caller.
 *   - The status word is cleared on `stream` at the start of each accepted call; if
 *     `status_out` (a device int32, may be NULL) is given, the call's final status word is
 *     copied there on `stream`.
 * No cudaMalloc, cudaFree or allocating library routine is called. Other arguments and
 * results are those of xattn_decode. */
#define XATTN_NOALLOC_SCRATCH_BYTES (32u << 20)
XATTN_API int xattn_decode_noalloc(const xattn_desc* desc, const void* q, const void* shared_k,
                                   const void* shared_v, const int32_t* shared_len,
                                   const void* ns_k_pool, const void* ns_v_pool,
                                   const int32_t* beam_tok_idx, int32_t step, void* out,
                                   float* lse, int32_t* status_out, xattn_stream_t stream);

/* Copies the status word of `workspace` (device) to *status_out (host), optionally
 * clearing it, and synchronises `stream`. */
XATTN_API int xattn_read_status(void* workspace, int32_t* status_out, int32_t clear, xattn_stream_t stream);

/* How xattn_decode will run these shapes (for tests and reports). */
typedef struct xattn_plan {
    int32_t shared_kernel;    /* 0 none (Lmax == 0), 1 tensor-core (tcgen05 kind::f16),
                                 2 CUDA-core, 3 tensor-core tf32 (tcgen05 kind::tf32, fp32
                                 storage)                                                  */
    int32_t num_splits;       /* pieces the prefix is cut into                           */
    int32_t split_tokens;     /* tokens per piece (multiple of 128)                      */
    int32_t rows_per_unit;    /* M = BW * G stacked query rows per (request, KV head)    */
    int32_t row_tiles;        /* 128-row tiles per (request, KV head)                    */
    int32_t shared_ctas;      /* CTAs of one Shared-stage launch                         */
    int32_t merge_ctas;       /* CTAs of one Non-Shared + Merge launch (0 when fused)    */
    int32_t fused;            /* 1: xattn_decode runs the Non-Shared part as one piece, then
                                 the Shared-stage kernel, whose epilogue merges (single
                                 prefix piece, step <= 32); 0: Shared stage, then the
                                 Non-Shared + Merge kernel(s)                              */
    int32_t piece_stride;     /* pieces per (request, KV head) in the workspace layout     */
    int32_t ns_tile;          /* 1: (fused only) the Shared-stage kernel gathers the Non-Shared
                                 tokens itself and attends to them as one more 128-key tile
                                 of each row tile (masked per beam), so xattn_decode is one
                                 launch; 0: a Non-Shared kernel runs first                  */
    int32_t reserved[1];
} xattn_plan;

XATTN_API int xattn_query_plan(const xattn_desc* desc, int32_t step, xattn_plan* plan);

/* Human-readable text for a return code. */
XATTN_API const char* xattn_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* XATTN_H_ */
