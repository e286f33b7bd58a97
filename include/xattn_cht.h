/*
 * Chunked hash tree (CHT) of a prefix-aware batch scheduler — host side, C ABI.
 *
 * "Requests of a Feather Must Flock Together", methodology, component 1 (Chunked Hash Tree):
 * each request is represented by the cumulative hashes of its prompt over fixed-size token
 * blocks; the structure keeps the working set of hashes of the active batch and a min-heap
 * of the waiting requests keyed by their missing count (blocks not covered by the active
 * batch), so that the waiting request sharing the most with the batch is found in
 * O(log W) for W waiting requests; insertion, admission to the batch and removal of
 * finished requests update only the requests that share the blocks involved, and stale
 * heap entries are dropped lazily when they reach the top.
 *
 * Definitions used here:
 *   - a block is B = block_tokens consecutive prompt tokens; only whole blocks count (a
 *     prompt of n tokens has floor(n / B) blocks);
 *   - block i of a request is covered when some active request has the same first
 *     (i + 1) * B tokens (equal cumulative hash); covered blocks form a prefix;
 *   - missing(r) = blocks(r) - covered blocks of r;
 *   - the best waiting request has the smallest missing count, ties to the earliest
 *     inserted.
 * Hashes are 64-bit (splitmix64 mixing of the token stream); two different prefixes that
 * collide would be taken as equal (probability about 2^-64 per pair).
 *
 * All functions are host-only: no device memory, no CUDA call. A handle is not
 * thread-safe (one scheduler thread drives it). Functions return XATTN_OK (0) or a
 * negative XATTN_ERR_* code from xattn.h, except xattn_cht_best (1 / 0 / negative).
 */
#ifndef XATTN_CHT_H_
#define XATTN_CHT_H_

#include <stdint.h>

#include "xattn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct xattn_cht xattn_cht;

/* A new, empty structure for blocks of block_tokens (>= 1) tokens; NULL on a bad size or
 * out of memory. Owned by the caller: release with xattn_cht_destroy. */
XATTN_API xattn_cht* xattn_cht_create(int32_t block_tokens);
XATTN_API void xattn_cht_destroy(xattn_cht* cht);

/* Adds a waiting request. tokens [num_tokens] int32 (host memory, copied as hashes; may be
 * NULL when num_tokens == 0). INVALID_ARG: NULL handle, num_tokens < 0, or request_id
 * already present (waiting or active). */
XATTN_API int xattn_cht_insert(xattn_cht* cht, int64_t request_id, const int32_t* tokens,
                               int64_t num_tokens);

/* The best waiting request (fewest missing blocks, ties to the earliest inserted): writes
 * its id and missing count and returns 1; returns 0 when nothing waits (outputs untouched);
 * INVALID_ARG for a NULL argument. */
XATTN_API int xattn_cht_best(xattn_cht* cht, int64_t* request_id, int32_t* missing_blocks);

/* Moves a waiting request into the active batch (its blocks join the working set).
 * INVALID_ARG if the request is not waiting. */
XATTN_API int xattn_cht_admit(xattn_cht* cht, int64_t request_id);

/* Removes an active request (finished, or its batch dispatched): its blocks leave the
 * working set unless another active request holds them. INVALID_ARG if not active. */
XATTN_API int xattn_cht_finish(xattn_cht* cht, int64_t request_id);

/* Removes a waiting request without admitting it. INVALID_ARG if not waiting. */
XATTN_API int xattn_cht_cancel(xattn_cht* cht, int64_t request_id);

/* Current missing count of a waiting request. INVALID_ARG if not waiting. */
XATTN_API int xattn_cht_missing(const xattn_cht* cht, int64_t request_id, int32_t* missing_blocks);

/* Sizes: waiting requests, active requests, distinct block hashes in the working set. */
XATTN_API int xattn_cht_counts(const xattn_cht* cht, int64_t* waiting, int64_t* active,
                               int64_t* working_hashes);

#ifdef __cplusplus
}
#endif

#endif /* XATTN_CHT_H_ */
