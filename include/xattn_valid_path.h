/*
 * Valid-path constraint of generative-recommendation beam search: host trie builder and
 * device masks, C ABI.
 *
 * xGR: Efficient Generative Recommendation Serving at Scale, section 2.2 (xBeam, valid path
 * constraint): only token sequences that map to real items may be generated; the masks come
 * from a pre-built vocabulary of valid items. Here that vocabulary is a trie of the item
 * catalogue's token paths, built on the host into caller-owned arrays and read by the
 * kernels from device memory:
 *   node 0 is the root; nodes are numbered level by level (breadth first); the children of
 *   node n are nodes child_off[n] + 1 .. child_off[n + 1], reached by the tokens
 *   child_tok[child_off[n] .. child_off[n + 1]), in increasing order.
 * A row's (a beam's) valid next tokens at step s are the children of the node its first s
 * tokens lead to; none if those tokens leave the trie.
 *
 * Two forms of the same mask: dense for early steps, when most tokens are valid (every
 * logit of the row is visited), sparse for late steps, when few are (only the valid
 * tokens' logits are read, and the best C of them come out sorted, in the form
 * xattn_beam_select takes).
 */
#ifndef XATTN_VALID_PATH_H_
#define XATTN_VALID_PATH_H_

#include <stdint.h>

#include "xattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Number of trie nodes for the catalogue items [num_items, path_len] (host int32, any order,
 * duplicates allowed): the root plus one node per distinct non-empty item prefix.
 * INVALID_ARG: NULL pointer, num_items < 1, path_len < 1, a negative token, or more than
 * 2^31 - 1 nodes. Host only. */
XATTN_API int xattn_trie_size(const int32_t* items, int64_t num_items, int32_t path_len,
                              int64_t* num_nodes);

/* Fills child_off [num_nodes + 1] and child_tok [num_nodes - 1] (host int32 buffers owned
 * by the caller) for the same items; num_nodes must be the value xattn_trie_size gave
 * (else INVALID_ARG). Host only. */
XATTN_API int xattn_trie_build(const int32_t* items, int64_t num_items, int32_t path_len,
                               int64_t num_nodes, int32_t* child_off, int32_t* child_tok);

/* Dense mask, in place: for every row r < rows, logp[r, v] (device fp32, rows of V) becomes
 * -inf unless v is a valid next token of r; the other entries are not touched (not even
 * read). valid_count [rows] (device int32, may be NULL) gets the number of valid next tokens
 * below V. prefix [rows, prefix_stride] (device int32; may be NULL when step == 0) holds the
 * rows' tokens, positions 0 .. step-1 used. child_off / child_tok: the trie in device memory.
 * Requires 0 <= step < path_len, 1 <= V <= 262144, rows >= 1, num_nodes >= 1, 4-byte
 * aligned pointers (else INVALID_ARG / UNSUPPORTED / MISALIGNED). A trie index out of range
 * sets XATTN_STATUS_BAD_TRIE in *status (device int32, may be NULL) and masks the whole row.
 * One CTA per row, the row's valid tokens as a V-bit map in shared memory. */
XATTN_API int xattn_valid_path_mask(const int32_t* child_off, const int32_t* child_tok,
                                    int64_t num_nodes, int32_t path_len, const int32_t* prefix,
                                    int32_t prefix_stride, int32_t step, int32_t rows, int32_t V,
                                    float* logp, int32_t* valid_count, int32_t* status,
                                    xattn_stream_t stream);

/* Sparse list: for every row r, the C valid next tokens of largest logp[r, v] (ties to the
 * smaller token), best first: cand_token [rows, C] (device int32) and cand_logp [rows, C]
 * (device fp32), padded with -1 and -inf; valid_count [rows] (device int32, may be NULL) as
 * above. logp is read at the valid tokens only (no NaN there). A row with more than 4096
 * valid tokens sets XATTN_STATUS_TOO_MANY_VALID in *status and gets an empty list (use the
 * dense mask for such steps). Requires 1 <= C <= 1024; otherwise as xattn_valid_path_mask.
 * One CTA per row: the valid tokens' keys are sorted in shared memory. */
XATTN_API int xattn_valid_path_topk(const int32_t* child_off, const int32_t* child_tok,
                                    int64_t num_nodes, int32_t path_len, const int32_t* prefix,
                                    int32_t prefix_stride, int32_t step, int32_t rows, int32_t V,
                                    const float* logp, int32_t C, int32_t* cand_token,
                                    float* cand_logp, int32_t* valid_count, int32_t* status,
                                    xattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* XATTN_VALID_PATH_H_ */
