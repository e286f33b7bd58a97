// Valid-path masks of generative-recommendation beam search (device side; C ABI in
// xattn_valid_path.h).
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.2 (xBeam, valid path
// constraint): only token sequences that map to real items may be generated; masks come from
// a pre-built vocabulary of valid items (here a trie, see trie.cpp). A row's valid next
// tokens are the children of the trie node its prefix leads to; the dense form masks every
// other logit of the row in place (early steps: most tokens valid), the sparse form reads
// only the valid tokens' logits and emits the best C of them sorted (late steps: few valid).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/xattn_valid_path.h"

namespace {

constexpr int kMaskThreads = 256;
constexpr int kMaxV = 262144;        // dense: the V-bit map fits in 32 KB of shared memory
constexpr int kTopThreads = 1024;
constexpr int kMaxValid = 4096;      // sparse: valid tokens sorted per row
constexpr int kMaxC = 1024;

__device__ __forceinline__ void set_status(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}

// The range [*b, *e) of child_tok holding the valid next tokens of `row`; empty when its
// prefix leaves the trie. Returns false (range empty) when a trie index is out of range.
__device__ bool walk_trie(const int32_t* __restrict__ child_off, const int32_t* __restrict__ child_tok,
                          int64_t num_nodes, const int32_t* __restrict__ prefix, int32_t step, int* b, int* e) {
    int64_t node = 0;
    for (int l = 0; l < step; ++l) {
        int lo = child_off[node], hi = child_off[node + 1];
        if (lo < 0 || lo > hi || hi > num_nodes - 1) {
            *b = *e = 0;
            return false;
        }
        const int32_t tok = prefix[l];
        while (lo < hi) {  // first child token >= tok
            const int mid = (lo + hi) >> 1;
            if (child_tok[mid] < tok) lo = mid + 1;
            else hi = mid;
        }
        if (lo >= child_off[node + 1] || child_tok[lo] != tok) {
            *b = *e = 0;  // the prefix starts no item
            return true;
        }
        node = (int64_t)lo + 1;
    }
    const int lo = child_off[node], hi = child_off[node + 1];
    if (lo < 0 || lo > hi || hi > num_nodes - 1) {
        *b = *e = 0;
        return false;
    }
    *b = lo;
    *e = hi;
    return true;
}

__global__ void __launch_bounds__(kMaskThreads) mask_kernel(const int32_t* __restrict__ child_off,
                                                            const int32_t* __restrict__ child_tok, int64_t num_nodes,
                                                            const int32_t* __restrict__ prefix, int32_t prefix_stride,
                                                            int32_t step, int32_t V, float* __restrict__ logp,
                                                            int32_t* __restrict__ valid_count, int32_t* status) {
    extern __shared__ uint32_t bits[];  // V bits
    __shared__ int s_b, s_e, s_cnt;
    const int row = blockIdx.x, t = threadIdx.x;
    const int words = (V + 31) / 32;
    for (int w = t; w < words; w += kMaskThreads) bits[w] = 0u;
    if (t == 0) {
        int b, e;
        if (!walk_trie(child_off, child_tok, num_nodes, prefix + (size_t)row * prefix_stride, step, &b, &e))
            set_status(status, XATTN_STATUS_BAD_TRIE);
        s_b = b;
        s_e = e;
        s_cnt = 0;
    }
    __syncthreads();
    int cnt = 0;
    for (int i = s_b + t; i < s_e; i += kMaskThreads) {
        const int32_t v = child_tok[i];
        if (v >= 0 && v < V) {
            atomicOr(&bits[v >> 5], 1u << (v & 31));
            ++cnt;  // children of a node are distinct tokens
        }
    }
    if (cnt) atomicAdd(&s_cnt, cnt);
    __syncthreads();
    float* lrow = logp + (size_t)row * V;
    for (int v = t; v < V; v += kMaskThreads)
        if (!((bits[v >> 5] >> (v & 31)) & 1u)) lrow[v] = -INFINITY;
    if (t == 0 && valid_count) valid_count[row] = s_cnt;
}

// Rank key, larger = better: the logit as an order-preserving integer (-0 as +0) above the
// complemented token, so that equal logits rank the smaller token first; 0 = no candidate.
__device__ __forceinline__ uint64_t rank_key(float s, uint32_t tok) {
    uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - tok);
}

__global__ void __launch_bounds__(kTopThreads) topk_kernel(const int32_t* __restrict__ child_off,
                                                           const int32_t* __restrict__ child_tok, int64_t num_nodes,
                                                           const int32_t* __restrict__ prefix, int32_t prefix_stride,
                                                           int32_t step, int32_t V, const float* __restrict__ logp,
                                                           int32_t C, int32_t* __restrict__ cand_token,
                                                           float* __restrict__ cand_logp,
                                                           int32_t* __restrict__ valid_count, int32_t* status) {
    __shared__ uint64_t keys[kMaxValid];
    __shared__ int s_b, s_e, s_cnt;
    const int row = blockIdx.x, t = threadIdx.x;
    if (t == 0) {
        int b, e;
        if (!walk_trie(child_off, child_tok, num_nodes, prefix + (size_t)row * prefix_stride, step, &b, &e))
            set_status(status, XATTN_STATUS_BAD_TRIE);
        s_b = b;
        s_e = e;
        s_cnt = 0;
    }
    __syncthreads();
    const int b = s_b, n = s_e - s_b;
    const float* lrow = logp + (size_t)row * V;
    if (n > kMaxValid) {  // too many for the sparse form: an empty list and a status bit
        if (t == 0) set_status(status, XATTN_STATUS_TOO_MANY_VALID);
        int cnt = 0;
        for (int i = t; i < n; i += kTopThreads) cnt += (child_tok[b + i] >= 0 && child_tok[b + i] < V) ? 1 : 0;
        if (cnt) atomicAdd(&s_cnt, cnt);
        for (int j = t; j < C; j += kTopThreads) {
            cand_token[(size_t)row * C + j] = -1;
            cand_logp[(size_t)row * C + j] = -INFINITY;
        }
        __syncthreads();
        if (t == 0 && valid_count) valid_count[row] = s_cnt;
        return;
    }
    int P = 1;
    while (P < n) P <<= 1;
    int cnt = 0;
    for (int i = t; i < P; i += kTopThreads) {
        uint64_t k = 0;
        if (i < n) {
            const int32_t v = child_tok[b + i];
            if (v >= 0 && v < V) {
                k = rank_key(lrow[v], (uint32_t)v);
                ++cnt;
            }
        }
        keys[i] = k;
    }
    if (cnt) atomicAdd(&s_cnt, cnt);
    __syncthreads();
    // bitonic sort of keys[0 .. P), descending
    for (int k2 = 2; k2 <= P; k2 <<= 1) {
        for (int jj = k2 >> 1; jj > 0; jj >>= 1) {
            for (int i = t; i < P; i += kTopThreads) {
                const int o = i ^ jj;
                if (o > i) {
                    const uint64_t x = keys[i], y = keys[o];
                    if (((i & k2) == 0) ? (x < y) : (x > y)) {
                        keys[i] = y;
                        keys[o] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
    const int valid = s_cnt;
    for (int j = t; j < C; j += kTopThreads) {
        int32_t tok = -1;
        float val = -INFINITY;
        if (j < valid) {
            tok = (int32_t)(0xFFFFFFFFu - (uint32_t)(keys[j] & 0xFFFFFFFFu));
            val = lrow[tok];
        }
        cand_token[(size_t)row * C + j] = tok;
        cand_logp[(size_t)row * C + j] = val;
    }
    if (t == 0 && valid_count) valid_count[row] = valid;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_common(const int32_t* child_off, const int32_t* child_tok, int64_t num_nodes, int32_t path_len,
                 const int32_t* prefix, int32_t prefix_stride, int32_t step, int32_t rows, int32_t V) {
    if (!child_off || (num_nodes > 1 && !child_tok) || num_nodes < 1 || num_nodes > 0x7fffffffLL || path_len < 1 ||
        step < 0 || step >= path_len || rows < 1 || V < 1 || (step > 0 && (!prefix || prefix_stride < step)))
        return XATTN_ERR_INVALID_ARG;
    if (!aligned4(child_off) || !aligned4(child_tok) || !aligned4(prefix)) return XATTN_ERR_MISALIGNED;
    return XATTN_OK;
}

}  // namespace

extern "C" {

int xattn_valid_path_mask(const int32_t* child_off, const int32_t* child_tok, int64_t num_nodes, int32_t path_len,
                          const int32_t* prefix, int32_t prefix_stride, int32_t step, int32_t rows, int32_t V,
                          float* logp, int32_t* valid_count, int32_t* status, xattn_stream_t stream) {
    int rc = check_common(child_off, child_tok, num_nodes, path_len, prefix, prefix_stride, step, rows, V);
    if (rc != XATTN_OK) return rc;
    if (!logp) return XATTN_ERR_INVALID_ARG;
    if (V > kMaxV) return XATTN_ERR_UNSUPPORTED;
    if (!aligned4(logp) || !aligned4(valid_count) || !aligned4(status)) return XATTN_ERR_MISALIGNED;
    const size_t smem = (size_t)((V + 31) / 32) * sizeof(uint32_t);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    mask_kernel<<<rows, kMaskThreads, smem, st>>>(child_off, child_tok, num_nodes, step > 0 ? prefix : child_off,
                                                  prefix_stride, step, V, logp, valid_count, status);
    return cudaGetLastError() == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

int xattn_valid_path_topk(const int32_t* child_off, const int32_t* child_tok, int64_t num_nodes, int32_t path_len,
                          const int32_t* prefix, int32_t prefix_stride, int32_t step, int32_t rows, int32_t V,
                          const float* logp, int32_t C, int32_t* cand_token, float* cand_logp, int32_t* valid_count,
                          int32_t* status, xattn_stream_t stream) {
    int rc = check_common(child_off, child_tok, num_nodes, path_len, prefix, prefix_stride, step, rows, V);
    if (rc != XATTN_OK) return rc;
    if (!logp || !cand_token || !cand_logp || C < 1) return XATTN_ERR_INVALID_ARG;
    if (C > kMaxC) return XATTN_ERR_UNSUPPORTED;
    if (!aligned4(logp) || !aligned4(cand_token) || !aligned4(cand_logp) || !aligned4(valid_count) ||
        !aligned4(status))
        return XATTN_ERR_MISALIGNED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    topk_kernel<<<rows, kTopThreads, 0, st>>>(child_off, child_tok, num_nodes, step > 0 ? prefix : child_off,
                                              prefix_stride, step, V, logp, C, cand_token, cand_logp, valid_count,
                                              status);
    return cudaGetLastError() == cudaSuccess ? XATTN_OK : XATTN_ERR_CUDA;
}

}  // extern "C"
