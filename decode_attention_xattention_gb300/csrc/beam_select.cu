// Beam selection of one beam-search step.
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.2 (xBeam, early sort
// termination): the Top-K sequences of a step are chosen from the candidates of every beam,
// and because the log-probabilities within a beam are already in order, a global min-heap
// of the best so far lets the walk down a beam's list stop at the first candidate that
// falls below the heap's minimum.
//
// On the GPU the heap becomes one CTA per request holding the best candidates so far as a
// sorted array in shared memory. The beams' lists are walked in rounds, one position per
// round for every beam still walking: a beam whose candidate does not beat the last entry
// of a full array stops there (its later candidates score no higher and have larger
// indices), the other candidates of the round are compacted, sorted (bitonic) and merged
// into the array (merge path), which keeps the best `W`. The set chosen is the plain one:
// the `W` largest scores beam_score[b] + cand_logp[b, k], equal scores to the smaller flat
// index b * K + k.
#include "xattn_internal.cuh"

namespace xattn {
namespace {

constexpr int kSelThreads = 1024;  // one thread per beam and per output position
constexpr int kSelPrefetch = 8;    // list entries a beam's thread loads at once

// Rank key of a candidate, larger = better. High half: the score mapped to an unsigned
// integer of the same order (-0 taken as +0, so that equal scores compare equal); low half:
// the complement of the flat index, so that of equal scores the smaller index ranks first.
// A real key is never 0 (NaN scores are excluded), so 0 marks "no candidate".
__device__ __forceinline__ uint64_t rank_key(float s, uint32_t flat) {
    uint32_t u = __float_as_uint(s == 0.f ? 0.f : s);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - flat);
}

__global__ void __launch_bounds__(kSelThreads) beam_select_kernel(
    int BW, int K, int W, const float* __restrict__ beam_score, const float* __restrict__ cand_logp,
    const int32_t* __restrict__ cand_token, int32_t* __restrict__ parent, int32_t* __restrict__ token,
    float* __restrict__ score) {
    __shared__ uint64_t best[kSelThreads];    // the best so far, descending, `cnt` entries
    __shared__ uint64_t batch[kSelThreads];   // the round's candidates, then sorted
    __shared__ uint64_t merged[kSelThreads];
    __shared__ int warp_off[kSelThreads / 32];
    __shared__ int s_nb;
    const int r = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const bool is_beam = t < BW;
    const float bs = is_beam ? beam_score[(size_t)r * BW + t] : 0.f;
    const float* lp = cand_logp + ((size_t)r * BW + (is_beam ? t : 0)) * K;
    const int kmax = min(K, W);  // no beam gives more than W of the chosen
    bool active = is_beam;
    int cnt = 0;
    float pre[kSelPrefetch];
#pragma unroll
    for (int u = 0; u < kSelPrefetch; ++u) pre[u] = -INFINITY;

#pragma unroll 1
    for (int j = 0; j < kmax; ++j) {
        // 1. position j of every beam still walking its list
        if (active && j % kSelPrefetch == 0) {
#pragma unroll
            for (int u = 0; u < kSelPrefetch; ++u) pre[u] = j + u < kmax ? __ldg(lp + j + u) : -INFINITY;
        }
        uint64_t key = 0;
        if (active) {
            key = rank_key(bs + pre[0], (uint32_t)t * (uint32_t)K + (uint32_t)j);
            // early termination: the array is full and this candidate does not beat its last
            // entry, so neither does any later candidate of the beam
            if (cnt == W && key < best[W - 1]) {
                active = false;
                key = 0;
            }
        }
#pragma unroll
        for (int u = 0; u + 1 < kSelPrefetch; ++u) pre[u] = pre[u + 1];

        // 2. compact the round's candidates into batch[0 .. nb)
        const unsigned bal = __ballot_sync(0xffffffffu, key != 0);
        if (lane == 0) warp_off[warp] = __popc(bal);
        __syncthreads();
        if (warp == 0) {
            const int v = warp_off[lane];
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            warp_off[lane] = incl - v;
            if (lane == 31) s_nb = incl;
        }
        __syncthreads();
        const int nb = s_nb;
        if (nb == 0) break;  // every beam has stopped (the array is full)
        if (key != 0) batch[warp_off[warp] + __popc(bal & ((1u << lane) - 1u))] = key;
        int P = 1;
        while (P < nb) P <<= 1;
        if (t >= nb && t < P) batch[t] = 0;
        __syncthreads();

        // 3. bitonic sort of batch[0 .. P), descending
        for (int k2 = 2; k2 <= P; k2 <<= 1) {
            for (int jj = k2 >> 1; jj > 0; jj >>= 1) {
                if (t < P) {
                    const int o = t ^ jj;
                    if (o > t) {
                        const uint64_t a = batch[t], b = batch[o];
                        if (((t & k2) == 0) ? (a < b) : (a > b)) {
                            batch[t] = b;
                            batch[o] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }

        // 4. merge best[0 .. cnt) and batch[0 .. nb), both descending, keeping the first W:
        //    output position t takes `a` entries of best before it, found by binary search
        const int n = min(W, cnt + nb);
        if (t < n) {
            int lo = max(0, t - nb), hi = min(t, cnt);
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (best[mid] > batch[t - 1 - mid]) lo = mid + 1;
                else hi = mid;
            }
            const int b = t - lo;
            merged[t] = (b >= nb || (lo < cnt && best[lo] > batch[b])) ? best[lo] : batch[b];
        }
        __syncthreads();
        if (t < n) best[t] = merged[t];
        cnt = n;
        __syncthreads();
    }

    // 5. the chosen candidates, best first (the array holds exactly W entries here)
    if (t < W) {
        const uint32_t flat = 0xFFFFFFFFu - (uint32_t)(best[t] & 0xFFFFFFFFu);
        const int b = (int)(flat / (uint32_t)K), k = (int)(flat - (uint32_t)b * (uint32_t)K);
        const size_t c = ((size_t)r * BW + b) * K + k;
        parent[(size_t)r * W + t] = b;
        token[(size_t)r * W + t] = cand_token[c];
        score[(size_t)r * W + t] = beam_score[(size_t)r * BW + b] + cand_logp[c];
    }
}

}  // namespace

cudaError_t launch_beam_select(int R, int BW, int K, int W, const float* beam_score, const float* cand_logp,
                               const int32_t* cand_token, int32_t* parent, int32_t* token, float* score,
                               cudaStream_t stream) {
    if (R < 1 || BW < 1 || BW > kSelThreads || W < 1 || W > kSelThreads || K < 1) return cudaErrorInvalidValue;
    beam_select_kernel<<<R, kSelThreads, 0, stream>>>(BW, K, W, beam_score, cand_logp, cand_token, parent, token,
                                                      score);
    return cudaGetLastError();
}

}  // namespace xattn
