// Trie of an item catalogue's token paths (host code, C ABI in xattn_valid_path.h).
//
// xGR: Efficient Generative Recommendation Serving at Scale, section 2.2 (xBeam, valid path
// constraint): the masks come from a pre-built vocabulary of valid items. The items are
// sorted and deduplicated; then the trie is laid out level by level: every node of a level
// owns the run of sorted items sharing its prefix, and its children are the runs of equal
// tokens at the next position within that run, numbered in order. Breadth-first numbering
// makes edge e lead to node e + 1, so one offset array and one token array describe it.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "../../include/xattn_valid_path.h"

namespace {

// The items sorted lexicographically with duplicates removed, as row indices into `items`.
bool sorted_unique(const int32_t* items, int64_t n, int32_t L, std::vector<int64_t>* order) {
    for (int64_t i = 0; i < n * L; ++i)
        if (items[i] < 0) return false;
    order->resize((size_t)n);
    std::iota(order->begin(), order->end(), (int64_t)0);
    auto less = [&](int64_t a, int64_t b) {
        return std::lexicographical_compare(items + a * L, items + (a + 1) * L, items + b * L, items + (b + 1) * L);
    };
    std::sort(order->begin(), order->end(), less);
    auto same = [&](int64_t a, int64_t b) { return std::memcmp(items + a * L, items + b * L, sizeof(int32_t) * L) == 0; };
    order->erase(std::unique(order->begin(), order->end(), same), order->end());
    return true;
}

struct Run {
    int64_t lo, hi;  // positions in the sorted order
};

// Walks the levels; calls edge(token) for every edge in breadth-first order and
// close(node) after the last edge of each node, in node order. Returns the node count.
template <typename Edge, typename Close>
int64_t walk(const int32_t* items, int32_t L, const std::vector<int64_t>& order, Edge edge, Close close) {
    std::vector<Run> level{{0, (int64_t)order.size()}}, next;
    int64_t nodes = 1;
    for (int32_t l = 0; l <= L; ++l) {
        next.clear();
        for (const Run& run : level) {
            if (l < L) {
                int64_t i = run.lo;
                while (i < run.hi) {
                    const int32_t tok = items[order[(size_t)i] * L + l];
                    int64_t j = i + 1;
                    while (j < run.hi && items[order[(size_t)j] * L + l] == tok) ++j;
                    edge(tok);
                    next.push_back(Run{i, j});
                    ++nodes;
                    i = j;
                }
            }
            close();
        }
        level.swap(next);
    }
    return nodes;
}

// Runs `body` so that no C++ exception crosses the C ABI (a failed allocation becomes
// XATTN_ERR_HOST_MEMORY).
template <typename F>
int guarded(F body) {
    try {
        return body();
    } catch (const std::bad_alloc&) {
        return XATTN_ERR_HOST_MEMORY;
    } catch (...) {
        return XATTN_ERR_INVALID_ARG;
    }
}

}  // namespace

extern "C" {

int xattn_trie_size(const int32_t* items, int64_t num_items, int32_t path_len, int64_t* num_nodes) {
    return guarded([&]() -> int {
        if (!items || !num_nodes || num_items < 1 || path_len < 1) return XATTN_ERR_INVALID_ARG;
        std::vector<int64_t> order;
        if (!sorted_unique(items, num_items, path_len, &order)) return XATTN_ERR_INVALID_ARG;
        const int64_t n = walk(items, path_len, order, [](int32_t) {}, [] {});
        if (n > 0x7fffffffLL) return XATTN_ERR_INVALID_ARG;
        *num_nodes = n;
        return XATTN_OK;
    });
}

int xattn_trie_build(const int32_t* items, int64_t num_items, int32_t path_len, int64_t num_nodes,
                     int32_t* child_off, int32_t* child_tok) {
    return guarded([&]() -> int {
        if (!items || !child_off || num_items < 1 || path_len < 1 || num_nodes < 1 || num_nodes > 0x7fffffffLL ||
            (num_nodes > 1 && !child_tok))
            return XATTN_ERR_INVALID_ARG;
        std::vector<int64_t> order;
        if (!sorted_unique(items, num_items, path_len, &order)) return XATTN_ERR_INVALID_ARG;
        // count first, so that nothing is written past the caller's buffers
        if (walk(items, path_len, order, [](int32_t) {}, [] {}) != num_nodes) return XATTN_ERR_INVALID_ARG;
        int64_t edges = 0, closed = 0;
        child_off[0] = 0;
        walk(
            items, path_len, order, [&](int32_t tok) { child_tok[edges++] = tok; },
            [&] { child_off[++closed] = (int32_t)edges; });
        return closed == num_nodes && edges == num_nodes - 1 ? XATTN_OK : XATTN_ERR_INVALID_ARG;
    });
}

}  // extern "C"
