// The host structures behind the C ABI (chunked hash tree, catalogue trie) under
// AddressSanitizer and UndefinedBehaviorSanitizer, built by tests/test_sanitizers.py.
// Random operation sequences with consistency checks (the best waiting request has the
// smallest missing count, ties to the earliest inserted; the trie's arrays are well
// formed), then the error paths. Exit 0 = clean.
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <map>
#include <random>
#include <vector>

#include "../../include/xattn_cht.h"
#include "../../include/xattn_valid_path.h"

static int fail(const char* what) {
    std::fprintf(stderr, "host_san: %s\n", what);
    return 1;
}

static int cht_case(int B, int groups, unsigned seed) {
    std::mt19937 rng(seed);
    std::vector<std::vector<int32_t>> bases(groups);
    for (auto& b : bases) {
        b.resize(rng() % (12 * B + 1));
        for (auto& t : b) t = (int32_t)(rng() % 40);
    }
    xattn_cht* t = xattn_cht_create(B);
    if (!t) return fail("create");
    std::map<int64_t, uint64_t> waiting;  // id -> insertion order
    std::vector<int64_t> active;
    uint64_t order = 0;
    int64_t next_id = 0;
    for (int step = 0; step < 600; ++step) {
        const unsigned op = rng() % 10;
        if (op < 4 || waiting.empty()) {
            const auto& b = bases[rng() % groups];
            std::vector<int32_t> p(b.begin(), b.begin() + (long)(rng() % (b.size() + 1)));
            for (unsigned k = rng() % (3 * B + 1); k; --k) p.push_back((int32_t)(rng() % 40));
            const int64_t id = next_id++;
            if (xattn_cht_insert(t, id, p.data(), (int64_t)p.size()) != XATTN_OK) return fail("insert");
            waiting[id] = order++;
        } else if (op < 7) {
            int64_t id = 0;
            int32_t miss = 0;
            if (xattn_cht_best(t, &id, &miss) != 1) return fail("best found nothing");
            // the smallest missing count, ties to the earliest inserted
            int32_t best_m = INT32_MAX;
            uint64_t best_o = UINT64_MAX;
            for (auto& kv : waiting) {
                int32_t m = 0;
                if (xattn_cht_missing(t, kv.first, &m) != XATTN_OK) return fail("missing");
                if (m < best_m || (m == best_m && kv.second < best_o)) best_m = m, best_o = kv.second;
            }
            if (miss != best_m || waiting.at(id) != best_o) return fail("best is not the best");
            if (xattn_cht_admit(t, id) != XATTN_OK) return fail("admit");
            waiting.erase(id);
            active.push_back(id);
        } else if (op < 9 && !active.empty()) {
            const size_t k = rng() % active.size();
            if (xattn_cht_finish(t, active[k]) != XATTN_OK) return fail("finish");
            active.erase(active.begin() + (long)k);
        } else {
            auto it = waiting.begin();
            std::advance(it, (long)(rng() % waiting.size()));
            if (xattn_cht_cancel(t, it->first) != XATTN_OK) return fail("cancel");
            waiting.erase(it);
        }
        int64_t w = -1, a = -1, h = -1;
        if (xattn_cht_counts(t, &w, &a, &h) != XATTN_OK || w != (int64_t)waiting.size() || a != (int64_t)active.size())
            return fail("counts");
    }
    if (xattn_cht_insert(t, 0, nullptr, -1) != XATTN_ERR_INVALID_ARG) return fail("negative length accepted");
    if (xattn_cht_admit(t, -12345) != XATTN_ERR_INVALID_ARG) return fail("unknown id admitted");
    xattn_cht_destroy(t);
    return 0;
}

static int trie_case(int64_t N, int32_t L, int32_t V, unsigned seed) {
    std::mt19937 rng(seed);
    std::vector<int32_t> items((size_t)(N * L));
    for (auto& x : items) x = (int32_t)(rng() % V);
    int64_t n = 0;
    if (xattn_trie_size(items.data(), N, L, &n) != XATTN_OK || n < 1) return fail("trie size");
    std::vector<int32_t> off((size_t)n + 1), tok((size_t)std::max<int64_t>(n - 1, 1));
    if (xattn_trie_build(items.data(), N, L, n, off.data(), tok.data()) != XATTN_OK) return fail("trie build");
    if (off[0] != 0 || off[(size_t)n] != n - 1) return fail("trie offsets");
    for (int64_t v = 0; v < n; ++v) {
        if (off[(size_t)v] > off[(size_t)v + 1]) return fail("trie offsets decrease");
        for (int32_t e = off[(size_t)v] + 1; e < off[(size_t)v + 1]; ++e)
            if (tok[(size_t)e - 1] >= tok[(size_t)e]) return fail("children not increasing");
    }
    if (xattn_trie_build(items.data(), N, L, n + 1, off.data(), tok.data()) != XATTN_ERR_INVALID_ARG)
        return fail("wrong node count accepted");
    items[0] = -1;
    if (xattn_trie_size(items.data(), N, L, &n) != XATTN_ERR_INVALID_ARG) return fail("negative token accepted");
    return 0;
}

int main() {
    const int cht[][3] = {{1, 3, 1}, {2, 4, 2}, {3, 2, 3}, {16, 5, 4}};
    for (auto& c : cht)
        if (cht_case(c[0], c[1], (unsigned)c[2])) return 1;
    if (trie_case(1, 1, 3, 5) || trie_case(300, 3, 7, 6) || trie_case(2000, 4, 50, 7) || trie_case(500, 2, 1000, 8))
        return 1;
    if (xattn_cht_create(0) != nullptr) return fail("block 0 accepted");
    std::printf("host_san: ok\n");
    return 0;
}
