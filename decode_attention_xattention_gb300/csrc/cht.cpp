// Chunked hash tree of a prefix-aware batch scheduler (host code, C ABI in xattn_cht.h).
//
// "Requests of a Feather Must Flock Together", methodology, component 1: requests as
// cumulative hashes over fixed-size token blocks, a working set of the active batch's
// hashes, and a min-heap of waiting requests keyed by their missing count, so that the
// request to add next is found in O(log W).
//
// Bookkeeping: the working set counts, per block hash, the active requests holding it. A
// waiting request's covered count is the number of its block hashes in the working set;
// since a block hash is cumulative (it fixes every token before the block's end), the
// covered blocks are a prefix and missing = blocks - covered. An inverted index from block
// hash to the waiting requests holding it lets admission and removal adjust exactly the
// requests whose coverage changes; each admission or removal then pushes one fresh heap
// entry per request it touched and bumps that request's version, and entries whose version
// is stale are dropped when they surface (lazy deletion). The heap is rebuilt from the waiting requests when stale entries
// outnumber live ones.
#include <cstdint>
#include <new>
#include <stdexcept>
#include <queue>
#include <unordered_map>
#include <vector>

#include "../../include/xattn_cht.h"

namespace {

// splitmix64 output mixing (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", 2014): a bijective avalanche of a 64-bit word.
inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

enum class State : uint8_t { kWaiting, kActive };

struct Request {
    std::vector<uint64_t> hashes;  // cumulative hash at the end of each whole block
    int32_t covered = 0;           // blocks in the working set (waiting requests only)
    uint64_t seq = 0;              // insertion order (ties) and identity of this insertion
    uint32_t version = 0;          // bumped whenever the heap key changes
    uint64_t touched = 0;          // last admission / removal that changed `covered`
    State state = State::kWaiting;
    int32_t missing() const { return (int32_t)hashes.size() - covered; }
};

struct Entry {
    int32_t missing;
    uint64_t seq;
    int64_t id;
    uint32_t version;
};
struct EntryAfter {  // priority_queue keeps the largest on top: "after" = worse
    bool operator()(const Entry& a, const Entry& b) const {
        return a.missing != b.missing ? a.missing > b.missing : a.seq > b.seq;
    }
};

struct Holder {  // a waiting request holding a block hash (seq identifies the insertion)
    int64_t id;
    uint64_t seq;
};

// Runs `body` (which returns an XATTN_* code) so that no C++ exception crosses the C ABI:
// a failed allocation becomes XATTN_ERR_HOST_MEMORY.
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

struct xattn_cht {
    int32_t block = 1;
    uint64_t next_seq = 0;
    uint64_t op = 0;                // admissions and removals so far
    std::vector<int64_t> touched;   // waiting requests whose coverage the current one changed
    int64_t waiting = 0, active = 0;
    std::unordered_map<int64_t, Request> reqs;
    std::unordered_map<uint64_t, int32_t> working;  // block hash -> active requests holding it
    std::unordered_map<uint64_t, std::vector<Holder>> holders;  // block hash -> waiting holders
    std::priority_queue<Entry, std::vector<Entry>, EntryAfter> heap;

    void push(int64_t id, const Request& r) { heap.push(Entry{r.missing(), r.seq, id, r.version}); }

    bool live(const Entry& e) const {
        auto it = reqs.find(e.id);
        return it != reqs.end() && it->second.state == State::kWaiting && it->second.seq == e.seq &&
               it->second.version == e.version;
    }

    // The waiting holders of hash h whose covered count moves by `delta`; holders that are
    // no longer waiting (or were re-inserted) are dropped from the list on the way. Each
    // holder is listed once per operation in `touched`; flush() then gives it one heap entry.
    void adjust_holders(uint64_t h, int32_t delta) {
        auto it = holders.find(h);
        if (it == holders.end()) return;
        std::vector<Holder>& v = it->second;
        size_t keep = 0;
        for (size_t i = 0; i < v.size(); ++i) {
            auto rq = reqs.find(v[i].id);
            if (rq == reqs.end() || rq->second.state != State::kWaiting || rq->second.seq != v[i].seq) continue;
            v[keep++] = v[i];
            Request& r = rq->second;
            r.covered += delta;
            if (r.touched != op) {
                r.touched = op;
                touched.push_back(v[i].id);
            }
        }
        v.resize(keep);
        if (v.empty()) holders.erase(it);
    }

    // One fresh heap entry per request whose coverage the current operation changed.
    void flush() {
        for (int64_t id : touched) {
            Request& r = reqs.find(id)->second;
            ++r.version;
            push(id, r);
        }
        touched.clear();
    }

    void maybe_rebuild() {
        if (heap.size() <= 64 || heap.size() <= 4 * (size_t)waiting) return;
        std::priority_queue<Entry, std::vector<Entry>, EntryAfter> fresh;
        for (auto& kv : reqs)
            if (kv.second.state == State::kWaiting)
                fresh.push(Entry{kv.second.missing(), kv.second.seq, kv.first, kv.second.version});
        heap.swap(fresh);
    }
};

extern "C" {

xattn_cht* xattn_cht_create(int32_t block_tokens) {
    if (block_tokens < 1) return nullptr;
    try {
        xattn_cht* t = new xattn_cht();
        t->block = block_tokens;
        return t;
    } catch (...) {
        return nullptr;
    }
}

void xattn_cht_destroy(xattn_cht* cht) { delete cht; }

int xattn_cht_insert(xattn_cht* cht, int64_t request_id, const int32_t* tokens, int64_t num_tokens) {
    return guarded([&]() -> int {
        if (!cht || num_tokens < 0 || (num_tokens > 0 && !tokens)) return XATTN_ERR_INVALID_ARG;
        if (cht->reqs.count(request_id)) return XATTN_ERR_INVALID_ARG;
        Request r;
        const int64_t nb = num_tokens / cht->block;
        r.hashes.reserve((size_t)nb);
        uint64_t h = 0x6A09E667F3BCC909ull;  // any fixed start value
        for (int64_t i = 0; i < nb * cht->block; ++i) {
            h = mix64(h + (uint64_t)(uint32_t)tokens[i] + 0x9E3779B97F4A7C15ull);
            if ((i + 1) % cht->block == 0) r.hashes.push_back(h);
        }
        // covered blocks are a prefix: find its length by binary search on membership
        int32_t lo = 0, hi = (int32_t)r.hashes.size();
        while (lo < hi) {
            const int32_t mid = (lo + hi) / 2;
            if (cht->working.count(r.hashes[(size_t)mid])) lo = mid + 1;
            else hi = mid;
        }
        r.covered = lo;
        r.seq = cht->next_seq++;
        for (uint64_t bh : r.hashes) cht->holders[bh].push_back(Holder{request_id, r.seq});
        auto ins = cht->reqs.emplace(request_id, std::move(r));
        cht->push(request_id, ins.first->second);
        ++cht->waiting;
        return XATTN_OK;
    });
}

int xattn_cht_best(xattn_cht* cht, int64_t* request_id, int32_t* missing_blocks) {
    return guarded([&]() -> int {
        if (!cht || !request_id || !missing_blocks) return XATTN_ERR_INVALID_ARG;
        while (!cht->heap.empty()) {
            const Entry e = cht->heap.top();
            if (!cht->live(e)) {
                cht->heap.pop();
                continue;
            }
            *request_id = e.id;
            *missing_blocks = e.missing;
            return 1;
        }
        return 0;
    });
}

int xattn_cht_admit(xattn_cht* cht, int64_t request_id) {
    return guarded([&]() -> int {
        if (!cht) return XATTN_ERR_INVALID_ARG;
        auto it = cht->reqs.find(request_id);
        if (it == cht->reqs.end() || it->second.state != State::kWaiting) return XATTN_ERR_INVALID_ARG;
        Request& r = it->second;
        r.state = State::kActive;  // its own holder entries and heap entries are now stale
        --cht->waiting;
        ++cht->active;
        ++cht->op;
        for (uint64_t h : r.hashes)
            if (++cht->working[h] == 1) cht->adjust_holders(h, +1);
        cht->flush();
        cht->maybe_rebuild();
        return XATTN_OK;
    });
}

int xattn_cht_finish(xattn_cht* cht, int64_t request_id) {
    return guarded([&]() -> int {
        if (!cht) return XATTN_ERR_INVALID_ARG;
        auto it = cht->reqs.find(request_id);
        if (it == cht->reqs.end() || it->second.state != State::kActive) return XATTN_ERR_INVALID_ARG;
        ++cht->op;
        for (uint64_t h : it->second.hashes) {
            auto w = cht->working.find(h);
            if (w != cht->working.end() && --w->second == 0) {
                cht->working.erase(w);
                cht->adjust_holders(h, -1);
            }
        }
        cht->flush();
        cht->reqs.erase(it);
        --cht->active;
        cht->maybe_rebuild();
        return XATTN_OK;
    });
}

int xattn_cht_cancel(xattn_cht* cht, int64_t request_id) {
    return guarded([&]() -> int {
        if (!cht) return XATTN_ERR_INVALID_ARG;
        auto it = cht->reqs.find(request_id);
        if (it == cht->reqs.end() || it->second.state != State::kWaiting) return XATTN_ERR_INVALID_ARG;
        for (uint64_t h : it->second.hashes) {  // its holder entries go now; heap entries lazily
            auto hv = cht->holders.find(h);
            if (hv == cht->holders.end()) continue;
            std::vector<Holder>& v = hv->second;
            for (size_t i = 0; i < v.size(); ++i)
                if (v[i].id == request_id && v[i].seq == it->second.seq) {
                    v[i] = v.back();
                    v.pop_back();
                    break;
                }
            if (v.empty()) cht->holders.erase(hv);
        }
        cht->reqs.erase(it);
        --cht->waiting;
        cht->maybe_rebuild();
        return XATTN_OK;
    });
}

int xattn_cht_missing(const xattn_cht* cht, int64_t request_id, int32_t* missing_blocks) {
    if (!cht || !missing_blocks) return XATTN_ERR_INVALID_ARG;
    auto it = cht->reqs.find(request_id);
    if (it == cht->reqs.end() || it->second.state != State::kWaiting) return XATTN_ERR_INVALID_ARG;
    *missing_blocks = it->second.missing();
    return XATTN_OK;
}

int xattn_cht_counts(const xattn_cht* cht, int64_t* waiting, int64_t* active, int64_t* working_hashes) {
    if (!cht) return XATTN_ERR_INVALID_ARG;
    if (waiting) *waiting = cht->waiting;
    if (active) *active = cht->active;
    if (working_hashes) *working_hashes = (int64_t)cht->working.size();
    return XATTN_OK;
}

}  // extern "C"
