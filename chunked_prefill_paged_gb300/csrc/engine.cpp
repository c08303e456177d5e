// engine.cpp -- host-side serving harness (include/cpa_engine.h): greedy
// token budget, incremental block allocation with a null block, and the
// full-block prefix hash chain.  Plain C++ on the host; the rules and the
// choices made where the pages leave them open are stated in the header.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/cpa_engine.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

struct Fnv1a {
    uint64_t h = kFnvOffset;
    void byte(uint8_t b) {
        h ^= b;
        h *= kFnvPrime;  // modulo 2^64
    }
    void u64(uint64_t v) {
        for (int i = 0; i < 8; ++i) byte(uint8_t(v >> (8 * i)));
    }
    void i32(int32_t v) {
        const uint32_t u = uint32_t(v);
        for (int i = 0; i < 4; ++i) byte(uint8_t(u >> (8 * i)));
    }
};

uint64_t block_hash(uint64_t parent, uint64_t scope, const int32_t *tokens, int n) {
    Fnv1a f;
    f.u64(parent);
    f.u64(scope);
    for (int i = 0; i < n; ++i) f.i32(tokens[i]);
    return f.h;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Request {
    int64_t id;
    std::vector<int32_t> tokens;  // prompt, then outputs
    int32_t prompt_len;
    int32_t max_new;
    int32_t num_computed = 0;
    std::vector<int32_t> blocks;
    std::vector<uint64_t> hashes;  // of the full blocks computed so far
    bool started = false;
    bool finished = false;
    int32_t outputs() const { return int32_t(tokens.size()) - prompt_len; }
    bool decoding() const { return started && num_computed >= prompt_len; }
};

// Free blocks: a queue kept as a doubly linked list over block ids, so a
// prefix hit can take a free cached block out of the middle in O(1).
struct FreeQueue {
    std::vector<int32_t> prev, next;
    std::vector<uint8_t> in;
    int32_t head = -1, tail = -1, size = 0;
    explicit FreeQueue(int32_t n) : prev(n, -1), next(n, -1), in(n, 0) {}
    void push_back(int32_t b) {
        prev[b] = tail;
        next[b] = -1;
        if (tail >= 0) next[tail] = b; else head = b;
        tail = b;
        in[b] = 1;
        ++size;
    }
    void remove(int32_t b) {
        if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
        if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
        in[b] = 0;
        --size;
    }
    int32_t pop_front() {
        const int32_t b = head;
        remove(b);
        return b;
    }
};

}  // namespace

struct cpa_engine {
    cpa_engine_config cfg;
    FreeQueue free;
    std::vector<int32_t> ref;
    std::vector<uint64_t> hash_of;   // cached content hash of a block
    std::vector<uint8_t> has_hash;
    std::unordered_map<uint64_t, int32_t> cache;  // hash -> block
    std::vector<Request> reqs;                    // arrival order (finished ones dropped)
    std::unordered_set<int64_t> known_ids;
    bool pending = false;
    // the last plan
    std::vector<int64_t> p_ids;
    std::vector<int32_t> p_cached, p_new, p_cu, p_table, p_tokens;
    std::vector<int32_t> p_rows;  // index into reqs of each plan row

    explicit cpa_engine(const cpa_engine_config &c)
        : cfg(c), free(c.num_blocks), ref(c.num_blocks, 0), hash_of(c.num_blocks, 0), has_hash(c.num_blocks, 0) {
        for (int32_t b = 1; b < c.num_blocks; ++b) free.push_back(b);  // block 0 is the null block
    }

    int32_t take_free() {
        const int32_t b = free.pop_front();
        if (has_hash[b]) {  // the block is reused for new data: its cached content goes
            auto it = cache.find(hash_of[b]);
            if (it != cache.end() && it->second == b) cache.erase(it);
            has_hash[b] = 0;
        }
        ref[b] = 1;
        return b;
    }

    void claim_cached(int32_t b) {
        if (ref[b] == 0) free.remove(b);
        ++ref[b];
    }

    bool allocate_slots(Request &r, int32_t num_new) {
        const int64_t need = cdiv(int64_t(r.num_computed) + num_new, cfg.block_size);
        if (need > cfg.max_blocks_per_seq) return false;
        const int64_t extra = need - int64_t(r.blocks.size());
        if (extra > free.size) return false;
        for (int64_t i = 0; i < extra; ++i) r.blocks.push_back(take_free());
        return true;
    }

    // leading full prompt blocks whose hashes are cached, leaving at least one
    // prompt token to compute; claim == false only counts them
    int32_t prefix_hit(Request &r, bool claim) {
        const int32_t bs = cfg.block_size;
        const int32_t limit = (r.prompt_len - 1) / bs;
        uint64_t parent = 0;
        int32_t hit = 0;
        for (int32_t i = 0; i < limit; ++i) {
            const uint64_t h = block_hash(parent, cfg.scope_key, r.tokens.data() + int64_t(i) * bs, bs);
            auto it = cache.find(h);
            if (it == cache.end()) break;
            if (claim) {
                claim_cached(it->second);
                r.blocks.push_back(it->second);
                r.hashes.push_back(h);
            }
            parent = h;
            ++hit;
        }
        if (claim) r.num_computed = hit * bs;
        return hit * bs;
    }

    void finish(Request &r) {
        r.finished = true;
        for (auto it = r.blocks.rbegin(); it != r.blocks.rend(); ++it) {
            if (--ref[*it] == 0) free.push_back(*it);
        }
        r.blocks.clear();
    }
};

extern "C" {

cpa_status cpa_engine_create(const cpa_engine_config *config, cpa_engine **out) {
    if (!out) return CPA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!config || config->num_blocks < 2 || config->block_size < 1 || config->max_blocks_per_seq < 1 ||
        config->max_batched_tokens < 1 || config->chunk_size < 1)
        return CPA_ERR_INVALID_ARG;
    cpa_engine *e = new (std::nothrow) cpa_engine(*config);
    if (!e) return CPA_ERR_INVALID_ARG;
    *out = e;
    return CPA_SUCCESS;
}

void cpa_engine_destroy(cpa_engine *engine) { delete engine; }

cpa_status cpa_engine_add_request(cpa_engine *e, int64_t request_id, const int32_t *prompt, int32_t prompt_len,
                                  int32_t max_new_tokens) {
    if (!e || !prompt || prompt_len < 1 || max_new_tokens < 1) return CPA_ERR_INVALID_ARG;
    if (e->known_ids.count(request_id)) return CPA_ERR_INVALID_ARG;
    Request r;
    r.id = request_id;
    r.tokens.assign(prompt, prompt + prompt_len);
    r.prompt_len = prompt_len;
    r.max_new = max_new_tokens;
    e->reqs.push_back(std::move(r));
    e->known_ids.insert(request_id);
    return CPA_SUCCESS;
}

cpa_status cpa_engine_schedule(cpa_engine *e, cpa_step_plan *plan) {
    if (!e || !plan) return CPA_ERR_INVALID_ARG;
    if (e->pending) return CPA_ERR_INVALID_ARG;  // the previous step was not committed
    e->p_rows.clear();
    const int32_t budget = e->cfg.max_batched_tokens;
    std::vector<int32_t> take;
    int32_t used = 0;
    // decodes first, one token each
    for (size_t i = 0; i < e->reqs.size(); ++i) {
        Request &r = e->reqs[i];
        if (r.finished || !r.decoding()) continue;
        if (used >= budget) break;
        if (!e->allocate_slots(r, 1)) continue;
        e->p_rows.push_back(int32_t(i));
        take.push_back(1);
        used += 1;
    }
    // then prompt chunks in arrival order
    for (size_t i = 0; i < e->reqs.size(); ++i) {
        Request &r = e->reqs[i];
        if (r.finished || r.decoding()) continue;
        if (used >= budget) break;
        if (!r.started) {
            e->prefix_hit(r, true);
            r.started = true;
        }
        const int32_t n = std::min(std::min(e->cfg.chunk_size, budget - used), r.prompt_len - r.num_computed);
        if (n <= 0 || !e->allocate_slots(r, n)) continue;
        e->p_rows.push_back(int32_t(i));
        take.push_back(n);
        used += n;
    }
    const int32_t nr = int32_t(e->p_rows.size()), cols = e->cfg.max_blocks_per_seq;
    e->p_ids.assign(nr, 0);
    e->p_cached.assign(nr, 0);
    e->p_new.assign(take.begin(), take.end());
    e->p_cu.assign(nr + 1, 0);
    e->p_table.assign(size_t(nr) * cols, 0);
    e->p_tokens.clear();
    for (int32_t k = 0; k < nr; ++k) {
        const Request &r = e->reqs[e->p_rows[k]];
        e->p_ids[k] = r.id;
        e->p_cached[k] = r.num_computed;
        e->p_cu[k + 1] = e->p_cu[k] + take[k];
        std::copy(r.blocks.begin(), r.blocks.end(), e->p_table.begin() + size_t(k) * cols);
        e->p_tokens.insert(e->p_tokens.end(), r.tokens.begin() + r.num_computed,
                           r.tokens.begin() + r.num_computed + take[k]);
    }
    plan->num_reqs = nr;
    plan->max_blocks_per_seq = cols;
    plan->total_new_tokens = e->p_cu[nr];
    plan->request_ids = e->p_ids.data();
    plan->cached_seq_len = e->p_cached.data();
    plan->num_new_tokens = e->p_new.data();
    plan->cu_new_tokens = e->p_cu.data();
    plan->block_table = e->p_table.data();
    plan->token_ids = e->p_tokens.data();
    e->pending = true;
    return CPA_SUCCESS;
}

cpa_status cpa_engine_commit(cpa_engine *e, const int32_t *sampled_tokens) {
    if (!e || !e->pending) return CPA_ERR_INVALID_ARG;
    if (!sampled_tokens && !e->p_rows.empty()) return CPA_ERR_INVALID_ARG;
    const int32_t bs = e->cfg.block_size;
    for (size_t k = 0; k < e->p_rows.size(); ++k) {
        Request &r = e->reqs[e->p_rows[k]];
        r.num_computed += e->p_new[k];
        while (int32_t(r.hashes.size()) < r.num_computed / bs) {
            const size_t i = r.hashes.size();
            const uint64_t parent = r.hashes.empty() ? 0 : r.hashes.back();
            const uint64_t h = block_hash(parent, e->cfg.scope_key, r.tokens.data() + i * bs, bs);
            r.hashes.push_back(h);
            const int32_t b = r.blocks[i];
            if (!e->cache.count(h)) {
                e->cache[h] = b;
                e->hash_of[b] = h;
                e->has_hash[b] = 1;
            }
        }
        if (r.num_computed >= r.prompt_len) {
            r.tokens.push_back(sampled_tokens[k]);
            if (r.outputs() >= r.max_new) e->finish(r);
        }
    }
    // drop finished requests, keeping arrival order
    e->reqs.erase(std::remove_if(e->reqs.begin(), e->reqs.end(), [](const Request &r) { return r.finished; }),
                  e->reqs.end());
    e->p_rows.clear();
    e->pending = false;
    return CPA_SUCCESS;
}

int32_t cpa_engine_num_free_blocks(const cpa_engine *e) { return e ? e->free.size : 0; }

int32_t cpa_engine_num_unfinished(const cpa_engine *e) { return e ? int32_t(e->reqs.size()) : 0; }

int32_t cpa_engine_prefix_hit_tokens(const cpa_engine *e, int64_t request_id) {
    if (!e) return 0;
    for (const Request &r : e->reqs) {
        if (r.id == request_id) {
            if (r.started) return 0;
            Request copy = r;
            return const_cast<cpa_engine *>(e)->prefix_hit(copy, false);
        }
    }
    return 0;
}

}  // extern "C"
